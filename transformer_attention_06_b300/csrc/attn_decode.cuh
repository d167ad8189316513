// K3: KV-cache single-token decode -- persistent, split over equal ranges of cache tiles, merged in the same launch.
//
// What it computes ("nanochat Admin & Developer Guide", section 7 "KV cache": FA3 layout (B, T, H, D), per-row
// cache_seqlens, in-place append; section 6: the SDPA decode case attends over a slice of the cache): for sequence b
// with p = cache_lens[b], the new query is roped at position p and normed; it attends over cache rows
// [max(0, p - window), p) -- plus row p when a new key/value is given, which is roped + normed at position p,
// written into the cache and attended to.
//
// Work split.  A segment is one (sequence b, kv head g): its visible cache rows, cut into tiles of 128 rows.  All
// segments' tiles, in (b, g) order, form one list of N tiles; CTA c of the C resident CTAs (one per SM) takes the
// contiguous range [c N / C, (c + 1) N / C), so every CTA streams the same number of bytes whatever the mix of cache
// lengths.  Each CTA computes N and its starting segment itself from cache_lens (the host never reads them).
// A segment that lies wholly inside one range is finished by that CTA; a segment cut by range borders leaves one
// partial (m, l, o) per CTA in the workspace, and the last CTA to arrive (atomic counter) merges them with the
// log-sum-exp rule and resets the counter.  The new key (when given) joins at the end as one more key.
//
// The contractions are tiny in M (the G <= 16 query heads of a group) but long in the cache dimension, so they run
// on the tensor cores with the cache rows in the M dimension:
//   S   [128 rows x 16]  = K_tile [128 x 128 dims] . Q^T      (A = K tile, K-major; B = Q, K-major)
//   O^T [128 dims x 16] += V_tile^T [128 dims x 128 rows] . P^T (A = V tile, MN-major; B = P^T, K-major)
// with Q and P padded to 16 heads (rows >= G are zero).  S and O^T live in TMEM; the CUDA cores only run the
// softmax.  The kernel is bound by HBM reads of the cache.
//
// Warp roles (384 threads):
//   warps 0-3   softmax (thread r = cache row r of the tile = TMEM lane r): scores of the G heads, block-wide tile
//               maximum, P^T into shared memory, lazy rescale of O^T; hands (m, row sums) of a finished segment
//               to the epilogue warps and goes on with the next tile;
//   warp 4      TMA producer: K and V tiles through two 3-stage rings (a K stage recycles once S of its tile is
//               computed, a V stage once P.V is);
//   warp 5      TMEM allocator and MMA issuer (one thread);
//   warp 6      query builder: RoPE + RMSNorm of the G queries of each segment into a 4-slot ring of Q operands;
//   warp 7      sequences with no visible cache row (p = 0, window 0, invalid length), handled without tiles;
//   warps 8-11  segment epilogue (thread d = dim d = TMEM lane d): reads O^T of a finished segment (double-buffered
//               by segment parity), then writes the output, or a partial that the last CTA of the segment merges.
#pragma once

#include "common.cuh"

namespace nc {
namespace dec {

constexpr int kRows = 128;                    // cache rows per tile
constexpr int kStages = 3;
constexpr int kHalfBytes = kRows * 128;       // one 64-dim half of a tile: 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;    // 32 KB
constexpr int kN = 16;                        // MMA N: heads of the group, padded
constexpr int kMaxG = 16;
constexpr int kOpBytes = kN * 256;            // a [16][128] bf16 operand (Q or P^T): 4 KB
constexpr int kOpHalf = kN * 128;             // one 64-element K half of it: 2 KB
constexpr int kQSlots = 4;
constexpr int kThreads = 384;
constexpr int kSoftThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kQWarp = 6;
constexpr int kEmptyWarp = 7;
constexpr int kEpiWarp0 = 8;                  // warps 8-11
constexpr uint32_t kBarSoft = 1, kBarEpi = 2; // named barrier ids of the softmax and epilogue warp groups
constexpr int kMaxParts = 256;                // upper bound on the grid (partials per CTA: 2)
constexpr int kOBufs = 4;                     // O^T buffers in TMEM, by segment index modulo 4
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0;                 // S buffers: [0,16) and [16,32)
constexpr uint32_t kColO = 32;                // O^T of segment k: [32 + 16 (k % 4), 48 + 16 (k % 4))
constexpr uint32_t kIdescS = idesc_bf16_f32(128, kN, false, false);  // A = K (K-major), B = Q (K-major)
constexpr uint32_t kIdescO = idesc_bf16_f32(128, kN, true, false);   // A = V (MN-major), B = P^T (K-major)
constexpr float kRescaleLog2 = 8.f;           // O, l are rescaled only when the maximum grows by more than 2^8
constexpr int kLensCache = 1024;              // cache_lens of the first 1024 sequences are kept in shared memory

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffQ = kOffV + kStages * kTileBytes;
constexpr int kOffP = kOffQ + kQSlots * kOpBytes;
constexpr int kOffRed = kOffP + 2 * kOpBytes;          // [2][16 heads][4 warps] f32 tile maxima
constexpr int kOffSegM = kOffRed + 2 * kN * 4 * 4;     // [4][16] f32 segment maxima (softmax -> epilogue)
constexpr int kOffSegL = kOffSegM + kOBufs * kN * 4;   // [4][16 heads][4 warps] f32 segment row sums
constexpr int kOffNewK = kOffSegL + kOBufs * kN * 4 * 4;  // new key (normed, bf16-rounded) [128] f32
constexpr int kOffNewV = kOffNewK + 128 * 4;           // new value [128] f32
constexpr int kOffSNew = kOffNewV + 128 * 4;           // score of the new key per head [16] f32
constexpr int kOffLens = kOffSNew + kN * 4;
constexpr int kOffParts = kOffLens + kLensCache * 4;   // partial slots of a segment's parts [kMaxParts] int
constexpr int kOffBar = kOffParts + kMaxParts * 4;
constexpr int kNumBars = 4 * kStages + 2 + 2 + 2 + 2 * kQSlots + 4 * kOBufs + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kMiscBytes = 256;
constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* kcache;
  __nv_bfloat16* vcache;
  const int* cache_lens;
  __nv_bfloat16* out;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  // Gated value embedding of the new token (both null, or both set with k_new): the new value is
  // v_new + sigmoid(ve_gate) ve_new, one gate logit per (b, kv head), rounded to bf16 once.
  const __nv_bfloat16* ve_new;
  const __nv_bfloat16* ve_gate;
  float* ws_ml;        // [C][2][G][2]   (m, l) of each partial, log2 domain
  float* ws_o;         // [C][2][G][128] unnormalised partial outputs
  unsigned* ws_cnt;    // [B][Hkv] arrival counters, zero between calls
  int B, Hq, Hkv, G, Tcap, window;
  float scale_log2;    // log2(e) / sqrt(D)
  unsigned long long wait_limit_ns;
};

// Lane `lane`'s four elements [4 lane, 4 lane + 4) of the new value of (b, kv head g), as bf16 pairs: v_new, or with a
// value embedding v_new + sigmoid(gate) ve_new in fp32, rounded to bf16.
__device__ __forceinline__ uint2 new_value4(const Params& p, int b, int g, int lane) {
  const size_t row = (static_cast<size_t>(b) * p.Hkv + g) * 128;
  const uint2 vv = __ldg(reinterpret_cast<const uint2*>(p.v_new + row) + lane);
  if (p.ve_new == nullptr) return vv;
  const uint2 ee = __ldg(reinterpret_cast<const uint2*>(p.ve_new + row) + lane);
  const float a = 1.f / (1.f + expf(-__bfloat162float(p.ve_gate[static_cast<size_t>(b) * p.Hkv + g])));
  return make_uint2(pack_bf16x2(fmaf(a, bf16_lo(ee.x), bf16_lo(vv.x)), fmaf(a, bf16_hi(ee.x), bf16_hi(vv.x))),
                    pack_bf16x2(fmaf(a, bf16_lo(ee.y), bf16_lo(vv.y)), fmaf(a, bf16_hi(ee.y), bf16_hi(vv.y))));
}

// ---- segment bookkeeping ------------------------------------------------------------------------------------------
struct SeqInfo {
  int pos;    // cache_lens[b]
  int lo;     // first visible cache row
  int rows;   // visible cache rows (0 when the length is invalid)
  int nt;     // tiles
  bool valid;
};

__device__ __forceinline__ SeqInfo seq_info(const Params& p, int b, const int* lens_s) {
  SeqInfo s;
  s.pos = b < kLensCache ? lens_s[b] : __ldg(p.cache_lens + b);
  const int max_pos = p.k_new != nullptr ? p.Tcap - 1 : p.Tcap;
  s.valid = s.pos >= 0 && s.pos <= max_pos;
  s.lo = (p.window < 0 || !s.valid) ? 0 : max(0, s.pos - p.window);
  s.rows = s.valid ? s.pos - s.lo : 0;
  s.nt = (s.rows + kRows - 1) / kRows;
  return s;
}

// Walks the tile list from a CTA's first tile: (b, g, i) = sequence, kv head, tile within the segment.
struct Cursor {
  int b, g, i;
  SeqInfo s;
  long long pref;  // global index of tile (b, g = 0, i = 0): Hkv * sum of nt over earlier sequences

  __device__ __forceinline__ long long seg_tile0(int Hkv) const { return pref + static_cast<long long>(g) * s.nt; }
  __device__ __forceinline__ void advance(const Params& p, const int* lens_s) {
    if (++i < s.nt) return;
    i = 0;
    if (++g < p.Hkv) return;
    g = 0;
    pref += static_cast<long long>(p.Hkv) * s.nt;
    for (++b; b < p.B; ++b) {
      s = seq_info(p, b, lens_s);
      if (s.nt > 0) break;
    }
  }
};

// floor(a / b) for 0 <= a, 0 < b; 32-bit division when both fit (the usual case), 64-bit otherwise.
__device__ __forceinline__ long long div_floor(long long a, long long b) {
  if (a < (1ll << 32) && b < (1ll << 32))
    return static_cast<long long>(static_cast<unsigned>(a) / static_cast<unsigned>(b));
  return a / b;
}
// CTA owning global tile x when N tiles are split into C ranges [c N / C, (c + 1) N / C).
__device__ __forceinline__ int tile_owner(long long x, long long N, int C) {
  return static_cast<int>(div_floor((x + 1) * C - 1, N));
}
__device__ __forceinline__ long long range_begin(int c, long long N, int C) { return div_floor(c * N, C); }
// With fewer tiles than CTAs some ranges are empty; they own no tile and leave no partial.
__device__ __forceinline__ bool range_empty(int c, long long N, int C) {
  return range_begin(c, N, C) == range_begin(c + 1, N, C);
}

// Byte offset of element (row j, column k) of a [16][128] bf16 operand in the 128-byte-swizzled K-major layout:
// two 64-column halves of 16 rows x 128 bytes, 16-byte chunk index xor (row % 8).
__device__ __forceinline__ uint32_t op_off(int j, int k) {
  return (k >> 6) * kOpHalf + j * 128 + ((((k & 63) >> 3) ^ (j & 7)) << 4) + ((k & 7) << 1);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// RoPE + RMSNorm of one 128-wide bf16 head vector by one warp: lane l owns pairs 2l and 2l+1, i.e. elements
// {2l, 2l+1} and {64+2l, 64+2l+1}, returned in y[0..3] = (x[2l], x[2l+1], x[64+2l], x[65+2l]).  cs / sn hold the
// cos / sin of the lane's two pair angles (warp_rope_angles).
__device__ __forceinline__ void warp_rope_angles(float pos, const RopeTable& tab, int lane, float (&cs)[2],
                                                 float (&sn)[2]) {
#pragma unroll
  for (int e = 0; e < 2; ++e) rope_cos_sin(pos, tab.hi[2 * lane + e], tab.lo[2 * lane + e], cs[e], sn[e]);
}
__device__ __forceinline__ void rope_norm_pairs(uint32_t a, uint32_t b, const float (&cs)[2], const float (&sn)[2],
                                                float (&y)[4]) {
  const float x1[2] = {bf16_lo(a), bf16_hi(a)};
  const float x2[2] = {bf16_lo(b), bf16_hi(b)};
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    y[e] = fmaf(x1[e], cs[e], x2[e] * sn[e]);
    y[2 + e] = fmaf(x2[e], cs[e], -(x1[e] * sn[e]));
    ss = fmaf(y[e], y[e], ss);
    ss = fmaf(y[2 + e], y[2 + e], ss);
  }
  const float inv = rsqrtf(warp_sum(ss) * (1.0f / 128.0f) + kRmsEps);
#pragma unroll
  for (int e = 0; e < 4; ++e) y[e] *= inv;
}
__device__ __forceinline__ void warp_rope_norm(const __nv_bfloat16* src, const float (&cs)[2], const float (&sn)[2],
                                               int lane, float (&y)[4]) {
  rope_norm_pairs(__ldg(reinterpret_cast<const uint32_t*>(src) + lane),
                  __ldg(reinterpret_cast<const uint32_t*>(src + 64) + lane), cs, sn, y);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ RopeTable tab, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sP = smem + kOffP;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* seg_m = reinterpret_cast<float*>(smem + kOffSegM);
  float* seg_l = reinterpret_cast<float*>(smem + kOffSegL);
  float* new_k = reinterpret_cast<float*>(smem + kOffNewK);
  float* new_v = reinterpret_cast<float*>(smem + kOffNewV);
  float* s_new = reinterpret_cast<float*>(smem + kOffSNew);
  int* lens_s = reinterpret_cast<int*>(smem + kOffLens);
  int* part_slot = reinterpret_cast<int*>(smem + kOffParts);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* k_full = bars;                       // [kStages]  TMA -> MMA
  uint64_t* v_full = bars + kStages;             // [kStages]  TMA -> MMA, softmax
  uint64_t* k_empty = bars + 2 * kStages;        // [kStages]  S issued from the K stage       MMA -> TMA
  uint64_t* v_empty = bars + 3 * kStages;        // [kStages]  P.V issued from the V stage     MMA -> TMA
  uint64_t* s_full = bars + 4 * kStages;         // [2]  S of tiles with that parity          MMA -> softmax
  uint64_t* p_full = s_full + 2;                 // [2]  P^T written (128 arrivals)          softmax -> MMA
  uint64_t* o_done = p_full + 2;                 // [2]  P.V of tiles with that parity        MMA -> softmax
  uint64_t* q_full = o_done + 2;                 // [kQSlots]                                  Q warp -> MMA
  uint64_t* q_empty = q_full + kQSlots;          // [kQSlots]                                  epilogue -> Q warp
  uint64_t* o_full = q_empty + kQSlots;          // [4]  O of segment k (k % 4) final          MMA -> epilogue
  uint64_t* o_free = o_full + kOBufs;            // [4]  O read by the epilogue               epilogue -> MMA
  uint64_t* seg_ready = o_free + kOBufs;         // [4]  (m, l) of a segment handed over      softmax -> epilogue
  uint64_t* seg_free = seg_ready + kOBufs;       // [4]  hand-over slot read                   epilogue -> softmax
  uint64_t* mma_final = seg_free + kOBufs;
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;
  int* last_flag = misc + 2;
  int* start_b = misc + 3;
  int* start_gi = misc + 4;                      // tile offset inside sequence start_b
  long long* ll = reinterpret_cast<long long*>(misc + 6);  // [0] N, [1] start pref, [2] scan carry, [4..15] sums
  int* warp_tot = misc + 40;                     // [12] per-warp scan totals

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = gridDim.x, c = blockIdx.x;
  const bool has_new = p.k_new != nullptr;
  const unsigned long long lim = p.wait_limit_ns;
  // Launched with programmatic dependent launch: the next kernel in the stream may be scheduled now (its CTAs take
  // SMs as this grid's CTAs exit, and wait for this grid to complete before reading anything), and this grid's own
  // set-up below runs while the previous kernel drains; nothing an earlier kernel may write (cache lengths, q, the
  // caches, the workspace) is read before the griddepcontrol.wait further down.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ------------------------------------------------------------------ set-up: barriers, TMEM, operand padding
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(p_full + s, kSoftThreads);
      mbar_init(o_done + s, 1);
    }
    for (int s = 0; s < kOBufs; ++s) {
      mbar_init(o_full + s, 1);
      mbar_init(o_free + s, 1);
      mbar_init(seg_ready + s, 1);
      mbar_init(seg_free + s, 1);
    }
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // Q slots and P buffers start all-zero: rows >= G are never written again and must contribute nothing.
  for (int i = tid; i < (kQSlots + 2) * kOpBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int b = tid; b < min(p.B, kLensCache); b += kThreads) lens_s[b] = p.cache_lens[b];
  __syncthreads();

  // ------------------------------------------------------------------ set-up: N and this CTA's first tile
  // Pass 1: N = Hkv * sum_b nt_b.  Pass 2: the sequence holding tile range_begin(c).
  {
    long long tot = 0;
    for (int b0 = 0; b0 < p.B; b0 += kThreads) {
      const int b = b0 + tid;
      tot += (b < p.B) ? seq_info(p, b, lens_s).nt : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) ll[4 + warp] = tot;
    __syncthreads();
    if (tid == 0) {
      long long n = 0;
      for (int w = 0; w < kThreads / 32; ++w) n += ll[4 + w];
      ll[0] = n * p.Hkv;
      ll[2] = 0;
      *start_b = -1;
    }
    __syncthreads();
    const long long N = ll[0];
    const long long t_begin = range_begin(c, N, C);
    if (t_begin < range_begin(c + 1, N, C)) {
      for (int b0 = 0; b0 < p.B; b0 += kThreads) {
        const int b = b0 + tid;
        const int nt = (b < p.B) ? seq_info(p, b, lens_s).nt : 0;
        int inc = nt;  // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += v;
        }
        if (lane == 31) warp_tot[warp] = inc;
        __syncthreads();
        int woff = 0;
        for (int w = 0; w < warp; ++w) woff += warp_tot[w];
        const long long carry = ll[2];
        const long long lo_t = (carry + woff + inc - nt) * p.Hkv;
        const long long hi_t = (carry + woff + inc) * p.Hkv;
        if (nt > 0 && t_begin >= lo_t && t_begin < hi_t) {
          *start_b = b;
          start_gi[0] = static_cast<int>(t_begin - lo_t);
          ll[1] = lo_t;
        }
        __syncthreads();
        if (tid == kThreads - 1) ll[2] = carry + woff + inc;
        const bool found = *start_b >= 0;
        __syncthreads();
        if (found) break;
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const long long N = ll[0];
  const long long t_begin = range_begin(c, N, C);
  const int ntiles = static_cast<int>(range_begin(c + 1, N, C) - t_begin);

  Cursor cur0;
  if (ntiles > 0) {
    cur0.b = *start_b;
    cur0.s = seq_info(p, cur0.b, lens_s);
    cur0.g = start_gi[0] / cur0.s.nt;
    cur0.i = start_gi[0] - cur0.g * cur0.s.nt;
    cur0.pref = ll[1];
  }

  if (warp == kProducerWarp) {
    if (lane == 0 && ntiles > 0) {
      // ---------------------------------------------------------------- TMA producer
      // Separate K and V rings: a K stage is free again once S of its tile has been computed, a V stage once P.V
      // has, so K loads run ahead of V loads.  Both queues are served in whichever order stages free up.
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      Cursor ck = cur0, cv = cur0;
      int tk = 0, tv = 0;
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      while (tv < ntiles) {
        bool progress = false;
        if (tk < ntiles && (tk < kStages || mbar_test(k_empty + tk % kStages, ((tk / kStages) - 1) & 1))) {
          const int st = tk % kStages;
          uint8_t* dk = sK + st * kTileBytes;
          const int row0 = ck.s.lo + ck.i * kRows;
          mbar_arrive_expect_tx(k_full + st, kTileBytes);
          tma_load_4d(dk, &tmK, k_full + st, 0, ck.g, row0, ck.b);
          tma_load_4d(dk + kHalfBytes, &tmK, k_full + st, 64, ck.g, row0, ck.b);
          ++tk;
          ck.advance(p, lens_s);
          progress = true;
        }
        if (tv < tk && (tv < kStages || mbar_test(v_empty + tv % kStages, ((tv / kStages) - 1) & 1))) {
          const int st = tv % kStages;
          uint8_t* dv = sV + st * kTileBytes;
          const int row0 = cv.s.lo + cv.i * kRows;
          mbar_arrive_expect_tx(v_full + st, kTileBytes);
          tma_load_4d(dv, &tmV, v_full + st, 0, cv.g, row0, cv.b);
          tma_load_4d(dv + kHalfBytes, &tmV, v_full + st, 64, cv.g, row0, cv.b);
          ++tv;
          cv.advance(p, lens_s);
          progress = true;
        }
        if (progress) {
          spins = 0;
          continue;
        }
        if ((++spins & 63u) == 0) {
          if (*abort_flag) break;
          const uint64_t now = global_timer_ns();
          if (spins == 64) t_idle = now;
          else if (now - t_idle > lim) {
            raise_status(NC_DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
      // Every copy this CTA started must land before the CTA exits (already true on the normal path).
      for (int t = max(0, tk - kStages); t < tk; ++t) mbar_wait(k_full + t % kStages, (t / kStages) & 1, lim, nullptr);
      for (int t = max(0, tv - kStages); t < tv; ++t) mbar_wait(v_full + t % kStages, (t / kStages) & 1, lim, nullptr);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      // ---------------------------------------------------------------- MMA issuer
      // Two queues, served in whichever order their inputs arrive: S_ts = K_ts Q^T (needs the K tile, the Q of its
      // segment, and P.V of tile ts-2 issued so that S buffer ts & 1 is free) and O^T += V_tp^T P_tp^T (needs P^T and
      // the V tile, and for a segment's first tile the O buffer released by the epilogue).  Serving P.V as soon as
      // it is ready keeps a segment's final P.V from waiting behind the next tile's K load.
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aP = smem_u32(sP);
      Cursor cs = cur0, cpv = cur0;
      int ts = 0, tp = 0, seg_s = -1, seg_p = -1;
      uint64_t t_idle = global_timer_ns();
      uint32_t spins = 0;
      while (tp < ntiles) {
        bool progress = false;
        if (ts < ntiles && ts <= tp + 1) {
          const bool first = (ts == 0 || cs.i == 0);
          const int sg = seg_s + (first ? 1 : 0);
          const int st = ts % kStages;
          if ((!first || mbar_test(q_full + sg % kQSlots, (sg / kQSlots) & 1)) &&
              mbar_test(k_full + st, (ts / kStages) & 1)) {
            seg_s = sg;
            tc_fence_after_sync();
            const uint32_t qa = aQ + (sg % kQSlots) * kOpBytes;
            const uint32_t ka = aK + st * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              umma_ss(tbase + kColS + (ts & 1) * kN,
                      sdesc_sw128(ka + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(qa + (kk >> 2) * kOpHalf + (kk & 3) * 32, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full + (ts & 1));
            umma_commit(k_empty + st);
            ++ts;
            cs.advance(p, lens_s);
            progress = true;
          }
        }
        if (tp < ts) {
          const bool first = (tp == 0 || cpv.i == 0);
          const bool last = (tp == ntiles - 1 || cpv.i == cpv.s.nt - 1);
          const int sg = seg_p + (first ? 1 : 0);
          const int st = tp % kStages;
          if ((!first || sg < kOBufs || mbar_test(o_free + sg % kOBufs, ((sg / kOBufs) - 1) & 1)) &&
              mbar_test(p_full + (tp & 1), (tp >> 1) & 1) && mbar_test(v_full + st, (tp / kStages) & 1)) {
            seg_p = sg;
            tc_fence_after_sync();
            const uint32_t va = aV + st * kTileBytes;
            const uint32_t pa = aP + (tp & 1) * kOpBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              umma_ss(tbase + kColO + (sg % kOBufs) * kN, sdesc_sw128(va + kk * 2048, kHalfBytes, 1024),
                      sdesc_sw128(pa + (kk >> 2) * kOpHalf + (kk & 3) * 32, 16, 1024), kIdescO,
                      (!first || kk > 0) ? 1u : 0u);
            }
            umma_commit(o_done + (tp & 1));
            umma_commit(v_empty + st);
            if (last) umma_commit(o_full + sg % kOBufs);
            ++tp;
            cpv.advance(p, lens_s);
            progress = true;
          }
        }
        if (progress) {
          spins = 0;
          continue;
        }
        // Bounded idle: give up (and stop the other roles) when nothing became ready for the wait limit.
        if ((++spins & 63u) == 0) {
          if (*abort_flag) break;
          const uint64_t now = global_timer_ns();
          if (spins == 64) t_idle = now;
          else if (now - t_idle > lim) {
            raise_status(NC_DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
      umma_commit(mma_final);  // all issued MMAs complete before TMEM is released
      mbar_wait(mma_final, 0, lim, nullptr);
    }
  } else if (warp == kQWarp) {
    if (ntiles > 0) {
      // ---------------------------------------------------------------- query builder
      // The raw queries of the next segment are loaded while the current one is normalised, so that a run of short
      // segments does not wait on one global-load round trip per head.
      Cursor cu = cur0;
      int seg = 0, t = 0;
      uint32_t raw[G][2];
      auto load_raw = [&](const Cursor& k) {
        const __nv_bfloat16* src = p.q + (static_cast<size_t>(k.b) * p.Hq + k.g * G) * 128;
#pragma unroll
        for (int j = 0; j < G; ++j) {
          raw[j][0] = __ldg(reinterpret_cast<const uint32_t*>(src + j * 128) + lane);
          raw[j][1] = __ldg(reinterpret_cast<const uint32_t*>(src + j * 128 + 64) + lane);
        }
      };
      load_raw(cu);
      while (t < ntiles) {
        const int slot = seg % kQSlots;
        float cs[2], sn[2];
        warp_rope_angles(static_cast<float>(cu.s.pos), tab, lane, cs, sn);
        float y[G][4];
#pragma unroll
        for (int j = 0; j < G; ++j) rope_norm_pairs(raw[j][0], raw[j][1], cs, sn, y[j]);
        // next segment of the range: skip the rest of this one
        const int left = cu.s.nt - cu.i;
        t += left;
        for (int k = 0; k < left; ++k) cu.advance(p, lens_s);
        if (t < ntiles) load_raw(cu);
        bool ok = true;
        if (seg >= kQSlots) ok = mbar_wait(q_empty + slot, ((seg / kQSlots) - 1) & 1, lim, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        uint8_t* qs = sQ + slot * kOpBytes;
#pragma unroll
        for (int j = 0; j < G; ++j) {
          *reinterpret_cast<uint32_t*>(qs + op_off(j, 2 * lane)) = pack_bf16x2(y[j][0], y[j][1]);
          *reinterpret_cast<uint32_t*>(qs + op_off(j, 64 + 2 * lane)) = pack_bf16x2(y[j][2], y[j][3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full + slot);
        ++seg;
      }
    }
  } else if (warp == kEmptyWarp) {
    // ------------------------------------------------------------------ sequences with no visible cache row
    for (int b = c; b < p.B; b += C) {
      const SeqInfo s = seq_info(p, b, lens_s);
      if (s.rows > 0) continue;
      if (!s.valid && lane == 0) raise_status(NC_DEV_BAD_CACHE_LEN);
      for (int g = 0; g < p.Hkv; ++g) {
        uint2* outg = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * p.Hq + g * G) * 128);
        if (s.valid && has_new) {
          // The new key is the only visible key: the output is v_new; k_new / v_new go to cache row pos.
          const size_t crow = ((static_cast<size_t>(b) * p.Tcap + s.pos) * p.Hkv + g) * 128;
          float y[4], cs[2], sn[2];
          warp_rope_angles(static_cast<float>(s.pos), tab, lane, cs, sn);
          warp_rope_norm(p.k_new + (static_cast<size_t>(b) * p.Hkv + g) * 128, cs, sn, lane, y);
          reinterpret_cast<uint32_t*>(p.kcache + crow)[lane] = pack_bf16x2(y[0], y[1]);
          reinterpret_cast<uint32_t*>(p.kcache + crow + 64)[lane] = pack_bf16x2(y[2], y[3]);
          const uint2 vv = new_value4(p, b, g, lane);
          reinterpret_cast<uint2*>(p.vcache + crow)[lane] = vv;
          for (int j = 0; j < G; ++j) outg[j * 32 + lane] = vv;
        } else {
          for (int j = 0; j < G; ++j) outg[j * 32 + lane] = make_uint2(0, 0);
        }
      }
    }
  } else if (warp < 4) {
    if (ntiles > 0) {
      // ---------------------------------------------------------------- softmax (warps 0-3)
      const int r = tid;  // cache row of the tile
      const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
      Cursor cu = cur0;
      int seg = -1;
      float m[G], l[G];
      bool ok = true;
      for (int t = 0; t < ntiles; ++t) {
        const bool first = (t == 0 || cu.i == 0);
        const bool last = (t == ntiles - 1 || cu.i == cu.s.nt - 1);
        const int n = min(kRows, cu.s.rows - cu.i * kRows);
        const int st = t % kStages;
        if (first) {
          ++seg;
#pragma unroll
          for (int j = 0; j < G; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
          }
        }
        const uint32_t tO = tbase + lane_base + kColO + (seg % kOBufs) * kN;
        // ---- scores of row r, block-wide tile maximum per head
        ok = ok && mbar_wait(s_full + (t & 1), (t >> 1) & 1, lim, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        float x[G];
        float* redb = red + (t & 1) * kN * 4;
        if (ok) {
          tc_fence_after_sync();
          uint32_t sv[16];
          tmem_ld16(tbase + lane_base + kColS + (t & 1) * kN, sv);
          tmem_ld_wait16(sv);
          float mx[G];
#pragma unroll
          for (int j = 0; j < G; ++j) x[j] = __uint_as_float(sv[j]) * p.scale_log2;
          if (r >= n) {
#pragma unroll
            for (int j = 0; j < G; ++j) x[j] = -INFINITY;
          }
#pragma unroll
          for (int j = 0; j < G; ++j) mx[j] = x[j];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int j = 0; j < G; ++j) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], o));
          }
          if (lane < G) {
            float v = mx[0];
#pragma unroll
            for (int j = 1; j < G; ++j) v = (lane == j) ? mx[j] : v;
            redb[lane * 4 + warp] = v;
          }
        }
        ok = named_bar_and(kBarSoft, kSoftThreads, ok);
        if (!ok) break;
        bool need = false;
        float corr[G], tm[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float4 v = *reinterpret_cast<const float4*>(redb + j * 4);
          tm[j] = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
          need |= tm[j] > m[j] + kRescaleLog2;
          corr[j] = 1.f;
        }
        if (need) {  // uniform: every thread read the same maxima
#pragma unroll
          for (int j = 0; j < G; ++j) {
            const float mn = fmaxf(m[j], tm[j]);
            corr[j] = ex2_approx(m[j] - mn);  // 0 when m was -inf
            m[j] = mn;
          }
        }
        // ---- probabilities; P^T buffer (t & 1) is free once P.V of tile t-2 has completed
        if (t >= 2) ok = mbar_wait(o_done + (t & 1), ((t >> 1) - 1) & 1, lim, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        uint8_t* pb = sP + (t & 1) * kOpBytes;
        if (ok) {
#pragma unroll
          for (int j = 0; j < G; ++j) {
            const __nv_bfloat16 pq = __float2bfloat16_rn(ex2_approx(x[j] - m[j]));
            l[j] = fmaf(l[j], corr[j], __bfloat162float(pq));
            *reinterpret_cast<__nv_bfloat16*>(pb + op_off(j, r)) = pq;
          }
          if (n < kRows) {
            // Rows past the segment end hold whatever the cache holds there: zero their V rows so 0 * V stays 0.
            // Rows n..127 of each 64-dim half are one contiguous block: consecutive 16-byte stores, no conflicts.
            ok = mbar_wait(v_full + st, (t / kStages) & 1, lim, abort_flag);
            if (ok) {
              const int nchunk = (kRows - n) * 8;  // 16-byte chunks per half
              uint4* v0 = reinterpret_cast<uint4*>(sV + st * kTileBytes + n * 128);
              uint4* v1 = reinterpret_cast<uint4*>(sV + st * kTileBytes + kHalfBytes + n * 128);
              for (int k = r; k < nchunk; k += kSoftThreads) {
                v0[k] = make_uint4(0, 0, 0, 0);
                v1[k] = make_uint4(0, 0, 0, 0);
              }
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok && need && !first) {
          // Rescale O^T (lane r = dim r, column j = head j) once P.V of tile t-1 has completed.
          ok = mbar_wait(o_done + ((t - 1) & 1), ((t - 1) >> 1) & 1, lim, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after_sync();
            uint32_t ov[16];
            tmem_ld16(tO, ov);
            tmem_ld_wait16(ov);
#pragma unroll
            for (int j = 0; j < G; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * corr[j]);
            tmem_st16(tO, ov);
            tmem_st_wait();
          }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(p_full + (t & 1));
        // (a failure after the barrier above is seen by every thread at the next barrier: the waits return false
        // once any thread has raised the abort flag)

        if (last) {
          // ---- hand (m, row sums) of the finished segment to the epilogue warps
          const int hs = seg % kOBufs;
          if (seg >= kOBufs) ok = mbar_wait(seg_free + hs, ((seg / kOBufs) - 1) & 1, lim, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          float ls[G];
#pragma unroll
          for (int j = 0; j < G; ++j) ls[j] = l[j];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int j = 0; j < G; ++j) ls[j] += __shfl_xor_sync(0xffffffffu, ls[j], off);
          }
          if (lane < G) {
            float v = ls[0], mv = m[0];
#pragma unroll
            for (int j = 1; j < G; ++j) {
              v = (lane == j) ? ls[j] : v;
              mv = (lane == j) ? m[j] : mv;
            }
            seg_l[(hs * kN + lane) * 4 + warp] = v;
            if (warp == 0) seg_m[hs * kN + lane] = mv;
          }
          named_bar_sync(kBarSoft, kSoftThreads);
          if (r == 0) mbar_arrive(seg_ready + hs);
        }
        cu.advance(p, lens_s);
      }
    }
  } else {
    if (ntiles > 0) {
      // ---------------------------------------------------------------- segment epilogue (warps 8-11)
      const int r = tid - kEpiWarp0 * 32;  // dim r = TMEM lane r
      const uint32_t lane_base = static_cast<uint32_t>((warp - kEpiWarp0) * 32) << 16;
      const int ew = warp - kEpiWarp0;
      Cursor cu = cur0;
      int seg = -1;
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t == 0 || cu.i == 0) ++seg;
        if (!(t == ntiles - 1 || cu.i == cu.s.nt - 1)) {
          cu.advance(p, lens_s);
          continue;
        }
        const int hs = seg % kOBufs;
        // ---- O^T and (m, l) of segment `seg`
        ok = mbar_wait(o_full + hs, (seg / kOBufs) & 1, lim, abort_flag);
        ok = ok && mbar_wait(seg_ready + hs, (seg / kOBufs) & 1, lim, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        float o[G], M[G], L[G];
        if (ok) {
          tc_fence_after_sync();
          uint32_t ov[16];
          tmem_ld16(tbase + lane_base + kColO + hs * kN, ov);
          tmem_ld_wait16(ov);
#pragma unroll
          for (int j = 0; j < G; ++j) {
            o[j] = __uint_as_float(ov[j]);
            M[j] = seg_m[hs * kN + j];
            const float4 v = *reinterpret_cast<const float4*>(seg_l + (hs * kN + j) * 4);
            L[j] = (v.x + v.y) + (v.z + v.w);
          }
          tc_fence_before_sync();
        }
        if (!named_bar_and(kBarEpi, 128, ok)) break;
        if (r == 0) {
          mbar_arrive(o_free + hs);    // the MMA may now overwrite this O buffer
          mbar_arrive(seg_free + hs);  // the softmax may now reuse this hand-over slot
        }

        const int b = cu.b, g = cu.g;
        const long long s0 = cu.seg_tile0(p.Hkv);
        const int c_first = tile_owner(s0, N, C);
        const int c_last = tile_owner(s0 + cu.s.nt - 1, N, C);
        bool finish = (c_first == c_last);
        if (!finish) {
          const int my_slot = (c * 2 + ((t_begin >= s0) ? 0 : 1)) * G;
          // Partial slots of the segment's parts, -1 for CTAs whose range is empty.
          for (int cc = c_first + r; cc <= c_last; cc += 128)
            part_slot[cc - c_first] =
                range_empty(cc, N, C) ? -1 : (cc * 2 + (range_begin(cc, N, C) >= s0 ? 0 : 1)) * G;
          named_bar_sync(kBarEpi, 128);
          unsigned* cnt = p.ws_cnt + static_cast<size_t>(b) * p.Hkv + g;
          unsigned nparts = 0;
          for (int k = 0; k <= c_last - c_first; ++k) nparts += part_slot[k] >= 0 ? 1u : 0u;
          // When every other part has already arrived, this CTA is the last one: it merges its own partial from
          // registers and need not publish it.
          if (r == 0) *last_flag = (ld_acquire_gpu(cnt) == nparts - 1u) ? 2 : 0;
          named_bar_sync(kBarEpi, 128);
          bool self_in_regs = *last_flag == 2;
          if (!self_in_regs) {
            // Publish this CTA's partial; the last CTA of the segment to arrive merges.
#pragma unroll
            for (int j = 0; j < G; ++j) {
              p.ws_o[(static_cast<size_t>(my_slot) + j) * 128 + r] = o[j];
              if (r == j) {
                p.ws_ml[(static_cast<size_t>(my_slot) + j) * 2] = M[j];
                p.ws_ml[(static_cast<size_t>(my_slot) + j) * 2 + 1] = L[j];
              }
            }
            // The barrier orders every thread's partial before thread 0's release; its acquire (when last) orders
            // the other parts' partials before every thread's reads after the next barrier.
            named_bar_sync(kBarEpi, 128);
            if (r == 0) *last_flag = (atom_add_acq_rel_gpu(cnt, 1u) == nparts - 1u) ? 1 : 0;
            named_bar_sync(kBarEpi, 128);
          }
          finish = *last_flag != 0;
          if (finish) {
            // Online log-sum-exp merge over the parts, always in part order (whichever CTA arrives last merges), so
            // that the result does not depend on the arrival order.  The loads of one part are independent of each
            // other; this CTA's own part comes from registers when it did not publish it.
            float own_m[G], own_l[G], own_o[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
              own_m[j] = M[j];
              own_l[j] = L[j];
              own_o[j] = o[j];
              M[j] = -INFINITY;
              L[j] = 0.f;
              o[j] = 0.f;
            }
            for (int k = 0; k <= c_last - c_first; ++k) {
              const int sl = part_slot[k];
              if (sl < 0) continue;
              const bool own = self_in_regs && sl == my_slot;
              float pm[G], pl[G], po[G];
#pragma unroll
              for (int j = 0; j < G; ++j) {
                pm[j] = own ? own_m[j] : __ldcg(p.ws_ml + (static_cast<size_t>(sl) + j) * 2);
                pl[j] = own ? own_l[j] : __ldcg(p.ws_ml + (static_cast<size_t>(sl) + j) * 2 + 1);
                po[j] = own ? own_o[j] : __ldcg(p.ws_o + (static_cast<size_t>(sl) + j) * 128 + r);
              }
#pragma unroll
              for (int j = 0; j < G; ++j) {
                const float mn = fmaxf(M[j], pm[j]);
                const float a = ex2_approx(M[j] - mn), w = ex2_approx(pm[j] - mn);
                L[j] = fmaf(L[j], a, pl[j] * w);
                o[j] = fmaf(o[j], a, po[j] * w);
                M[j] = mn;
              }
            }
            if (r == 0) *cnt = 0u;  // leave the counter zero for the next call
          }
        }
        if (finish) {
          __nv_bfloat16* outg = p.out + (static_cast<size_t>(b) * p.Hq + g * G) * 128;
          if (has_new) {
            // The new key joins as one more key: roped + normed at p, written to cache row p with v_new.
            const size_t crow = ((static_cast<size_t>(b) * p.Tcap + cu.s.pos) * p.Hkv + g) * 128;
            if (ew == 0) {
              float y[4], cs[2], sn[2];
              warp_rope_angles(static_cast<float>(cu.s.pos), tab, lane, cs, sn);
              warp_rope_norm(p.k_new + (static_cast<size_t>(b) * p.Hkv + g) * 128, cs, sn, lane, y);
              const uint32_t w0 = pack_bf16x2(y[0], y[1]), w1 = pack_bf16x2(y[2], y[3]);
              reinterpret_cast<uint32_t*>(p.kcache + crow)[lane] = w0;
              reinterpret_cast<uint32_t*>(p.kcache + crow + 64)[lane] = w1;
              new_k[2 * lane] = bf16_lo(w0);
              new_k[2 * lane + 1] = bf16_hi(w0);
              new_k[64 + 2 * lane] = bf16_lo(w1);
              new_k[65 + 2 * lane] = bf16_hi(w1);
            } else if (ew == 1) {
              const uint2 vv = new_value4(p, b, g, lane);
              reinterpret_cast<uint2*>(p.vcache + crow)[lane] = vv;
              new_v[4 * lane] = bf16_lo(vv.x);
              new_v[4 * lane + 1] = bf16_hi(vv.x);
              new_v[4 * lane + 2] = bf16_lo(vv.y);
              new_v[4 * lane + 3] = bf16_hi(vv.y);
            }
            named_bar_sync(kBarEpi, 128);
            const uint8_t* qs = sQ + (seg % kQSlots) * kOpBytes;
            for (int j = ew; j < G; j += 4) {
              float a = 0.f;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int d = 4 * lane + k;
                a = fmaf(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(qs + op_off(j, d))), new_k[d], a);
              }
              a = warp_sum(a);
              if (lane == 0) s_new[j] = a * p.scale_log2;
            }
            named_bar_sync(kBarEpi, 128);
            const float vd = new_v[r];
#pragma unroll
            for (int j = 0; j < G; ++j) {
              const float sn = s_new[j];
              const float Mx = fmaxf(M[j], sn);
              const float a = ex2_approx(M[j] - Mx), w = ex2_approx(sn - Mx);
              outg[j * 128 + r] = __float2bfloat16_rn(fmaf(o[j], a, w * vd) / fmaf(L[j], a, w));
            }
          } else {
#pragma unroll
            for (int j = 0; j < G; ++j) outg[j * 128 + r] = __float2bfloat16_rn(o[j] / L[j]);
          }
        }
        // The Q slot of this segment is free again; the scratch above may be reused by the next epilogue.
        named_bar_sync(kBarEpi, 128);
        if (r == 0) mbar_arrive(q_empty + seg % kQSlots);
        cu.advance(p, lens_s);
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace dec
}  // namespace nc
