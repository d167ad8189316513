// K5: backward pass of the attention block on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: the gradients of sum(dout * out) with respect to the raw q, k and v of the prefill forward
// (out = attention(norm(rope(q)), norm(rope(k)), v), causal with the window, logits scaled by qk_gain / sqrt(D),
// contiguous GQA groups; "nanochat Admin & Developer Guide", section 3 -- the model trains through this block).
// The chain rule, per (b, query head h, kv head g = h / G), with P = softmax(S), O = P V, c = qk_gain / sqrt(D):
//   dV_g += P^T dO,  dP = dO V_g^T,  dS = P * (dP - rowsum(dO * O)),  dqn_h = c dS kn_g,  dkn_g += c dS^T qn_h;
// then the RMSNorm backward dx = (dy - yn (dy . yn) / D) / r (r the forward's RMS, eps included) and the RoPE
// backward, the rotation of each pair (i, i + D/2) by -t theta_i.
//
// The launches of one backward call (nc_attn_bwd_ws):
//   1. the forward prologue (K1): qn' = qn c log2(e) and kn in bf16, exactly as the forward uses them;
//   2. the forward attention kernel (K2) in its statistics mode: per query row the base-2 log-sum-exp of its logits
//      and rowsum(dO * O) (O in fp32 before rounding), nothing else stored;
//   3. bwd_kernel<false> (dK, dV): a work item is one 128-key tile of one (b, kv head); K and V stay in shared memory
//      while the packed Q tiles (P = 128 / G positions x the G heads of the group, as in the forward) and dO tiles
//      that see the keys stream through a 2-stage TMA ring.  Per Q tile:  S^T = K Q'^T and dP^T = V dO^T (tcgen05,
//      fp32 in TMEM), P^T = 2^(S^T - lse) and dS^T = P^T (dP^T - rowsum) on the CUDA cores (bf16, back into TMEM over
//      S^T and dP^T), then dV += P^T dO and dK += dS^T Q' (A from TMEM, B = the streamed tiles read MN-major);
//   4. bwd_kernel<true> (dQ): a work item is one packed Q tile; Q' and dO stay, K and V tiles of its band stream.
//      Per key tile: S = Q' K^T, dP = dO V^T, P and dS on the CUDA cores, dQ += dS K;
//   5. bwd_norm_rope_kernel: the RMSNorm and RoPE backward of every dq and dk row, in place (memory-bound).
// Step 4 recomputes S and dP (7 products per (key tile, Q tile) pair instead of 5) so that every gradient is written
// by exactly one CTA: no atomics, and the result does not depend on the schedule.
//
// Scales: the products use qn' (base-2 logits, as in the forward), so dK = dS^T Q' carries a factor c log2(e): dkn =
// ln 2 dK; dqn = c dQ with dQ = dS kn.  The probabilities and dS are rounded to bf16 for the tensor core, like P in
// the forward; every accumulation is fp32.
#pragma once

#include <climits>

#include "common.cuh"

namespace nc {
namespace bwd {

// ---- the RMSNorm + RoPE backward -----------------------------------------------------------------------------
// The RMSNorm + RoPE backward of every q and k head vector, token-major like the forward prologue: an 8-lane group per
// token, lane kq owning the pairs [8 kq, 8 kq + 8) (elements [8 kq, 8 kq + 8) and [64 + 8 kq, 64 + 8 kq + 8)) of every
// head, so that a pair sits in one lane and the cos / sin of the token are computed once for its Hq + Hkv heads.  dq
// and dk hold the gradients with respect to the normed vectors; each is replaced in place by the gradient with respect
// to the raw vector: yn and r recomputed from the raw bf16 input in fp32, dx = (dy - yn (dy . yn) / D) / r, then the
// rotation by -angle.  Sums over a head vector are reduced across the group with xor-shuffles.
constexpr int kPostThreads = 256;
constexpr int kPostTokensPerBlock = kPostThreads / 8;

__device__ __forceinline__ void norm_rope_bwd_head(const __nv_bfloat16* __restrict__ x_raw, float* __restrict__ g,
                                                   int kq, const float (&c)[8], const float (&s)[8], unsigned gmask) {
  const uint4 lo = __ldg(reinterpret_cast<const uint4*>(x_raw) + kq);
  const uint4 hi = __ldg(reinterpret_cast<const uint4*>(x_raw) + 8 + kq);
  float4* gl = reinterpret_cast<float4*>(g + 8 * kq);
  float4* gh = reinterpret_cast<float4*>(g + 64 + 8 * kq);
  const float4 d0 = gl[0], d1 = gl[1], d2 = gh[0], d3 = gh[1];
  const float dy1[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
  const float dy2[8] = {d2.x, d2.y, d2.z, d2.w, d3.x, d3.y, d3.z, d3.w};
  const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w}, b[4] = {hi.x, hi.y, hi.z, hi.w};
  float y1[8], y2[8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float x1 = (i & 1) ? bf16_hi(a[i >> 1]) : bf16_lo(a[i >> 1]);
    const float x2 = (i & 1) ? bf16_hi(b[i >> 1]) : bf16_lo(b[i >> 1]);
    y1[i] = fmaf(x1, c[i], x2 * s[i]);
    y2[i] = fmaf(x2, c[i], -(x1 * s[i]));
    ss = fmaf(y1[i], y1[i], fmaf(y2[i], y2[i], ss));
  }
  ss += __shfl_xor_sync(gmask, ss, 1);
  ss += __shfl_xor_sync(gmask, ss, 2);
  ss += __shfl_xor_sync(gmask, ss, 4);
  const float inv_r = rsqrtf(ss * (1.0f / 128.0f) + kRmsEps);
  float pr = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    y1[i] *= inv_r;
    y2[i] *= inv_r;
    pr = fmaf(dy1[i], y1[i], fmaf(dy2[i], y2[i], pr));
  }
  pr += __shfl_xor_sync(gmask, pr, 1);
  pr += __shfl_xor_sync(gmask, pr, 2);
  pr += __shfl_xor_sync(gmask, pr, 4);
  pr *= 1.0f / 128.0f;
  float o1[8], o2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float e1 = (dy1[i] - y1[i] * pr) * inv_r, e2 = (dy2[i] - y2[i] * pr) * inv_r;
    // transpose of the forward rotation (y1 = x1 c + x2 s, y2 = -x1 s + x2 c)
    o1[i] = fmaf(e1, c[i], -(e2 * s[i]));
    o2[i] = fmaf(e2, c[i], e1 * s[i]);
  }
  gl[0] = make_float4(o1[0], o1[1], o1[2], o1[3]);
  gl[1] = make_float4(o1[4], o1[5], o1[6], o1[7]);
  gh[0] = make_float4(o2[0], o2[1], o2[2], o2[3]);
  gh[1] = make_float4(o2[4], o2[5], o2[6], o2[7]);
}

__global__ void __launch_bounds__(kPostThreads)
    bwd_norm_rope_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, float* dq,
                         float* dk, int BT, int T, int Hq, int Hkv, const __grid_constant__ RopeTable tab) {
  const int tok = blockIdx.x * kPostTokensPerBlock + (threadIdx.x >> 3);
  const int kq = threadIdx.x & 7;
  if (tok >= BT) return;  // whole 8-lane groups leave together
  const unsigned gmask = 0xFFu << ((threadIdx.x & 31) & ~7);
  const float pos = static_cast<float>(tok % T);
  float c[8], s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rope_cos_sin(pos, tab.hi[kq * 8 + i], tab.lo[kq * 8 + i], c[i], s[i]);
  for (int h = 0; h < Hq; ++h)
    norm_rope_bwd_head(q + (static_cast<size_t>(tok) * Hq + h) * 128, dq + (static_cast<size_t>(tok) * Hq + h) * 128,
                       kq, c, s, gmask);
  for (int h = 0; h < Hkv; ++h)
    norm_rope_bwd_head(k + (static_cast<size_t>(tok) * Hkv + h) * 128,
                       dk + (static_cast<size_t>(tok) * Hkv + h) * 128, kq, c, s, gmask);
}

// ---- rowsum(dO * O) from a kept forward output ---------------------------------------------------------------------
// For a backward that reuses the forward's output and log-sum-exp instead of recomputing them: the rowsum of dout *
// out (both bf16) of every packed query row, in the layout the tcgen05 kernels read -- row r of Q tile m of (b, kv
// head g) is position m P + r / G of query head g G + r % G, and rows that hold no query get 0.  One 8-lane group
// per row, 16 elements per lane; memory-bound.
constexpr int kDrowThreads = 256;
__global__ void __launch_bounds__(kDrowThreads)
    drow_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout, float* __restrict__ drow,
                int T, int Hq, int Hkv, int G, int P, int n_qtiles, long long n_rows) {
  const long long row = static_cast<long long>(blockIdx.x) * (kDrowThreads / 8) + (threadIdx.x >> 3);
  const int kq = threadIdx.x & 7;
  if (row >= n_rows) return;  // whole 8-lane groups leave together
  const unsigned gmask = 0xFFu << ((threadIdx.x & 31) & ~7);
  const int r = static_cast<int>(row & 127);
  const long long tile_row = row >> 7;
  const int m = static_cast<int>(tile_row % n_qtiles);
  const long long bg = tile_row / n_qtiles;
  const int g = static_cast<int>(bg % Hkv);
  const long long b = bg / Hkv;
  const int t = m * P + r / G;
  float acc = 0.f;
  if (r < G * P && t < T) {
    const size_t off = ((static_cast<size_t>(b) * T + t) * Hq + g * G + r % G) * 128;
    const uint4* o4 = reinterpret_cast<const uint4*>(out + off);
    const uint4* d4 = reinterpret_cast<const uint4*>(dout + off);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 a = __ldg(o4 + kq + 8 * u), d = __ldg(d4 + kq + 8 * u);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(bf16_lo(aw[e]), bf16_lo(dw[e]), acc);
        acc = fmaf(bf16_hi(aw[e]), bf16_hi(dw[e]), acc);
      }
    }
  }
  acc += __shfl_xor_sync(gmask, acc, 1);
  acc += __shfl_xor_sync(gmask, acc, 2);
  acc += __shfl_xor_sync(gmask, acc, 4);
  if (kq == 0) drow[row] = acc;
}

// ---- tcgen05 kernels ---------------------------------------------------------------------------------------------
constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr int kHalfBytes = 128 * 128;        // one 64-column half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalfBytes;   // 32 KB
constexpr int kEwWarps = 8;                  // warps 0-7: elementwise step and epilogue
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kRegsEw = 208, kRegsOther = 88;  // 2 x 128 x 208 + 128 x 88 = 384 x 168
constexpr uint32_t kTmemCols = 512;
// TMEM: X = S^T / P^T (dK,dV) or S (dQ); Y = dP^T / dS^T or dP / dS; accumulators dK, dV (dK,dV), or dQ of the even
// and of the odd items (dQ: the epilogue of one item overlaps the next item's first step).
constexpr uint32_t kColX = 0, kColY = 128, kColAcc0 = 256, kColAcc1 = 384;

// Accumulator buffer of the k-th item of a CTA and the phase of its barriers: the dQ kernel alternates two buffers.
template <bool kDQ>
__device__ __forceinline__ int acc_buf(int k) { return kDQ ? (k & 1) : 0; }
template <bool kDQ>
__device__ __forceinline__ uint32_t acc_phase(int k) { return kDQ ? ((k >> 1) & 1) : (k & 1); }
constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false, false);  // A, B both K-major (smem)
constexpr uint32_t kIdescTM = idesc_bf16_f32(128, 128, false, true);   // A from TMEM, B MN-major (smem)

// Shared memory: A1, A2 (resident per item), kStages x (B1, B2), kStages slots of the (lse, rowsum) vectors of the
// streamed Q tiles (dK,dV kernel; 128 + 128 floats each), barriers, scheduler slots.
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + 2 * kTileBytes;
constexpr int kOffVec = kOffB + kStages * 2 * kTileBytes;
constexpr int kVecBytes = 2 * 128 * 4;
constexpr int kOffBar = kOffVec + kStages * kVecBytes;
constexpr int kBarAFull = 0;
constexpr int kBarAEmpty = 1;
constexpr int kBarBFull = 2;                          // [kStages]
constexpr int kBarBEmpty = kBarBFull + kStages;       // [kStages]
constexpr int kBarXFull = kBarBEmpty + kStages;
constexpr int kBarYFull = kBarXFull + 1;
constexpr int kBarPFull = kBarYFull + 1;
constexpr int kBarDsFull = kBarPFull + 1;
constexpr int kBarAccDone = kBarDsFull + 1;           // [2]: accumulator buffer
constexpr int kBarAccFree = kBarAccDone + 2;          // [2]
constexpr int kBarSchedFull = kBarAccFree + 2;        // [2]
constexpr int kBarSchedEmpty = kBarSchedFull + 2;     // [2]
constexpr int kBarMmaFinal = kBarSchedEmpty + 2;
constexpr int kNumBars = kBarMmaFinal + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kAlignSlack = 768;
constexpr int kSmemBytes = kOffMisc + 32 + kAlignSlack;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  float* dst_a;        // dK,dV kernel: dk rows (gradient w.r.t. kn); dQ kernel: dq rows (w.r.t. qn)
  float* dst_b;        // dK,dV kernel: dv rows; dQ kernel: unused
  const float* lse;    // [B, Hkv, n_qtiles, 128]: base-2 log-sum-exp of every packed query row
  const float* drow;   // same layout: rowsum(dO * O)
  unsigned* item_ctr;  // zero at launch
  int B, T, Hq, Hkv, G, P, n_qtiles, n_ktiles, n_items;
  int window;          // -1: unbounded (the host maps windows >= T to -1)
  float scale_a;       // factor on the dst_a accumulator: ln 2 (dK) or qk_gain / sqrt(128) (dQ)
  unsigned long long wait_limit_ns;
};

struct Item {
  int b, g;
  int tile;    // key tile (dK,dV) or Q tile (dQ) of the item
  int lo, hi;  // streamed tiles: Q tiles (dK,dV) or key tiles (dQ)
};

template <bool kDQ>
__device__ __forceinline__ Item decode_item(const Params& p, int item) {
  Item it;
  const int bh = p.B * p.Hkv;
  const int ord = item / bh;
  const int bg = item - ord * bh;
  it.b = bg / p.Hkv;
  it.g = bg - it.b * p.Hkv;
  if (!kDQ) {
    // key tile ord: queries at positions [128 ord, min(T - 1, 128 ord + 127 + window)] see its keys; under a causal
    // mask the first key tiles are seen by the most queries, so they come first
    it.tile = ord;
    const int k0 = ord * 128;
    const int last = p.window < 0 ? p.T - 1 : min(p.T - 1, k0 + 127 + p.window);
    it.lo = k0 / p.P;
    it.hi = last / p.P;
  } else {
    // Q tile n_qtiles - 1 - ord (latest, heaviest first): keys [max(0, t0 - window), t_last]
    it.tile = p.n_qtiles - 1 - ord;
    const int t0 = it.tile * p.P;
    const int t_last = min(t0 + p.P, p.T) - 1;
    it.lo = (p.window < 0 ? 0 : max(0, t0 - p.window)) / 128;
    it.hi = t_last / 128;
  }
  return it;
}

// 32-column visibility mask of the column interval [lo, hi] within columns [c0, c0 + 32).
__device__ __forceinline__ uint32_t interval_mask(int lo, int hi, int c0) {
  const int a = lo - c0, b = hi - c0;
  const uint32_t m_hi = b >= 31 ? ~0u : (b < 0 ? 0u : (2u << b) - 1u);
  const uint32_t m_lo = a <= 0 ? ~0u : (a > 31 ? 0u : ~((1u << a) - 1u));
  return m_hi & m_lo;
}

// kDQ = false: dK and dV; kDQ = true: dQ.  Maps: tmQ = qn' and tmDO = dout ([B, T, Hq, 128], box {64, G, P, 1}),
// tmK = kn and tmV = v ([B, T, Hkv, 128], box {64, 1, 128, 1}); all bf16, 128-byte swizzle.
template <bool kDQ>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  float* sVec = reinterpret_cast<float*>(smem + kOffVec);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_full = bars + kBarAFull;        // A1, A2 (and the dQ item's vectors) landed       TMA -> MMA, ew
  uint64_t* a_empty = bars + kBarAEmpty;      // every product reading A1, A2 done                MMA -> TMA
  uint64_t* b_full = bars + kBarBFull;        // [kStages] B1, B2 (and the dK,dV vectors) landed  TMA -> MMA, ew
  uint64_t* b_empty = bars + kBarBEmpty;      // [kStages] every product reading the stage done   MMA -> TMA
  uint64_t* x_full = bars + kBarXFull;        // X = A1 B1^T in TMEM                              MMA -> ew
  uint64_t* y_full = bars + kBarYFull;        // Y = A2 B2^T in TMEM                              MMA -> ew
  uint64_t* p_full = bars + kBarPFull;        // X consumed: P^T over it (dK,dV) or read (dQ); per warp ew -> MMA
  uint64_t* ds_full = bars + kBarDsFull;      // dS written over Y (one arrival per warp)         ew -> MMA
  uint64_t* acc_done = bars + kBarAccDone;    // [2] the item's last accumulation complete        MMA -> ew
  uint64_t* acc_free = bars + kBarAccFree;    // [2] accumulators read by the epilogue (per warp) ew -> MMA
  uint64_t* sched_full = bars + kBarSchedFull;
  uint64_t* sched_empty = bars + kBarSchedEmpty;
  uint64_t* mma_final = bars + kBarMmaFinal;
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;
  int* sched = misc + 2;  // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned long long lim = p.wait_limit_ns;
  if (static_cast<int>(smem - smem_raw) > kAlignSlack) {
    if (threadIdx.x == 0) raise_status(NC_DEV_SMEM_BASE);
    return;
  }
  const int GP = p.G * p.P;  // rows of a packed Q tile that hold queries
  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(b_full + s, 1);
      mbar_init(b_empty + s, 1);
    }
    mbar_init(x_full, 1);
    mbar_init(y_full, 1);
    mbar_init(p_full, kEwWarps);
    mbar_init(ds_full, kEwWarps);
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_done + s, 1);
      mbar_init(acc_free + s, kEwWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sched_full + s, 1);
      mbar_init(sched_empty + s, 2);
    }
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (GP < 128 && threadIdx.x < 256) {
    // Rows of the packed Q / dO tiles that TMA never fills (128 is not a multiple of G) are zeroed once, so that a
    // zero probability never meets a non-finite value in a product.  dQ: the resident A tiles; dK,dV: every stage.
    const int r = threadIdx.x & 127;
    if (r >= GP) {
      const int nbuf = kDQ ? 2 : 2 * kStages;
      for (int bi = (threadIdx.x >> 7); bi < nbuf; bi += 2) {
        uint8_t* base = (kDQ ? sA : sB) + bi * kTileBytes;
        uint4* r0 = reinterpret_cast<uint4*>(base + r * 128);
        uint4* r1 = reinterpret_cast<uint4*>(base + kHalfBytes + r * 128);
        for (int i = 0; i < 8; ++i) {
          r0[i] = make_uint4(0, 0, 0, 0);
          r1[i] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t q_bytes = 2u * 128u * static_cast<uint32_t>(GP);  // one packed Q or dO tile: box {64, G, P, 1} x 2

  if (warp >= kEwWarps) {
    warpgroup_reg_dec<kRegsOther>();
    if (warp == kProducerWarp && lane == 0) {
      // ---------------------------------------------------------------- scheduler + TMA producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int nb = 0;   // B stages filled so far
      int na = 0;   // A fills so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (k >= 2 && !(ok = mbar_wait(sched_empty + slot, ((k >> 1) - 1) & 1, lim, abort_flag))) break;
        const int item = static_cast<int>(atomicAdd(p.item_ctr, 1u));
        sched[slot] = item < p.n_items ? item : -1;
        mbar_arrive(sched_full + slot);
        if (item >= p.n_items) break;
        const Item it = decode_item<kDQ>(p, item);
        // A tiles once every product of the previous item that reads them has completed
        if (na > 0 && !(ok = mbar_wait(a_empty, (na - 1) & 1, lim, abort_flag))) break;
        if (!kDQ) {
          mbar_arrive_expect_tx(a_full, 2 * kTileBytes);
          tma_load_4d(sA, &tmK, a_full, 0, it.g, it.tile * 128, it.b);
          tma_load_4d(sA + kHalfBytes, &tmK, a_full, 64, it.g, it.tile * 128, it.b);
          tma_load_4d(sA + kTileBytes, &tmV, a_full, 0, it.g, it.tile * 128, it.b);
          tma_load_4d(sA + kTileBytes + kHalfBytes, &tmV, a_full, 64, it.g, it.tile * 128, it.b);
        } else {
          const int t0 = it.tile * p.P;
          mbar_arrive_expect_tx(a_full, 2 * q_bytes);
          tma_load_4d(sA, &tmQ, a_full, 0, it.g * p.G, t0, it.b);
          tma_load_4d(sA + kHalfBytes, &tmQ, a_full, 64, it.g * p.G, t0, it.b);
          tma_load_4d(sA + kTileBytes, &tmDO, a_full, 0, it.g * p.G, t0, it.b);
          tma_load_4d(sA + kTileBytes + kHalfBytes, &tmDO, a_full, 64, it.g * p.G, t0, it.b);
        }
        ++na;
        for (int j = it.lo; ok && j <= it.hi; ++j, ++nb) {
          const int st = nb % kStages;
          if (nb >= kStages && !(ok = mbar_wait(b_empty + st, ((nb / kStages) - 1) & 1, lim, abort_flag))) break;
          uint8_t* b1 = sB + (2 * st) * kTileBytes;
          uint8_t* b2 = b1 + kTileBytes;
          if (!kDQ) {
            const int t0 = j * p.P;
            const size_t vi = ((static_cast<size_t>(it.b) * p.Hkv + it.g) * p.n_qtiles + j) * 128;
            mbar_arrive_expect_tx(b_full + st, 2 * q_bytes + kVecBytes);
            tma_load_4d(b1, &tmQ, b_full + st, 0, it.g * p.G, t0, it.b);
            tma_load_4d(b1 + kHalfBytes, &tmQ, b_full + st, 64, it.g * p.G, t0, it.b);
            tma_load_4d(b2, &tmDO, b_full + st, 0, it.g * p.G, t0, it.b);
            tma_load_4d(b2 + kHalfBytes, &tmDO, b_full + st, 64, it.g * p.G, t0, it.b);
            bulk_load(sVec + st * 256, p.lse + vi, 512, b_full + st);
            bulk_load(sVec + st * 256 + 128, p.drow + vi, 512, b_full + st);
          } else {
            mbar_arrive_expect_tx(b_full + st, 2 * kTileBytes);
            tma_load_4d(b1, &tmK, b_full + st, 0, it.g, j * 128, it.b);
            tma_load_4d(b1 + kHalfBytes, &tmK, b_full + st, 64, it.g, j * 128, it.b);
            tma_load_4d(b2, &tmV, b_full + st, 0, it.g, j * 128, it.b);
            tma_load_4d(b2 + kHalfBytes, &tmV, b_full + st, 64, it.g, j * 128, it.b);
          }
        }
      }
      // every copy this CTA started lands before the CTA exits (already true on the normal path)
      for (int t = max(0, nb - kStages); t < nb; ++t) mbar_wait(b_full + t % kStages, (t / kStages) & 1, lim, nullptr);
      if (na > 0) mbar_wait(a_full, (na - 1) & 1, lim, nullptr);
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------------- MMA issuer (lane 0; the warp waits together)
      const bool leader = lane == 0;
      const uint32_t aA = smem_u32(sA), aB = smem_u32(sB);
      constexpr uint64_t kTileDesc = kTileBytes >> 4;
      const uint64_t dA = sdesc_sw128(aA, 16, 1024);            // K-major: A1 at +0, A2 at +1 tile
      const uint64_t dBk = sdesc_sw128(aB, 16, 1024);           // K-major view of the B tiles
      const uint64_t dBm = sdesc_sw128(aB, kHalfBytes, 1024);   // MN-major view of the B tiles
      const uint32_t tX = tbase + kColX, tY = tbase + kColY, tAcc0 = tbase + kColAcc0, tAcc1 = tbase + kColAcc1;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, lim, abort_flag));
      };
      auto commit = [&](uint64_t* bar) {
        if (leader) umma_commit(bar);
        __syncwarp();
      };
      // D (tmem) = A (smem tile ai) B (smem tile bi)^T, both K-major
      auto mma_kk = [&](uint32_t d, int ai, int bi) {
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
            umma_ss(d, dA + ai * kTileDesc + off, dBk + bi * kTileDesc + off, kIdescKK, kk > 0 ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      // D (tmem) (+)= A (bf16 pairs in tmem, half h's columns at [64 h, 64 h + 32)) B (smem tile bi, MN-major)
      auto mma_tm = [&](uint32_t d, uint32_t a, int bi, uint32_t acc0) {
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(d, a + (kk >> 2) * 64 + (kk & 3) * 8,
                    dBm + bi * kTileDesc + static_cast<uint64_t>((kk * 2048) >> 4), kIdescTM, kk > 0 ? 1u : acc0);
        }
        __syncwarp();
      };
      int nb = 0, ns = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!(ok = wait(sched_full + slot, (k >> 1) & 1))) break;
        const int item = sched[slot];
        __syncwarp();
        if (leader) mbar_arrive(sched_empty + slot);
        if (item < 0) break;
        const Item it = decode_item<kDQ>(p, item);
        if (!(ok = wait(a_full, k & 1))) break;
        // Products of a step (B stage st: b1 = Q' / K tile, b2 = dO / V tile):
        //   X = A1 b1^T (dK,dV: S^T = K Q'^T; dQ: S = Q' K^T),  Y = A2 b2^T (dP^T = V dO^T; dP = dO V^T),
        //   dK,dV: dV += P^T dO (A = X) and dK += dS^T Q' (A = Y);  dQ: dQ += dS K (A = Y).
        // The next step's X goes in as soon as this step's X has been consumed (P^T written over it, or read), and
        // its Y right after the product that reads this step's dS: the tensor core runs them while the elementwise
        // warps work on this step's dS and the next step's P.  Products of one thread run in issue order, so a
        // product that overwrites X or Y follows the one that reads it.
        if (!(ok = wait(b_full + nb % kStages, (nb / kStages) & 1))) break;
        tc_fence_after_sync();
        mma_kk(tX, 0, 2 * (nb % kStages));
        commit(x_full);
        mma_kk(tY, 1, 2 * (nb % kStages) + 1);
        commit(y_full);
        if (it.lo == it.hi) commit(a_empty);
        for (int j = it.lo; j <= it.hi; ++j, ++nb, ++ns) {
          const int st = nb % kStages, st1 = (nb + 1) % kStages;
          const int b1 = 2 * st, b2 = 2 * st + 1;
          const bool more = j < it.hi;
          // the accumulators this item reuses (the previous item's, or in the dQ kernel the one before it) must have
          // been read out before the first accumulation
          const int kprev = kDQ ? k - 2 : k - 1;
          if (j == it.lo && kprev >= 0 && !(ok = wait(acc_free + acc_buf<kDQ>(kprev), acc_phase<kDQ>(kprev)))) break;
          const uint32_t acc0 = j > it.lo ? 1u : 0u;
          if (!(ok = wait(p_full, ns & 1))) break;  // X consumed
          if (more && !(ok = wait(b_full + st1, ((nb + 1) / kStages) & 1))) break;
          tc_fence_after_sync();
          if (!kDQ) mma_tm(tAcc1, tX, b2, acc0);  // dV += P^T dO
          if (more) {
            mma_kk(tX, 0, 2 * st1);  // next X
            commit(x_full);
          }
          if (!(ok = wait(ds_full, ns & 1))) break;
          tc_fence_after_sync();
          mma_tm(kDQ ? ((k & 1) ? tAcc1 : tAcc0) : tAcc0, tY, b1, acc0);  // dK += dS^T Q'  /  dQ += dS K
          commit(b_empty + st);
          if (more) {
            mma_kk(tY, 1, 2 * st1 + 1);  // next Y
            commit(y_full);
            if (j + 1 == it.hi) commit(a_empty);
          } else {
            commit(acc_done + acc_buf<kDQ>(k));
          }
        }
      }
      if (leader) umma_commit(mma_final);  // every issued product completes before TMEM is released
      __syncwarp();
      mbar_wait(mma_final, 0, lim, nullptr);
    }
  } else {
    // ------------------------------------------------------------------ elementwise + epilogue (warps 0-7)
    warpgroup_reg_inc<kRegsEw>();
    const int r = threadIdx.x & 127;   // TMEM lane = row of X, Y and the accumulators
    const int h = warp >> 2;           // column half [64 h, 64 h + 64)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tX = tbase + lane_base + kColX, tY = tbase + lane_base + kColY;
    constexpr uint32_t kBarAll = 1;    // named barrier of the 256 elementwise threads
    // ---- epilogue of the k-th item: its accumulators, scaled, to global memory (fp32).  Every elementwise thread
    // calls it at the same point; returns false (for all) when a wait failed.
    auto epilogue = [&](const Item& it, int k) {
      bool fail = !__all_sync(0xffffffffu, mbar_wait(acc_done + acc_buf<kDQ>(k), acc_phase<kDQ>(k), lim, abort_flag));
      if (!named_bar_and(kBarAll, 2 * 128, !fail)) return false;
      tc_fence_after_sync();
      size_t row_off = 0;
      bool store = false;
      if (!kDQ) {
        const int key_row = it.tile * 128 + r;
        store = key_row < p.T;
        row_off = ((static_cast<size_t>(it.b) * p.T + key_row) * p.Hkv + it.g) * 128;
      } else {
        const int t = it.tile * p.P + r / p.G;
        store = r < GP && t < p.T;
        row_off = ((static_cast<size_t>(it.b) * p.T + t) * p.Hq + it.g * p.G + r % p.G) * 128;
      }
#pragma unroll
      for (int a = 0; a < (kDQ ? 1 : 2); ++a) {
        float* dst = (a == 0 ? p.dst_a : p.dst_b) + row_off + 64 * h;
        const float sc = a == 0 ? p.scale_a : 1.f;
        // dK,dV: dK in accumulator 0, dV in 1; dQ: the item's own buffer
        const uint32_t col = kDQ ? ((k & 1) ? kColAcc1 : kColAcc0) : (a == 0 ? kColAcc0 : kColAcc1);
        const uint32_t tacc = tbase + lane_base + col + 64 * h;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t av[32];
          tmem_ld32(tacc + 32 * c2, av);
          tmem_ld_wait(av);
          if (store) {
#pragma unroll
            for (int w = 0; w < 8; ++w)
              reinterpret_cast<float4*>(dst + 32 * c2)[w] =
                  make_float4(__uint_as_float(av[4 * w]) * sc, __uint_as_float(av[4 * w + 1]) * sc,
                              __uint_as_float(av[4 * w + 2]) * sc, __uint_as_float(av[4 * w + 3]) * sc);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_free + acc_buf<kDQ>(k));
      return true;
    };
    int nb = 0, ns = 0;
    bool ok = true;
    Item pending;          // dQ: the item whose epilogue waits for the next item's first step
    int pending_k = -1;
    bool failed = false;   // the same for all 256 threads: set only where a barrier AND has failed for everyone
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(sched_full + slot, (k >> 1) & 1, lim, abort_flag));
      if (!named_bar_and(kBarAll, 2 * 128, ok)) {
        failed = true;
        break;
      }
      const int item = sched[slot];
      named_bar_sync(kBarAll, 2 * 128);
      if (threadIdx.x == 0) mbar_arrive(sched_empty + slot);
      if (item < 0) break;
      const Item it = decode_item<kDQ>(p, item);
      bool fail = false;
      // dQ: this row's query position, log-sum-exp and rowsum, read from global memory (written by an earlier
      // launch); the padding rows of a tile hold zeros there, and see no key below
      int t_row = 0;
      float lse_r = 0.f, dr_r = 0.f;
      if (kDQ) {
        t_row = it.tile * p.P + r / p.G;
        const size_t vi = ((static_cast<size_t>(it.b) * p.Hkv + it.g) * p.n_qtiles + it.tile) * 128 + r;
        lse_r = __ldg(p.lse + vi);
        dr_r = __ldg(p.drow + vi);
      }
      const bool row_ok = !kDQ || (r < GP && t_row < p.T);
      const int key_row = it.tile * 128 + r;  // dK,dV: this row's key position
      // Every thread runs every step of the item (a thread whose wait failed skips the work), so that all of them
      // meet the barrier of the deferred epilogue after the first step.
      for (int j = it.lo; j <= it.hi; ++j, ++nb, ++ns) {
        if (!fail) {
          const int st = nb % kStages;
          // visible columns of this thread's row: one interval [lo_c, hi_c] of the tile's 128 columns
          int lo_c, hi_c;
          if (!kDQ) {
            // columns = packed query rows of Q tile j: c -> position j P + c / G
            const int t0 = j * p.P;
            lo_c = p.G * (key_row - t0);
            hi_c = min(GP, p.G * (p.T - t0)) - 1;
            if (p.window >= 0) hi_c = min(hi_c, p.G * (key_row + p.window - t0) + p.G - 1);
          } else {
            // columns = keys j 128 + c
            hi_c = row_ok ? t_row - j * 128 : -1;
            lo_c = p.window < 0 ? INT_MIN / 2 : hi_c - p.window;
          }
          const float* vec = sVec + st * 256;  // dK,dV: lse and rowsum of the columns (Q tile j), landed with B
          if (!kDQ) fail = !__all_sync(0xffffffffu, mbar_wait(b_full + st, (nb / kStages) & 1, lim, abort_flag));
          if (!fail) fail = !__all_sync(0xffffffffu, mbar_wait(x_full, ns & 1, lim, abort_flag));
          if (!fail) {
            tc_fence_after_sync();
            // ---- probabilities: P = 2^(X - lse) on the visible columns, 0 elsewhere
            float pv[2][32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int c0 = 64 * h + 32 * c2;
              uint32_t sv[32];
              tmem_ld32(tX + c0, sv);
              tmem_ld_wait(sv);
              const uint32_t vis = interval_mask(lo_c, hi_c, c0);
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const float l = kDQ ? lse_r : vec[c0 + c];
                pv[c2][c] = ((vis >> c) & 1u) ? ex2_approx(__uint_as_float(sv[c]) - l) : 0.f;
              }
              if (!kDQ) {  // P^T is an operand of dV += P^T dO: bf16 pairs over the S^T columns just read
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pv[c2][2 * c], pv[c2][2 * c + 1]);
                tmem_st16(tX + 64 * h + 16 * c2, pk);
              }
            }
            // X consumed (dK,dV: P^T written over it; dQ: read into registers): the next step's X may go in
            if (!kDQ) tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            // ---- dS = P (dP - rowsum), bf16 pairs over the dP columns just read
            fail = !__all_sync(0xffffffffu, mbar_wait(y_full, ns & 1, lim, abort_flag));
            if (!fail) {
              tc_fence_after_sync();
#pragma unroll
              for (int c2 = 0; c2 < 2; ++c2) {
                const int c0 = 64 * h + 32 * c2;
                uint32_t dv[32];
                tmem_ld32(tY + c0, dv);
                tmem_ld_wait(dv);
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                  const float d0 = kDQ ? dr_r : vec[128 + c0 + 2 * c];
                  const float d1 = kDQ ? dr_r : vec[128 + c0 + 2 * c + 1];
                  pk[c] = pack_bf16x2(pv[c2][2 * c] * (__uint_as_float(dv[2 * c]) - d0),
                                      pv[c2][2 * c + 1] * (__uint_as_float(dv[2 * c + 1]) - d1));
                }
                tmem_st16(tY + 64 * h + 16 * c2, pk);
              }
              tmem_st_wait();
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(ds_full);
            }
          }
        }
        if (kDQ && j == it.lo && pending_k >= 0) {
          // the previous item's epilogue, while the tensor core works on this item's next step
          if (!named_bar_and(kBarAll, 2 * 128, !fail) || !epilogue(pending, pending_k)) fail = true;
          pending_k = -1;
        }
      }
      if (!named_bar_and(kBarAll, 2 * 128, !fail)) {
        failed = true;
        break;
      }
      if (kDQ) {
        pending = it;
        pending_k = k;
      } else if (!epilogue(it, k)) {
        failed = true;
        break;
      }
    }
    if (kDQ && !failed && pending_k >= 0) epilogue(pending, pending_k);
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

}  // namespace bwd
}  // namespace nc
