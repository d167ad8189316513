// K3: KV-cache single-token decode, split over key chunks, merged inside the same launch.
//
// What it computes ("nanochat Admin & Developer Guide", section 7 "KV cache": FA3 layout (B, T, H, D), per-row
// cache_seqlens, in-place append; section 6: the SDPA decode case attends over a slice of the cache): for sequence b
// with p = cache_lens[b], the new query is roped at position p and normed; it attends over cache rows
// [max(0, p - window), p) -- plus row p when a new key/value is given, which is roped + normed at position p,
// written into the cache and attended to.
//
// Work split.  One CTA per (key chunk of kC = 128 positions, kv head g, sequence b); it serves the G query heads of
// the group.  The chunk's K and V rows (256 B each) arrive by TMA as 128-byte-swizzled half tiles, fully coalesced.
// Scores: thread r owns key row r and computes its G dot products in fp32 against the normed query kept in shared
// memory (swizzled reads are bank-conflict free).  Softmax over the chunk: block max / sum with warp shuffles.
// P.V: thread (rsub, dch) accumulates 8 dims x G heads over rows rsub, rsub+8, ...; the 8 partial sums are added
// through shared memory.  With one chunk the CTA writes the output; otherwise it writes (m, l, o) partials and the
// last CTA of the (b, g) pair to arrive (atomic counter) merges them with the log-sum-exp rule and resets the
// counter.  All work runs on CUDA cores: M = G <= 8 query rows is far too small for the tensor cores, and the
// kernel is bound by HBM reads of the cache.
#pragma once

#include "common.cuh"
#include "prologue.cuh"

namespace nc {
namespace dec {

constexpr int kC = 128;                  // keys per CTA
constexpr int kThreads = 128;
constexpr int kHalfBytes = kC * 128;     // one 64-column half of the chunk's rows: 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr int kMaxG = 8;

constexpr int kOffK = 0;                             // K rows; reused for the P.V reduction [8][G][128] f32
constexpr int kOffV = kOffK + kTileBytes;            // V rows
constexpr int kOffQ = kOffV + kTileBytes;            // normed queries [G][128] f32
constexpr int kOffP = kOffQ + kMaxG * 128 * 4;       // probabilities [G][kC] f32
constexpr int kOffRed = kOffP + kMaxG * kC * 4;      // block max / sum scratch [2][4 warps][G] f32
constexpr int kOffNew = kOffRed + 2 * 4 * kMaxG * 4; // new key row and new value row (bf16), 2 x 256 B
constexpr int kOffBar = kOffNew + 512;
constexpr int kSmemBytes = kOffBar + 64 + 1024;

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* kcache;
  __nv_bfloat16* vcache;
  const int* cache_lens;
  __nv_bfloat16* out;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  float* ws_ml;        // [B][Hkv][n_chunks][G][2]  (m, l) per chunk, log2 domain
  float* ws_o;         // [B][Hkv][n_chunks][G][128] unnormalised partial outputs
  unsigned* ws_cnt;    // [B][Hkv] arrival counters, zero between calls
  int B, Hq, Hkv, Tcap, window, n_chunks;
  float scale_log2;
  unsigned long long wait_limit_ns;
};

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

// Offset of 16-byte chunk `ch` (0..15, i.e. dims [8ch, 8ch+8)) of row `r` inside a TMA tile of 128-byte-swizzled
// half rows: half ch / 8 at + half * kHalfBytes, row r at r * 128, chunk slot (ch % 8) xor (r % 8).
__device__ __forceinline__ int swz_off(int r, int ch) {
  return (ch >> 3) * kHalfBytes + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

template <int G>
__global__ void __launch_bounds__(kThreads)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ RopeTable tab, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  float* qs = reinterpret_cast<float*>(smem + kOffQ);
  float* ps = reinterpret_cast<float*>(smem + kOffP);
  float* red_m = reinterpret_cast<float*>(smem + kOffRed);
  float* red_l = red_m + 4 * kMaxG;
  uint4* new_k = reinterpret_cast<uint4*>(smem + kOffNew);
  uint4* new_v = reinterpret_cast<uint4*>(smem + kOffNew + 256);
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* v_full = k_full + 1;
  int* flag = reinterpret_cast<int*>(smem + kOffBar + 16);

  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool has_new = p.k_new != nullptr;
  const int pos = __ldg(p.cache_lens + b);
  const int max_pos = has_new ? p.Tcap - 1 : p.Tcap;
  __nv_bfloat16* outg = p.out + (static_cast<size_t>(b) * p.Hq + g * G) * 128;
  const __nv_bfloat16 zero = __float2bfloat16(0.f);

  if (pos < 0 || pos > max_pos) {  // invalid cache length: zero row, sticky device status, no cache access
    if (c == 0) {
      if (tid == 0) raise_status(NC_DEV_BAD_CACHE_LEN);
      for (int i = tid; i < G * 128; i += kThreads) outg[i] = zero;
    }
    return;
  }
  const int L = pos + (has_new ? 1 : 0);
  const int lo = p.window < 0 ? 0 : max(0, pos - p.window);
  const int nvis = L - lo;
  const int nc = (nvis + kC - 1) / kC;
  if (nvis <= 0) {  // nothing visible: zero row
    if (c == 0)
      for (int i = tid; i < G * 128; i += kThreads) outg[i] = zero;
    return;
  }
  if (c >= nc) return;
  const int s0 = lo + c * kC;
  const int n = min(kC, L - s0);
  const bool has_row_p = has_new && c == nc - 1;  // row `pos` is the last visible row
  const int row_p = pos - s0;

  if (tid == 0) {
    mbar_init(k_full, 1);
    mbar_init(v_full, 1);
    *flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(k_full, kTileBytes);
    tma_load_4d(sK, &tmK, k_full, 0, g, s0, b);
    tma_load_4d(sK + kHalfBytes, &tmK, k_full, 64, g, s0, b);
    mbar_arrive_expect_tx(v_full, kTileBytes);
    tma_load_4d(sV, &tmV, v_full, 0, g, s0, b);
    tma_load_4d(sV + kHalfBytes, &tmV, v_full, 64, g, s0, b);
  }

  // ---- prologue while the copies are in flight: normed queries (groups 0..G-1), the new key (group G) and the
  // new value (group G+1).  8 lanes per head vector, lane kq owns pairs [8kq, 8kq+8).
  {
    const int grp = tid >> 3, kq = tid & 7;
    const unsigned gmask = 0xFFu << (lane & ~7);
    if (grp < G || (has_row_p && grp == G)) {
      float cs[8], sn[8];
      const float fpos = static_cast<float>(pos);
#pragma unroll
      for (int i = 0; i < 8; ++i) rope_cos_sin(fpos, tab.hi[kq * 8 + i], tab.lo[kq * 8 + i], cs[i], sn[i]);
      const uint4* src = reinterpret_cast<const uint4*>(
          grp < G ? p.q + (static_cast<size_t>(b) * p.Hq + g * G + grp) * 128
                  : p.k_new + (static_cast<size_t>(b) * p.Hkv + g) * 128);
      float y1[8], y2[8];
      rope_norm_slices(__ldg(src + kq), __ldg(src + 8 + kq), cs, sn, gmask, y1, y2);
      if (grp < G) {
        float4* qd = reinterpret_cast<float4*>(qs + grp * 128);
        qd[2 * kq] = make_float4(y1[0], y1[1], y1[2], y1[3]);
        qd[2 * kq + 1] = make_float4(y1[4], y1[5], y1[6], y1[7]);
        qd[16 + 2 * kq] = make_float4(y2[0], y2[1], y2[2], y2[3]);
        qd[16 + 2 * kq + 1] = make_float4(y2[4], y2[5], y2[6], y2[7]);
      } else {
        const uint4 a = pack8_bf16(y1), bb = pack8_bf16(y2);
        uint4* dst = reinterpret_cast<uint4*>(p.kcache + ((static_cast<size_t>(b) * p.Tcap + pos) * p.Hkv + g) * 128);
        dst[kq] = a;
        dst[8 + kq] = bb;
        new_k[kq] = a;
        new_k[8 + kq] = bb;
      }
    } else if (has_row_p && grp == G + 1) {
      const uint4* src = reinterpret_cast<const uint4*>(p.v_new + (static_cast<size_t>(b) * p.Hkv + g) * 128);
      uint4* dst = reinterpret_cast<uint4*>(p.vcache + ((static_cast<size_t>(b) * p.Tcap + pos) * p.Hkv + g) * 128);
      const uint4 a = __ldg(src + kq), bb = __ldg(src + 8 + kq);
      dst[kq] = a;
      dst[8 + kq] = bb;
      new_v[kq] = a;
      new_v[8 + kq] = bb;
    }
  }
  __syncthreads();

  const unsigned long long lim = p.wait_limit_ns;
  bool ok = mbar_wait(k_full, 0, lim, nullptr);
  if (ok && has_row_p && tid < 16) *reinterpret_cast<uint4*>(sK + swz_off(row_p, tid)) = new_k[tid];
  if (__syncthreads_or(!ok)) {  // a copy never landed: wait once more (bounded) for both, then leave
    if (tid == 0) {
      mbar_wait(k_full, 0, lim, nullptr);
      mbar_wait(v_full, 0, lim, nullptr);
    }
    return;
  }

  // ---- scores: thread r owns key row r
  const int r = tid;
  float x[G];
  {
    float acc[G];
#pragma unroll
    for (int j = 0; j < G; ++j) acc[j] = 0.f;
    const float4* q4 = reinterpret_cast<const float4*>(qs);
#pragma unroll 4
    for (int ch = 0; ch < 16; ++ch) {
      const uint4 kv = *reinterpret_cast<const uint4*>(sK + swz_off(r, ch));
      const float k0 = bf16_lo(kv.x), k1 = bf16_hi(kv.x), k2 = bf16_lo(kv.y), k3 = bf16_hi(kv.y);
      const float k4 = bf16_lo(kv.z), k5 = bf16_hi(kv.z), k6 = bf16_lo(kv.w), k7 = bf16_hi(kv.w);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float4 qa = q4[j * 32 + 2 * ch];
        const float4 qb = q4[j * 32 + 2 * ch + 1];
        float a = acc[j];
        a = fmaf(k0, qa.x, a);
        a = fmaf(k1, qa.y, a);
        a = fmaf(k2, qa.z, a);
        a = fmaf(k3, qa.w, a);
        a = fmaf(k4, qb.x, a);
        a = fmaf(k5, qb.y, a);
        a = fmaf(k6, qb.z, a);
        a = fmaf(k7, qb.w, a);
        acc[j] = a;
      }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) x[j] = (r < n) ? acc[j] * p.scale_log2 : -INFINITY;
  }
  float mg[G], lg[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const float mx = warp_max(x[j]);
    if (lane == 0) red_m[warp * kMaxG + j] = mx;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < G; ++j) {
    mg[j] = fmaxf(fmaxf(red_m[j], red_m[kMaxG + j]), fmaxf(red_m[2 * kMaxG + j], red_m[3 * kMaxG + j]));
    const float pj = ex2_approx(x[j] - mg[j]);
    ps[j * kC + r] = pj;
    const float sm = warp_sum(pj);
    if (lane == 0) red_l[warp * kMaxG + j] = sm;
  }
  ok = mbar_wait(v_full, 0, lim, nullptr);
  if (ok && has_row_p && tid < 16) *reinterpret_cast<uint4*>(sV + swz_off(row_p, tid)) = new_v[tid];
  if (__syncthreads_or(!ok)) {
    if (tid == 0) mbar_wait(v_full, 0, lim, nullptr);
    return;
  }
#pragma unroll
  for (int j = 0; j < G; ++j) lg[j] = (red_l[j] + red_l[kMaxG + j]) + (red_l[2 * kMaxG + j] + red_l[3 * kMaxG + j]);

  // ---- P.V: thread (rsub, dch) accumulates dims [8 dch, 8 dch + 8) over rows rsub, rsub + 8, ...
  const int dch = tid & 15, rsub = tid >> 4;
  float o[G][8];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[j][e] = 0.f;
#pragma unroll 4
  for (int rr = rsub; rr < n; rr += 8) {
    const uint4 vv = *reinterpret_cast<const uint4*>(sV + swz_off(rr, dch));
    const float v[8] = {bf16_lo(vv.x), bf16_hi(vv.x), bf16_lo(vv.y), bf16_hi(vv.y),
                        bf16_lo(vv.z), bf16_hi(vv.z), bf16_lo(vv.w), bf16_hi(vv.w)};
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float pj = ps[j * kC + rr];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[j][e] = fmaf(pj, v[e], o[j][e]);
    }
  }
  float* red = reinterpret_cast<float*>(sK);  // [8][G][128]; K rows are no longer read
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float4* d4 = reinterpret_cast<float4*>(red + (rsub * G + j) * 128 + dch * 8);
    d4[0] = make_float4(o[j][0], o[j][1], o[j][2], o[j][3]);
    d4[1] = make_float4(o[j][4], o[j][5], o[j][6], o[j][7]);
  }
  __syncthreads();
  float res[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float a = 0.f;
#pragma unroll
    for (int rs = 0; rs < 8; ++rs) a += red[(rs * G + j) * 128 + tid];
    res[j] = a;
  }

  if (nc == 1) {
#pragma unroll
    for (int j = 0; j < G; ++j) outg[j * 128 + tid] = __float2bfloat16_rn(res[j] / lg[j]);
    return;
  }

  // ---- split: publish the partial, the last CTA of (b, g) merges
  const size_t slot0 = (static_cast<size_t>(b) * p.Hkv + g) * p.n_chunks;
  const size_t slot = slot0 + c;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    p.ws_o[(slot * G + j) * 128 + tid] = res[j];
    if (tid == j) {
      p.ws_ml[(slot * G + j) * 2] = mg[j];
      p.ws_ml[(slot * G + j) * 2 + 1] = lg[j];
    }
  }
  __threadfence();
  __syncthreads();
  unsigned* cnt = p.ws_cnt + static_cast<size_t>(b) * p.Hkv + g;
  if (tid == 0) *flag = (atomicAdd(cnt, 1u) == static_cast<unsigned>(nc - 1)) ? 1 : 0;
  __syncthreads();
  if (*flag == 0) return;
  __threadfence();
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float M = -INFINITY;
    for (int cc = 0; cc < nc; ++cc) M = fmaxf(M, __ldcg(p.ws_ml + ((slot0 + cc) * G + j) * 2));
    float Ls = 0.f, O = 0.f;
    for (int cc = 0; cc < nc; ++cc) {
      const float w = ex2_approx(__ldcg(p.ws_ml + ((slot0 + cc) * G + j) * 2) - M);
      Ls = fmaf(w, __ldcg(p.ws_ml + ((slot0 + cc) * G + j) * 2 + 1), Ls);
      O = fmaf(w, __ldcg(p.ws_o + ((slot0 + cc) * G + j) * 128 + tid), O);
    }
    outg[j * 128 + tid] = __float2bfloat16_rn(O / Ls);
  }
  if (tid == 0) *cnt = 0u;  // leave the counter zero for the next call
}

}  // namespace dec
}  // namespace nc
