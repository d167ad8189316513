// K5: backward pass of the attention block on the CUDA cores (fp32), correctness first.
//
// What it computes: the gradients of sum(dout * out) with respect to the raw q, k and v of the prefill forward
// (out = attention(norm(rope(q)), norm(rope(k)), v), causal with the window, logits scaled by qk_gain / sqrt(D),
// contiguous GQA groups; "nanochat Admin & Developer Guide", section 3 -- the model trains through this block).
// The chain rule, per (b, query head h, kv head g = h / G), with P = softmax(S), O = P V, c = qk_gain / sqrt(D):
//   dV_g += P^T dO,  dP = dO V_g^T,  dS = P * (dP - rowsum(dO * O)),  dqn_h = c dS kn_g,  dkn_g += c dS^T qn_h;
// then the RMSNorm backward dx = (dy - qn (dy . qn) / D) / r (r the forward's RMS, eps included) and the RoPE
// backward, the rotation of each pair (i, i + D/2) by -t theta_i.
//
// Four kernels, one warp per output row, lane l holding dims [4 l', 4 l' + 4) of half l / 16 (l' = l % 16), so that
// a RoPE pair (i, i + 64) sits in lanes l and l ^ 16; dot products over the 128 dims are xor-shuffle reductions.
//   bwd_prep_kernel      qn, kn (fp32) and 1 / r of every q and k head vector;
//   bwd_rowstats_kernel  per query row: log-sum-exp of its logits and rowsum(dO * O), with O recomputed by an online
//                        softmax pass over the row's keys;
//   bwd_dq_kernel        per query row: dqn over its keys, then the norm and RoPE backward -> dq;
//   bwd_dkv_kernel       per key row of a kv head: dV and dkn over the queries (all heads of the group) that see it,
//                        then the norm and RoPE backward -> dk.
// No shared memory, no barriers, no waits.  The contractions run as warp dot products, far from the tensor cores'
// rate: this kernel set establishes the gradients; a tcgen05 version is the next step for it.
#pragma once

#include "common.cuh"

namespace nc {
namespace bwd {

constexpr int kWarpsPerBlock = 8;

struct Params {
  const __nv_bfloat16* q;     // [B, T, Hq, 128]
  const __nv_bfloat16* k;     // [B, T, Hkv, 128]
  const __nv_bfloat16* v;     // [B, T, Hkv, 128]
  const __nv_bfloat16* dout;  // [B, T, Hq, 128]
  float* dq;                  // [B, T, Hq, 128]
  float* dk;                  // [B, T, Hkv, 128]
  float* dv;                  // [B, T, Hkv, 128]
  float* qn;                  // [B, T, Hq, 128]  workspace
  float* kn;                  // [B, T, Hkv, 128] workspace
  float* inv_rq;              // [B, T, Hq]       workspace
  float* inv_rk;              // [B, T, Hkv]      workspace
  float* lse;                 // [B, T, Hq]       workspace
  float* drow;                // [B, T, Hq]       workspace: rowsum(dO * O)
  int B, T, Hq, Hkv, G, window;
  float c;                    // qk_gain / sqrt(128)
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Dims of lane l: half l / 16, indices [4 (l % 16), 4 (l % 16) + 4) within the half.
__device__ __forceinline__ int lane_dim0(int lane) { return (lane >> 4) * 64 + (lane & 15) * 4; }

__device__ __forceinline__ void load4_bf16(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  x[0] = bf16_lo(u.x);
  x[1] = bf16_hi(u.x);
  x[2] = bf16_lo(u.y);
  x[3] = bf16_hi(u.y);
}

__device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  x[0] = u.x;
  x[1] = u.y;
  x[2] = u.z;
  x[3] = u.w;
}

__device__ __forceinline__ void store4(float* p, const float (&x)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}

__device__ __forceinline__ float dot4(const float (&a)[4], const float (&b)[4]) {
  return fmaf(a[0], b[0], fmaf(a[1], b[1], fmaf(a[2], b[2], a[3] * b[3])));
}

// cos / sin of this lane's four pair angles at position t.
__device__ __forceinline__ void lane_cos_sin(const RopeTable& tab, int lane, int t, float (&cs)[4], float (&sn)[4]) {
  const int i0 = (lane & 15) * 4;
#pragma unroll
  for (int e = 0; e < 4; ++e) rope_cos_sin(static_cast<float>(t), tab.hi[i0 + e], tab.lo[i0 + e], cs[e], sn[e]);
}

// Rotation of the pairs by +angle (forward RoPE, sign = 1) or -angle (its backward, sign = -1).
__device__ __forceinline__ void rotate(float (&x)[4], const float (&cs)[4], const float (&sn)[4], int lane,
                                       float sign) {
  const bool first = lane < 16;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
    const float s = sign * sn[e];
    // forward: y_i = x_i c + x_{i+64} s,  y_{i+64} = -x_i s + x_{i+64} c
    x[e] = first ? fmaf(x[e], cs[e], other * s) : fmaf(x[e], cs[e], -other * s);
  }
}

// qn, kn and 1 / r for every q head vector (rows [0, B T Hq)) and k head vector (the next B T Hkv rows).
__global__ void __launch_bounds__(kWarpsPerBlock * 32) bwd_prep_kernel(const Params p, const __grid_constant__ RopeTable tab) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const long long nq = static_cast<long long>(p.B) * p.T * p.Hq, nk = static_cast<long long>(p.B) * p.T * p.Hkv;
  if (row >= nq + nk) return;
  const bool is_q = row < nq;
  const long long r = is_q ? row : row - nq;
  const int H = is_q ? p.Hq : p.Hkv;
  const int t = static_cast<int>((r / H) % p.T);
  const int d0 = lane_dim0(lane);
  float x[4];
  load4_bf16((is_q ? p.q : p.k) + r * 128 + d0, x);
  float cs[4], sn[4];
  lane_cos_sin(tab, lane, t, cs, sn);
  rotate(x, cs, sn, lane, 1.f);
  const float inv_r = rsqrtf(warp_sum(dot4(x, x)) * (1.f / 128.f) + kRmsEps);
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] *= inv_r;
  store4((is_q ? p.qn : p.kn) + r * 128 + d0, x);
  if (lane == 0) (is_q ? p.inv_rq : p.inv_rk)[r] = inv_r;
}

// Per query row (b, t, h): lse = log sum_j exp(s_j) and drow = dO . O, O = softmax(s) V recomputed online.
__global__ void __launch_bounds__(kWarpsPerBlock * 32) bwd_rowstats_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(p.B) * p.T * p.Hq) return;
  const int h = static_cast<int>(row % p.Hq);
  const long long bt = row / p.Hq;
  const int t = static_cast<int>(bt % p.T), b = static_cast<int>(bt / p.T), g = h / p.G;
  const int d0 = lane_dim0(lane);
  float qv[4];
  load4(p.qn + row * 128 + d0, qv);
  const int lo = p.window < 0 ? 0 : max(0, t - p.window);
  float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = lo; j <= t; ++j) {
    const long long kr = (static_cast<long long>(b) * p.T + j) * p.Hkv + g;
    float kv[4], vv[4];
    load4(p.kn + kr * 128 + d0, kv);
    load4_bf16(p.v + kr * 128 + d0, vv);
    const float s = p.c * warp_sum(dot4(qv, kv));
    const float m2 = fmaxf(m, s);
    const float a = expf(m - m2), e = expf(s - m2);
    l = fmaf(l, a, e);
#pragma unroll
    for (int d = 0; d < 4; ++d) o[d] = fmaf(o[d], a, e * vv[d]);
    m = m2;
  }
  float dov[4];
  load4_bf16(p.dout + row * 128 + d0, dov);
  const float inv_l = 1.f / l;
#pragma unroll
  for (int d = 0; d < 4; ++d) o[d] *= inv_l;
  const float dr = warp_sum(dot4(dov, o));
  if (lane == 0) {
    p.lse[row] = m + logf(l);
    p.drow[row] = dr;
  }
}

// Norm backward then RoPE backward of this lane's 4 dims of dy (gradient w.r.t. the normed vector yn).
__device__ __forceinline__ void norm_rope_bwd(float (&dy)[4], const float (&yn)[4], float inv_r, const RopeTable& tab,
                                              int lane, int t) {
  const float proj = warp_sum(dot4(dy, yn)) * (1.f / 128.f);
#pragma unroll
  for (int e = 0; e < 4; ++e) dy[e] = (dy[e] - yn[e] * proj) * inv_r;
  float cs[4], sn[4];
  lane_cos_sin(tab, lane, t, cs, sn);
  rotate(dy, cs, sn, lane, -1.f);
}

// Per query row (b, t, h): dq.
__global__ void __launch_bounds__(kWarpsPerBlock * 32) bwd_dq_kernel(const Params p, const __grid_constant__ RopeTable tab) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(p.B) * p.T * p.Hq) return;
  const int h = static_cast<int>(row % p.Hq);
  const long long bt = row / p.Hq;
  const int t = static_cast<int>(bt % p.T), b = static_cast<int>(bt / p.T), g = h / p.G;
  const int d0 = lane_dim0(lane);
  float qv[4], dov[4];
  load4(p.qn + row * 128 + d0, qv);
  load4_bf16(p.dout + row * 128 + d0, dov);
  const float lse = p.lse[row], dr = p.drow[row];
  const int lo = p.window < 0 ? 0 : max(0, t - p.window);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = lo; j <= t; ++j) {
    const long long kr = (static_cast<long long>(b) * p.T + j) * p.Hkv + g;
    float kv[4], vv[4];
    load4(p.kn + kr * 128 + d0, kv);
    load4_bf16(p.v + kr * 128 + d0, vv);
    const float s = p.c * warp_sum(dot4(qv, kv));
    const float dp = warp_sum(dot4(dov, vv));
    const float ds = expf(s - lse) * (dp - dr);
#pragma unroll
    for (int d = 0; d < 4; ++d) acc[d] = fmaf(ds, kv[d], acc[d]);
  }
#pragma unroll
  for (int d = 0; d < 4; ++d) acc[d] *= p.c;
  norm_rope_bwd(acc, qv, p.inv_rq[row], tab, lane, t);
  store4(p.dq + row * 128 + d0, acc);
}

// Per key row (b, j, g): dk and dv over every query (of every head of the group) that sees key j.
__global__ void __launch_bounds__(kWarpsPerBlock * 32) bwd_dkv_kernel(const Params p, const __grid_constant__ RopeTable tab) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(p.B) * p.T * p.Hkv) return;
  const int g = static_cast<int>(row % p.Hkv);
  const long long bj = row / p.Hkv;
  const int j = static_cast<int>(bj % p.T), b = static_cast<int>(bj / p.T);
  const int d0 = lane_dim0(lane);
  float kv[4], vv[4];
  load4(p.kn + row * 128 + d0, kv);
  load4_bf16(p.v + row * 128 + d0, vv);
  const int hi = p.window < 0 ? p.T - 1 : min(p.T - 1, j + p.window);
  float dk_acc[4] = {0.f, 0.f, 0.f, 0.f}, dv_acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int t = j; t <= hi; ++t) {
    for (int jh = 0; jh < p.G; ++jh) {
      const long long qr = (static_cast<long long>(b) * p.T + t) * p.Hq + g * p.G + jh;
      float qv[4], dov[4];
      load4(p.qn + qr * 128 + d0, qv);
      load4_bf16(p.dout + qr * 128 + d0, dov);
      const float s = p.c * warp_sum(dot4(qv, kv));
      const float dp = warp_sum(dot4(dov, vv));
      const float pr = expf(s - p.lse[qr]);
      const float ds = pr * (dp - p.drow[qr]);
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        dv_acc[d] = fmaf(pr, dov[d], dv_acc[d]);
        dk_acc[d] = fmaf(ds, qv[d], dk_acc[d]);
      }
    }
  }
  store4(p.dv + row * 128 + d0, dv_acc);
#pragma unroll
  for (int d = 0; d < 4; ++d) dk_acc[d] *= p.c;
  norm_rope_bwd(dk_acc, kv, p.inv_rk[row], tab, lane, j);
  store4(p.dk + row * 128 + d0, dk_acc);
}

}  // namespace bwd
}  // namespace nc
