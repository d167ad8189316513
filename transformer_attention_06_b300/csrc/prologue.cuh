// K1: fused RoPE + QK-norm prologue of the prefill forward.
//
// For every token (b, t) and every q head and k head: rotate the half-split pairs (i, i + 64) by t * theta_i, then
// divide the vector by sqrt(mean(y^2) + eps).  ("nanochat Admin & Developer Guide", section 3: RoPE base 100000,
// QK-norm, RMSNorm without parameters; "nanochat (Fucina port)", "Architecture": half-split RoPE.)
//
// Memory-bound: it reads q and k once and writes qn and kn once (2 * 2 * B*T*(Hq+Hkv)*128 bytes).  Mapping: an
// 8-lane group per token; lane kq of the group owns pairs [8kq, 8kq+8), i.e. two 16-byte slices of every head
// vector of the token, so the cos/sin of the token are computed once and reused across all Hq + Hkv heads.  The
// sum of squares is reduced across the group with three xor-shuffles.  The normalised q vectors may be multiplied
// by a constant on the way out (the attention kernel takes the softmax scale log2(e) / sqrt(D) this way).  The fp8
// variant writes qn and kn as e4m3 (1 byte per element) times per-tensor scales, for the e4m3 score contraction.
#pragma once

#include "common.cuh"

namespace nc {

// Rotates the 8 pairs held in (lo, hi) -- elements [8kq, 8kq+8) and [64+8kq, 64+8kq+8) of a 128-wide head
// vector -- and normalises by the RMS of the whole vector (reduced over the 8-lane group `gmask`), times `scale`.
// Two neighbouring elements travel together through packed fp32 pairs (f32x2: one instruction for both), so the
// rotation, the sum of squares and the scaling cost half the instructions of scalar code.
__device__ __forceinline__ void rope_norm_slices(const uint4& lo, const uint4& hi, const float (&c)[8],
                                                 const float (&s)[8], unsigned gmask, float scale,
                                                 float (&y1)[8], float (&y2)[8]) {
  const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w};
  const uint32_t b[4] = {hi.x, hi.y, hi.z, hi.w};
  uint64_t r1[4], r2[4];
  uint64_t ss2 = 0ull;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t x1 = f32x2(bf16_lo(a[i]), bf16_hi(a[i]));
    const uint64_t x2 = f32x2(bf16_lo(b[i]), bf16_hi(b[i]));
    const uint64_t cc = f32x2(c[2 * i], c[2 * i + 1]);
    const uint64_t sp = f32x2(s[2 * i], s[2 * i + 1]);
    const uint64_t sn = f32x2(-s[2 * i], -s[2 * i + 1]);
    r1[i] = fma_f32x2(x1, cc, mul_f32x2(x2, sp));   // x1 c + x2 s
    r2[i] = fma_f32x2(x2, cc, mul_f32x2(x1, sn));   // x2 c - x1 s
    ss2 = fma_f32x2(r1[i], r1[i], ss2);
    ss2 = fma_f32x2(r2[i], r2[i], ss2);
  }
  float s0, s1;
  f32x2_split(ss2, s0, s1);
  float ss = s0 + s1;
  ss += __shfl_xor_sync(gmask, ss, 1);
  ss += __shfl_xor_sync(gmask, ss, 2);
  ss += __shfl_xor_sync(gmask, ss, 4);
  const float inv = rsqrtf(ss * (1.0f / 128.0f) + kRmsEps) * scale;
  const uint64_t inv2 = f32x2(inv, inv);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f32x2_split(mul_f32x2(r1[i], inv2), y1[2 * i], y1[2 * i + 1]);
    f32x2_split(mul_f32x2(r2[i], inv2), y2[2 * i], y2[2 * i + 1]);
  }
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&y)[8]) {
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

__device__ __forceinline__ uint2 pack8_e4m3(const float (&y)[8]) {
  return make_uint2(pack_e4m3x4(y[0], y[1], y[2], y[3]), pack_e4m3x4(y[4], y[5], y[6], y[7]));
}

__device__ __forceinline__ void store_head(void* dst, int kq, const float (&y1)[8], const float (&y2)[8], bool e4m3) {
  if (e4m3) {
    uint2* out = reinterpret_cast<uint2*>(dst);
    out[kq] = pack8_e4m3(y1);
    out[8 + kq] = pack8_e4m3(y2);
  } else {
    uint4* out = reinterpret_cast<uint4*>(dst);
    out[kq] = pack8_bf16(y1);
    out[8 + kq] = pack8_bf16(y2);
  }
}

// The first round of rope_norm_token: slices kq and kq + 8 of heads i0 .. i0 + 3 (those below i1) of the token's
// list of Hq q heads followed by its Hkv k heads.  It depends on nothing but the token, so callers issue it before
// computing the position's cos / sin (and, in the chunked prefill, before the cache length has arrived).
__device__ __forceinline__ void load_first_heads(const __nv_bfloat16* __restrict__ q,
                                                 const __nv_bfloat16* __restrict__ k, int Hq, int i0, int i1, int kq,
                                                 uint4 (&lo)[4], uint4 (&hi)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + u;
    if (i < i1) {
      const uint4* p = reinterpret_cast<const uint4*>(i < Hq ? q + i * 128 : k + (i - Hq) * 128);
      lo[u] = __ldg(p + kq);
      hi[u] = __ldg(p + 8 + kq);
    }
  }
}

// Heads [i0, i1) of one token's list of its Hq q heads followed by its Hkv k heads (q, k, qn, kn point at the
// token's head 0), in rounds of four heads whose loads are issued one round ahead: while a round is rotated,
// normalised and stored, the next round's sixteen 16-byte loads per lane are in flight.  (lo0, hi0) hold the first
// round, from load_first_heads.  OutT = __nv_bfloat16 writes bf16 rows of 256 bytes; OutT = uint8_t writes e4m3 rows
// of 128 bytes (the values times the scale, rounded to nearest even).
template <typename OutT>
__device__ __forceinline__ void rope_norm_token(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                                                OutT* __restrict__ qn, OutT* __restrict__ kn, int Hq, int i0, int i1,
                                                int kq, const float (&c)[8], const float (&s)[8], unsigned gmask,
                                                float q_scale, float k_scale, const uint4 (&lo0)[4],
                                                const uint4 (&hi0)[4]) {
  constexpr bool kE4m3 = sizeof(OutT) == 1;
  const int H = i1;
  auto src = [&](int i) {
    return reinterpret_cast<const uint4*>(i < Hq ? q + i * 128 : k + (i - Hq) * 128);
  };
  uint4 lo[2][4], hi[2][4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    lo[0][u] = lo0[u];
    hi[0][u] = hi0[u];
  }
  for (int h0 = i0; h0 < H; h0 += 8) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int base = h0 + 4 * half;
      if (base >= H) break;
      const int nb = half ^ 1;  // buffer of the next round
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + 4 + u;
        if (i < H) {
          lo[nb][u] = __ldg(src(i) + kq);
          hi[nb][u] = __ldg(src(i) + 8 + kq);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u;
        if (i < H) {
          float y1[8], y2[8];
          rope_norm_slices(lo[half][u], hi[half][u], c, s, gmask, i < Hq ? q_scale : k_scale, y1, y2);
          void* dst = i < Hq ? static_cast<void*>(qn + i * 128) : static_cast<void*>(kn + (i - Hq) * 128);
          store_head(dst, kq, y1, y2, kE4m3);
        }
      }
    }
  }
}

// Gated value embedding (the catalog pages list value embeddings with a sigmoid gate, in the ResFormer manner; they give
// no formula, the reading is v' = v + sigmoid(g) ve with one gate logit g per token and kv head): the H value
// vectors of one token, 16-byte slices kq and kq + 8 of each, mixed in fp32 and rounded to bf16.
// Four heads per round, all their loads issued before the first store.
__device__ __forceinline__ void mix_values(const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ ve,
                                           const __nv_bfloat16* __restrict__ gate, __nv_bfloat16* __restrict__ vmix,
                                           int H, int kq) {
  for (int h0 = 0; h0 < H; h0 += 4) {
    uint4 x[4][2], e[4][2];
    float g[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (h0 + u < H) {
        g[u] = __bfloat162float(gate[h0 + u]);
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          const int i = (h0 + u) * 16 + kq + 8 * i2;
          x[u][i2] = __ldg(reinterpret_cast<const uint4*>(v) + i);
          e[u][i2] = __ldg(reinterpret_cast<const uint4*>(ve) + i);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (h0 + u < H) {
        const float a = 1.f / (1.f + expf(-g[u]));
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          const uint32_t xs[4] = {x[u][i2].x, x[u][i2].y, x[u][i2].z, x[u][i2].w};
          const uint32_t es[4] = {e[u][i2].x, e[u][i2].y, e[u][i2].z, e[u][i2].w};
          uint32_t o[4];
#pragma unroll
          for (int w = 0; w < 4; ++w)
            o[w] = pack_bf16x2(fmaf(a, bf16_lo(es[w]), bf16_lo(xs[w])), fmaf(a, bf16_hi(es[w]), bf16_hi(xs[w])));
          reinterpret_cast<uint4*>(vmix)[(h0 + u) * 16 + kq + 8 * i2] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
}

// Copies n 16-byte words, lane kq of an 8-lane group taking words kq, kq + 8, ..., with eight loads in flight
// before the stores.  src and dst do not overlap.
__device__ __forceinline__ void copy_words(uint4* dst, const uint4* src, int n, int kq) {
  for (int i0 = kq; i0 < n; i0 += 64) {
    uint4 t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i0 + 8 * u < n) t[u] = src[i0 + 8 * u];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i0 + 8 * u < n) dst[i0 + 8 * u] = t[u];
  }
}

constexpr int kPrologueThreads = 256;
constexpr int kPrologueTokensPerBlock = kPrologueThreads / 8;  // 8-lane groups per block
constexpr int kMaxSlices = 4;

// A token's work split over n_slices 8-lane groups, so that short inputs still give every SM enough groups: slice sl
// takes heads [H sl / n, H (sl + 1) / n) of its H = Hq + Hkv q and k heads and the same share of its Hkv value heads.
struct Slice {
  int tok, i0, i1, v0, v1;
};
__device__ __forceinline__ Slice slice_of(int gid, int n_slices, int Hq, int Hkv) {
  Slice r;
  r.tok = gid / n_slices;
  const int sl = gid - r.tok * n_slices, H = Hq + Hkv;
  r.i0 = H * sl / n_slices;
  r.i1 = H * (sl + 1) / n_slices;
  r.v0 = Hkv * sl / n_slices;
  r.v1 = Hkv * (sl + 1) / n_slices;
  return r;
}

// OutT: __nv_bfloat16 (qn, kn in bf16) or uint8_t (qn, kn in e4m3, scaled by q_scale and k_scale).
template <typename OutT>
__global__ void __launch_bounds__(kPrologueThreads)
    qk_prologue_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       OutT* __restrict__ qn, OutT* __restrict__ kn, int BT, int T, int Hq,
                       int Hkv, const __grid_constant__ RopeTable tab, float q_scale, float k_scale, unsigned* zero_word,
                       const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ ve,
                       const __nv_bfloat16* __restrict__ ve_gate, __nv_bfloat16* __restrict__ vmix, int n_slices) {
  // The attention kernel that follows in stream order may be scheduled now; it waits for this grid to complete
  // before reading anything written here.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The attention kernel takes its work items from this counter.
  if (zero_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0u;
  const Slice w = slice_of(blockIdx.x * kPrologueTokensPerBlock + (threadIdx.x >> 3), n_slices, Hq, Hkv);
  const int tok = w.tok;
  const int kq = threadIdx.x & 7;
  if (tok >= BT) return;  // whole 8-lane groups leave together
  const unsigned gmask = 0xFFu << ((threadIdx.x & 31) & ~7);
  const __nv_bfloat16* qt = q + static_cast<size_t>(tok) * Hq * 128;
  const __nv_bfloat16* kt = k + static_cast<size_t>(tok) * Hkv * 128;
  uint4 lo0[4], hi0[4];
  load_first_heads(qt, kt, Hq, w.i0, w.i1, kq, lo0, hi0);
  const float pos = static_cast<float>(tok % T);
  float c[8], s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rope_cos_sin(pos, tab.hi[kq * 8 + i], tab.lo[kq * 8 + i], c[i], s[i]);
  rope_norm_token(qt, kt, qn + static_cast<size_t>(tok) * Hq * 128, kn + static_cast<size_t>(tok) * Hkv * 128, Hq,
                  w.i0, w.i1, kq, c, s, gmask, q_scale, k_scale, lo0, hi0);
  if (ve != nullptr) {
    const size_t o = static_cast<size_t>(tok) * Hkv + w.v0;
    mix_values(v + o * 128, ve + o * 128, ve_gate + o, vmix + o * 128, w.v1 - w.v0, kq);
  }
}

// Chunked prefill against a KV cache ("nanochat Admin & Developer Guide", section 6, SDPA case 3 "chunked /
// sliding-window inference"; section 7, the in-place KV-cache append).  For sequence b with p0 = cache_lens[b]:
//   * the chunk's queries q[b, t] and keys k_new[b, t] are roped at position p0 + t and normed; qn goes to the
//     workspace (times q_scale), the keys go straight into kcache[b, p0 + t] and the values v_new[b, t] into
//     vcache[b, p0 + t] (with a value embedding: v_new + sigmoid(ve_gate) ve_new, rounded to bf16 once);
//   * the V tile that holds the chunk's last key (rows [128 hb, 128 hb + 128), hb = (p0 + Tq - 1) / 128) is copied
//     into vtail[b] with the rows past the chunk set to zero, so that the attention kernel never multiplies a zero
//     probability by whatever the cache holds beyond its valid rows;
//   * a sequence whose p0 is outside [0, Tcap - Tq] gets a zero output, its cache is left alone and the device
//     status records NC_DEV_BAD_CACHE_LEN.
// Blocks [0, n_tok_blocks) take one slice of a token per 8-lane group, the rest one row of a V tail copy per group.
// Two blocks per SM (at most 128 registers a thread), as for the full-prefill prologue.
__global__ void __launch_bounds__(kPrologueThreads, 2)
    chunk_prologue_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
                          const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* __restrict__ qn,
                          __nv_bfloat16* kcache, __nv_bfloat16* vcache, __nv_bfloat16* __restrict__ vtail,
                          __nv_bfloat16* __restrict__ out, const int* __restrict__ cache_lens, int B, int Tq, int Hq,
                          int Hkv, int Tcap, int n_tok_blocks, const __grid_constant__ RopeTable tab, float q_scale,
                          unsigned* zero_word, const __nv_bfloat16* __restrict__ ve_new,
                          const __nv_bfloat16* __restrict__ ve_gate, int n_slices) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (zero_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0u;
  const int grp = threadIdx.x >> 3;
  const int kq = threadIdx.x & 7;
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  if (static_cast<int>(blockIdx.x) < n_tok_blocks) {
    const Slice w = slice_of(blockIdx.x * kPrologueTokensPerBlock + grp, n_slices, Hq, Hkv);
    const int tok = w.tok;
    if (tok >= B * Tq) return;  // whole 8-lane groups leave together
    const int b = tok / Tq, t = tok - b * Tq;
    // Everything read from the chunk is independent of the cache length: the first round of q / k heads and the
    // first value words of this slice are requested together with it.
    const __nv_bfloat16* qt = q + static_cast<size_t>(tok) * Hq * 128;
    const __nv_bfloat16* kt = k_new + static_cast<size_t>(tok) * Hkv * 128;
    const size_t vo = static_cast<size_t>(tok) * Hkv + w.v0;  // this slice's value heads
    const int vw = (w.v1 - w.v0) * 16;                        // and their 16-byte words
    const uint4* vs = reinterpret_cast<const uint4*>(v_new + vo * 128);
    const int p0 = __ldg(cache_lens + b);
    uint4 lo0[4], hi0[4], v0[4];
    load_first_heads(qt, kt, Hq, w.i0, w.i1, kq, lo0, hi0);
    const bool plain_v = ve_new == nullptr;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (plain_v && kq + 8 * u < vw) v0[u] = __ldg(vs + kq + 8 * u);
    if (p0 < 0 || p0 > Tcap - Tq) {
      if (w.i0 > 0) return;  // the token's first slice writes its zero output row
      uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(tok) * Hq * 128);
      for (int i = kq; i < Hq * 16; i += 8) o[i] = zero4;
      if (t == 0 && kq == 0) raise_status(NC_DEV_BAD_CACHE_LEN);
      return;
    }
    const unsigned gmask = 0xFFu << ((threadIdx.x & 31) & ~7);
    const int pos = p0 + t;
    float c[8], s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) rope_cos_sin(static_cast<float>(pos), tab.hi[kq * 8 + i], tab.lo[kq * 8 + i], c[i], s[i]);
    const size_t row = static_cast<size_t>(b) * Tcap + pos;  // cache row of this token
    uint4* vd = reinterpret_cast<uint4*>(vcache + (row * Hkv + w.v0) * 128);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (plain_v && kq + 8 * u < vw) vd[kq + 8 * u] = v0[u];
    rope_norm_token(qt, kt, qn + static_cast<size_t>(tok) * Hq * 128, kcache + row * Hkv * 128, Hq, w.i0, w.i1, kq,
                    c, s, gmask, q_scale, 1.0f, lo0, hi0);
    if (!plain_v) {  // the chunk's values with their gated embedding, into the cache
      mix_values(v_new + vo * 128, ve_new + vo * 128, ve_gate + vo, vcache + (row * Hkv + w.v0) * 128, w.v1 - w.v0,
                 kq);
      return;
    }
    if (vw > 32) copy_words(vd + 32, vs + 32, vw - 32, kq);  // words past the first four per lane
    return;
  }
  // V tail copy: row i of sequence b
  const int id = (blockIdx.x - n_tok_blocks) * kPrologueTokensPerBlock + grp;
  if (id >= B * 128) return;
  const int b = id >> 7, i = id & 127;
  const int p0 = __ldg(cache_lens + b);
  if (p0 < 0 || p0 > Tcap - Tq) return;
  const int key = ((p0 + Tq - 1) / 128) * 128 + i;
  uint4* d = reinterpret_cast<uint4*>(vtail + (static_cast<size_t>(b) * 128 + i) * Hkv * 128);
  if (key < p0) {  // an earlier cache row (not written by this kernel)
    copy_words(d, reinterpret_cast<const uint4*>(vcache + (static_cast<size_t>(b) * Tcap + key) * Hkv * 128),
               Hkv * 16, kq);
  } else if (key < p0 + Tq) {  // a row of the chunk (mixed with its value embedding, as the cache row is)
    const size_t tk = static_cast<size_t>(b) * Tq + (key - p0);
    if (ve_new != nullptr) {
      mix_values(v_new + tk * Hkv * 128, ve_new + tk * Hkv * 128, ve_gate + tk * Hkv,
                 vtail + (static_cast<size_t>(b) * 128 + i) * Hkv * 128, Hkv, kq);
    } else {
      copy_words(d, reinterpret_cast<const uint4*>(v_new + tk * Hkv * 128), Hkv * 16, kq);
    }
  } else {
    for (int e = kq; e < Hkv * 16; e += 8) d[e] = zero4;
  }
}

}  // namespace nc
