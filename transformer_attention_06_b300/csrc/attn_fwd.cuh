// K2: causal / sliding-window GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ("nanochat Admin & Developer Guide", sections 3 and 6): for query row (b, t, h) with kv head
// g = h / G, out = softmax_j(qn . kn_j / sqrt(D)) . v_j over the visible keys j (j <= t, and t - j <= window when
// window >= 0).  qn / kn are the roped + normed vectors written by K1.
//
// Tiling.  One CTA owns one tile of 128 MMA rows: P = 128 / G consecutive query positions times the G query heads
// of kv head g (row r = position (r / G), head (r % G)), so every K/V tile brought in by TMA is shared by the whole
// GQA group.  Keys are processed in tiles of 128; only tiles that intersect the causal / window band of the query
// tile are visited, and only tiles that straddle the band edge pay for the element mask.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread r owns TMEM lane r = query row r; online softmax in the log2 domain, writes P
//              (bf16) over its S row in TMEM, rescales its O row when the row maximum grows, and runs the epilogue;
//   warp 4     TMA producer: Q tile once, then K and V tiles through a 2-stage ring;
//   warp 5     TMEM allocator and MMA issuer (one thread): S = Q K^T into one of two S buffers, O += P V with P read
//              from TMEM (A operand) and V from shared memory (MN-major B operand).
// TMEM (512 columns): S0 = [0,128), S1 = [128,256), O = [256,384); P_i overlays the first 64 columns of S_i.
// Shared memory: Q 32 KB + 2 x (K 32 KB + V 32 KB), all in the 128-byte-swizzled K-major layout written by TMA.
#pragma once

#include <climits>

#include "common.cuh"

namespace nc {
namespace fwd {

constexpr int kD = 128;
constexpr int kBlockN = 128;                  // keys per KV tile
constexpr int kStages = 2;
constexpr int kHalfBytes = 128 * 128;         // one 64-column half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalfBytes;    // 32 KB
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);  // A = Q, B = K, both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);   // A = P (TMEM), B = V (MN-major)

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
constexpr int kOffMisc = kOffBar + 16 * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;   // + slack to align the base to 1024 bytes

struct Params {
  __nv_bfloat16* out;
  int B, T, Hq, Hkv, G, P, n_qtiles, window;
  float scale_log2;                   // log2(e) / sqrt(D)
  unsigned long long wait_limit_ns;
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [kStages]
  uint64_t* v_full = bars + 3;    // [kStages]
  uint64_t* kv_empty = bars + 5;  // [kStages]
  uint64_t* s_full = bars + 7;    // [2]  S_i written by the MMA
  uint64_t* p_full = bars + 9;    // [2]  P_i written (and O rescaled) by the 128 softmax threads
  uint64_t* o_done = bars + 11;   // one completion per P.V product
  uint64_t* mma_final = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x / p.Hkv;
  const int g = blockIdx.x - b * p.Hkv;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // heaviest (latest) query tiles first
  const int t0 = qt * p.P;
  const int t_last = min(t0 + p.P, p.T) - 1;
  const int key_lo = p.window < 0 ? 0 : max(0, t0 - p.window);
  const int kt0 = key_lo / kBlockN;
  const int n_kv = t_last / kBlockN - kt0 + 1;
  const int rows_used = p.G * p.P;
  const unsigned long long lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(p_full + s, 128);
    }
    mbar_init(o_done, 1);
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x < 128 && static_cast<int>(threadIdx.x) >= rows_used) {
    // Rows of the Q tile that TMA does not fill (128 is not a multiple of G): zero them so they stay finite.
    uint4* r0 = reinterpret_cast<uint4*>(sQ + threadIdx.x * 128);
    uint4* r1 = reinterpret_cast<uint4*>(sQ + kHalfBytes + threadIdx.x * 128);
    for (int i = 0; i < 8; ++i) {
      r0[i] = make_uint4(0, 0, 0, 0);
      r1[i] = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, 2u * 128u * static_cast<uint32_t>(rows_used));
      tma_load_4d(sQ, &tmQ, q_full, 0, g * p.G, t0, b);
      tma_load_4d(sQ + kHalfBytes, &tmQ, q_full, 64, g * p.G, t0, b);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (j >= kStages && !mbar_wait(kv_empty + st, ((j >> 1) - 1) & 1, lim, abort_flag)) break;
        const int s0 = (kt0 + j) * kBlockN;
        uint8_t* dk = sK + st * kTileBytes;
        uint8_t* dv = sV + st * kTileBytes;
        mbar_arrive_expect_tx(k_full + st, kTileBytes);
        tma_load_4d(dk, &tmK, k_full + st, 0, g, s0, b);
        tma_load_4d(dk + kHalfBytes, &tmK, k_full + st, 64, g, s0, b);
        mbar_arrive_expect_tx(v_full + st, kTileBytes);
        tma_load_4d(dv, &tmV, v_full + st, 0, g, s0, b);
        tma_load_4d(dv + kHalfBytes, &tmV, v_full + st, 64, g, s0, b);
        issued = j + 1;
      }
      // Every copy this CTA started must land before the CTA exits (already true on the normal path).
      mbar_wait(q_full, 0, lim, nullptr);
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        mbar_wait(k_full + (j & 1), (j >> 1) & 1, lim, nullptr);
        mbar_wait(v_full + (j & 1), (j >> 1) & 1, lim, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t aK = smem_u32(sK);
      const uint32_t aV = smem_u32(sV);
      bool ok = mbar_wait(q_full, 0, lim, abort_flag);
      tc_fence_after_sync();
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {  // S_j = Q K_j^T
          const int st = j & 1;
          if (!(ok = mbar_wait(k_full + st, (j >> 1) & 1, lim, abort_flag))) break;
          tc_fence_after_sync();
          const uint32_t dS = tbase + kColS + st * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            umma_ss(dS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + st * kTileBytes + off, 16, 1024),
                    kIdescQK, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full + st);
        }
        if (j > 0) {  // O += P_{j-1} V_{j-1}
          const int i = j - 1;
          const int st = i & 1;
          if (!(ok = mbar_wait(p_full + st, (i >> 1) & 1, lim, abort_flag))) break;
          if (!(ok = mbar_wait(v_full + st, (i >> 1) & 1, lim, abort_flag))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            umma_ts(tbase + kColO, tbase + kColS + st * 128 + kk * 8,
                    sdesc_sw128(aV + st * kTileBytes + kk * 2048, kHalfBytes, 1024), kIdescPV,
                    (i > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(o_done);
          umma_commit(kv_empty + st);
        }
      }
      umma_commit(mma_final);  // all issued MMAs complete before TMEM is released
      mbar_wait(mma_final, 0, lim, nullptr);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    const int r = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int tpos = r / p.G;
    const int jh = r - tpos * p.G;
    const int t = t0 + tpos;
    const bool row_ok = (r < rows_used) && (t < p.T);
    const float sl2 = p.scale_log2;
    const uint32_t tO = tbase + lane_base + kColO;
    float m = -INFINITY;  // running maximum of the raw scores of this row
    float l = 0.f;        // running softmax denominator (relative to m)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      ok = mbar_wait(s_full + st, (j >> 1) & 1, lim, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t tS = tbase + lane_base + kColS + st * 128;
      uint32_t sv[4][32];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(tS + c4 * 32, sv[c4]);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) tmem_ld_wait(sv[c4]);

      const int s0 = (kt0 + j) * kBlockN;
      const bool full_tile = (s0 + kBlockN - 1 <= t0) && (p.window < 0 || t_last - s0 <= p.window);
      float mt = -INFINITY;
      if (full_tile) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
          for (int c = 0; c < 32; ++c) mt = fmaxf(mt, __uint_as_float(sv[c4][c]));
      } else {
        const int hi_c = t - s0;                                        // key index <= t
        const int lo_c = p.window < 0 ? INT_MIN : t - s0 - p.window;  // t - key <= window
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int col = c4 * 32 + c;
            float x = __uint_as_float(sv[c4][c]);
            if (col > hi_c || col < lo_c) x = -INFINITY;
            sv[c4][c] = __float_as_uint(x);
            mt = fmaxf(mt, x);
          }
      }
      const float m_new = fmaxf(m, mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // a row with nothing visible yet keeps P = 0
      const float nms = -m_use * sl2;
      const float corr = ex2_approx((m - m_use) * sl2);           // 0 on the first visible tile
      float rs = 0.f;
      uint32_t pk[4][16];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sv[c4][2 * c]), sl2, nms));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sv[c4][2 * c + 1]), sl2, nms));
          rs += p0 + p1;
          pk[c4][c] = pack_bf16x2(p0, p1);
        }
      l = fmaf(l, corr, rs);
      if (j > 0) {
        // O holds the sum over tiles < j once the previous P.V has completed; rescale it to the new maximum.
        ok = mbar_wait(o_done, (j - 1) & 1, lim, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, corr < 1.0f)) {
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t ov[32];
            tmem_ld32(tO + c4 * 32, ov);
            tmem_ld_wait(ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * corr);
            tmem_st32(tO + c4 * 32, ov);
          }
        }
      }
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) tmem_st16(tS + c4 * 16, pk[c4]);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(p_full + st);
      m = m_new;
    }
    if (ok) {
      ok = mbar_wait(o_done, (n_kv - 1) & 1, lim, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after_sync();
      const float inv_l = 1.f / l;
      uint4* dst = reinterpret_cast<uint4*>(
          p.out + ((static_cast<size_t>(b) * p.T + (row_ok ? t : 0)) * p.Hq + g * p.G + jh) * kD);
#pragma unroll 1
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t ov[32];
        tmem_ld32(tO + c4 * 32, ov);
        tmem_ld_wait(ov);
        if (row_ok) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint32_t q4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              q4[e] = pack_bf16x2(__uint_as_float(ov[8 * w + 2 * e]) * inv_l,
                                  __uint_as_float(ov[8 * w + 2 * e + 1]) * inv_l);
            dst[c4 * 4 + w] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
          }
        }
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

}  // namespace fwd
}  // namespace nc
