// K2: causal / sliding-window GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ("nanochat Admin & Developer Guide", sections 3 and 6): for query row (b, t, h) with kv head
// g = h / G, out = softmax_j(qn . kn_j / sqrt(D)) . v_j over the visible keys j (j <= t, and t - j <= window when
// window >= 0).  qn / kn are the roped + normed vectors written by K1.  With per-sequence offsets p0 (chunked
// prefill against a KV cache, "nanochat Admin & Developer Guide" section 6, SDPA case 3), query t sits at
// position p0 + t and the keys come from the cache: positions replace t in the band and the mask.
//
// Tiling.  A Q tile is 128 MMA rows: P = 128 / G consecutive query positions times the G query heads of kv head g
// (row r = position r / G, head r % G), so every K/V tile brought in by TMA serves the whole GQA group.  A work item
// is two consecutive Q tiles (A and B) of one (b, g): every K/V tile is loaded once for both.  When pairs would
// leave SMs without an item, an item is a single Q tile whose key range runs as two chains A and B (first and second
// half of its key tiles, visited alternately) whose partial sums the epilogue adds.  Keys are processed in tiles of 128; a Q tile only visits the key tiles
// that intersect its causal / window band, and only tiles that straddle the band edge pay for the element mask.
//
// Persistent grid: one CTA per SM takes work items from a global counter (zeroed by the prologue kernel), the
// latest (heaviest under a causal mask) Q tiles first, so the tail of the launch is made of the lightest items.
//
// Warp roles (384 threads, three warpgroups; launched at 168 registers per thread, the softmax warpgroups take 208
// and the third warpgroup keeps 88: 2 x 128 x 208 + 128 x 88 = 384 x 168):
//   warps 0-7   softmax and epilogue.  Both Q tiles are handled by all eight warps, one tile at a time (A, then B,
//               in every key-tile round), so each tile's softmax runs alone on the exponential and issue units
//               while the tensor core works on the other tile.  Thread (warp w, lane) owns row r = 32 (w % 4) + lane
//               (= TMEM lane r) and the column half h = w / 4: exponentials of its 64 base-2 logits (no running
//               maximum, see below), P (bf16) written over its part of the S row in TMEM, and its half of the
//               epilogue.  The two halves of a row combine their row sums only in the epilogue, which writes
//               O / l into a shared-memory staging tile that one thread sends out with a TMA store;
//   warp 8      TMA producer and scheduler: fetches work items and serves three queues in whichever order their
//               buffers free up -- Q_A, Q_B once per item, K and V tiles through 2-stage rings;
//   warps 9, 10 MMA issuers, one per Q tile X (warp 9 also allocates TMEM; warp 11 idle): per key tile j,
//               O_X += P_X(j) V_j then S_X = Q_X K_{j+1}^T.  The two tiles' chains are independent (disjoint TMEM,
//               and a commit only tracks its own thread's MMAs), so the tensor core serves whichever tile is ready
//               while the other tile's softmax runs.  K, V stages and the Q tiles are released by one commit from
//               each issuer (barriers of count 2).
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512); P_X (bf16 pairs) overlays S_X:
// the P of keys [64 h, 64 h + 64) goes to columns [64 h, 64 h + 32), inside the S columns the same thread read.  Shared memory: Q_A, Q_B 32 KB each, 2-stage K and V rings of 32 KB tiles, all in the
// 128-byte-swizzled K-major layout written by TMA, and one 32 KB output staging tile in the same layout.
#pragma once

#include <climits>

#include "common.cuh"

namespace nc {
namespace fwd {

constexpr int kD = 128;
constexpr int kBlockN = 128;                  // keys per KV tile
constexpr int kKStages = 2;                   // K ring: a stage is free once both S products of its tile are done
constexpr int kVStages = 2;                   // V ring: a stage is free once both P.V products of its tile are done
constexpr int kHalfBytes = 128 * 128;         // one 64-column half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalfBytes;    // 32 KB
constexpr int kSoftThreads = 128;             // one softmax warpgroup = the 128 rows (TMEM lanes) of a Q tile
constexpr int kSoftWarps = 8;                 // softmax warps; each arrives once on p_full / o_free
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;                   // MMA issuer of Q tile A; also allocates TMEM
constexpr int kMmaWarpB = 10;                 // MMA issuer of Q tile B
constexpr int kThreads = 384;
constexpr uint32_t kRegsSoftmax = 208, kRegsOther = 88;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                 // S_X at kColS + 128 X
constexpr uint32_t kColO = 256;               // O_X at kColO + 128 X
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);  // A = Q, B = K, both K-major
constexpr uint32_t kIdescQK8 = idesc_e4m3_f32(128, 128);                // the same with e4m3 Q and K
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);   // A = P (TMEM), B = V (MN-major)
// Softmax without a running maximum.  kn and qn are RMS-normalised by the prologue (RMSNorm without weight,
// eps > 0), and qn leaves it multiplied by c = g log2(e) / sqrt(128) (g: the QK-norm gain, 1 or e.g. 1.2, at most
// 4), so the S tile holds base-2 logits.  Before rounding, |kn| <= sqrt(128) and |qn| <= c sqrt(128); bf16 rounding
// adds at most a factor (1 + 2^-9) to each, so |S| <= c 128 (1 + 2^-9)^2 < 16.5 g <= 66.  P = 2^S then lies in
// [2^-66, 2^66] -- no overflow or underflow in fp32 or bf16, and row sums of at most 2^31 keys stay below 2^97 --
// so the exponentials need no offset and neither O nor the row sums ever need rescaling; softmax(x) =
// 2^S / sum 2^S exactly as with a maximum.

// mbarrier slots (each 8 bytes), derived from the ring depths so that no two barriers can overlap.
constexpr int kBarKFull = 0;
constexpr int kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarVFull = kBarKEmpty + kKStages;
constexpr int kBarVEmpty = kBarVFull + kVStages;
constexpr int kBarQFull = kBarVEmpty + kVStages;
constexpr int kBarQEmpty = kBarQFull + 2;
constexpr int kBarSFull = kBarQEmpty + 1;
constexpr int kBarPFull = kBarSFull + 2;
constexpr int kBarODone = kBarPFull + 2;
constexpr int kBarOFree = kBarODone + 2;
constexpr int kBarSchedFull = kBarOFree + 2;
constexpr int kBarSchedEmpty = kBarSchedFull + 2;
constexpr int kBarMmaFinal = kBarSchedEmpty + 2;   // [2], one per MMA warp
constexpr int kNumBars = kBarMmaFinal + 2;
static_assert(kNumBars <= 32, "barrier block");
// The dynamic shared memory base is aligned up to 1024 bytes inside the kernel; 768 bytes of slack cover bases
// that are at least 256-byte aligned (in practice it is 1024-byte aligned), and the kernel checks this.
constexpr int kAlignSlack = 768;

// Shared-memory layout.  Q and K tiles hold 128 rows of 128 elements: 32 KB in bf16 (two 64-column halves of 128
// bytes per row), 16 KB in e4m3 (one 128-byte row each).  V and the output staging tile are bf16 in both variants.
template <bool kFp8>
struct Smem {
  static constexpr int kQKBytes = kFp8 ? 128 * 128 : kTileBytes;  // one Q or K tile
  static constexpr int kOffQ = 0;                                  // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kQKBytes;
  static constexpr int kOffV = kOffK + kKStages * kQKBytes;
  static constexpr int kOffO = kOffV + kVStages * kTileBytes;      // output staging of one Q tile (TMA store source)
  static constexpr int kOffBar = kOffO + kTileBytes;
  static constexpr int kOffXch = kOffBar + kNumBars * 8;           // row-sum exchange, [2 halves][128] f32 (1 KB used)
  static constexpr int kOffMisc = kOffXch + 2048;
  static constexpr int kBytes = kOffMisc + 16 + kAlignSlack;
  static_assert(kBytes <= 232448, "shared memory budget");
};
constexpr int kSmemBytes = Smem<false>::kBytes;
constexpr int kSmemBytesFp8 = Smem<true>::kBytes;

struct Params {
  __nv_bfloat16* out;
  unsigned* item_ctr;                 // work-item counter, zero at launch (written by the prologue kernel)
  // Position of query 0 of sequence b (chunked prefill against a cache: the cache length); null means 0.
  const int* pos0;
  // n_pairs: work items per (b, kv head) (pairs of Q tiles, or single tiles when tiles_per_item is 1)
  int B, T, Hq, Hkv, G, P, n_pairs, n_items, window;
  int tiles_per_item;                 // 2 (Q tiles A and B share every K/V tile), or 1 when pairs would leave SMs idle
  int Tk;                             // key rows per sequence that the K / V maps address (T, or the cache size)
  unsigned long long wait_limit_ns;
  // Row statistics for the backward pass (all null in a plain forward).  When `lse` is set, every query row's
  // log2(sum_j 2^S_j) of its base-2 logits is written at lse[((b Hkv + g) n_qtiles + m) 128 + r] (Q tile m, tile row
  // r); when `drow` is also set, rowsum(dout * out) of the row (fp32 out, before rounding) goes to the same index of
  // drow, dout being [B, T, Hq, 128] bf16.  `store_out` = 0 skips writing out.
  float* lse;
  float* drow;
  const __nv_bfloat16* dout;
  int n_qtiles;
  int store_out;
};

// Key-tile range of one Q tile: tiles [lo, hi] intersect its band; n = 0 when the tile lies past T.  Query rows
// t0 .. t_last sit at positions a0 .. a_last (= p0 + t).
struct QRange {
  int t0, t_last, a0, a_last, lo, hi, n;
};

__device__ __forceinline__ QRange q_range(const Params& p, int t0, int p0) {
  QRange q;
  q.t0 = t0;
  q.a0 = p0 + t0;
  if (t0 >= p.T) {
    q.t_last = t0 - 1;
    q.a_last = q.a0 - 1;
    q.lo = 0;
    q.hi = -1;
    q.n = 0;
    return q;
  }
  q.t_last = min(t0 + p.P, p.T) - 1;
  q.a_last = p0 + q.t_last;
  const int key_lo = p.window < 0 ? 0 : max(0, q.a0 - p.window);
  q.lo = key_lo / kBlockN;
  q.hi = q.a_last / kBlockN;
  q.n = q.hi - q.lo + 1;
  return q;
}

// A work item walks its key tiles in rounds, one K/V tile per round.  Two-tile items (split = false): round i visits
// key tile lo + i, which Q tile X uses when it lies in X's range.  Single-tile items (split = true): the tile's key
// range is cut into two halves run as two chains -- chain A over the first na tiles, chain B over the last nb --
// visited alternately (A, B, A, B, ..., then A's last tile when na > nb), so that each chain's softmax overlaps the
// other chain's products.  Without a running maximum the partial sums of the two chains add up exactly: the epilogue
// returns (O_A + O_B) / (l_A + l_B).
struct Item {
  int b, g;
  QRange qa, qb;
  int lo, hi;   // union of the two key-tile ranges
  int na, nb;   // split: rounds of chain A and of chain B
  int tail;     // key tile read from the zero-padded V tail copy (-1: none)
  bool valid;   // false: the sequence's cache length is out of range; nothing is stored
  bool split;
};

__device__ __forceinline__ Item decode_item(const Params& p, int item) {
  Item it;
  const int bh = p.B * p.Hkv;
  const int pair = p.n_pairs - 1 - item / bh;  // latest Q tiles first
  const int bg = item - (item / bh) * bh;
  it.b = bg / p.Hkv;
  it.g = bg - it.b * p.Hkv;
  const int pp = p.pos0 != nullptr ? __ldg(p.pos0 + it.b) : 0;
  it.valid = pp >= 0 && pp <= p.Tk - p.T;
  const int p0 = it.valid ? pp : 0;
  // n_pairs counts the items of one (b, g); with one tile per item, tile B starts past T (empty)
  it.qa = q_range(p, pair * p.tiles_per_item * p.P, p0);
  it.qb = q_range(p, p.tiles_per_item == 2 ? pair * 2 * p.P + p.P : p.T, p0);
  it.lo = it.qa.lo;
  it.hi = it.qb.n > 0 ? max(it.qa.hi, it.qb.hi) : it.qa.hi;
  // The statistics launch of the backward keeps one chain per item: its row sums then add the key tiles in the same
  // order whether the items are pairs or single tiles, so the gradients do not depend on the batch composition.
  it.split = p.tiles_per_item == 1 && p.lse == nullptr;
  it.na = (it.qa.n + 1) / 2;
  it.nb = it.qa.n / 2;
  it.tail = p.pos0 != nullptr ? (p0 + p.T - 1) / kBlockN : -1;
  return it;
}

__device__ __forceinline__ int n_rounds(const Item& it) { return it.hi - it.lo + 1; }

// key tile of round i
__device__ __forceinline__ int round_tile(const Item& it, int i) {
  if (!it.split) return it.lo + i;
  return i < 2 * it.nb ? it.lo + ((i & 1) ? it.na : 0) + (i >> 1) : it.lo + i - it.nb;
}

// chain (Q tile) x takes part in round i
__device__ __forceinline__ bool in_chain(const Item& it, int x, int i) {
  if (it.split) return x == 0 ? (i >= 2 * it.nb || (i & 1) == 0) : (i < 2 * it.nb && (i & 1) == 1);
  const QRange& q = x == 0 ? it.qa : it.qb;
  const int j = it.lo + i;
  return q.n > 0 && j >= q.lo && j <= q.hi;
}

// chain x has at least one round, and its first round
__device__ __forceinline__ bool chain_active(const Item& it, int x) {
  return it.split ? (x == 0 ? it.na > 0 : it.nb > 0) : (x == 0 ? it.qa.n > 0 : it.qb.n > 0);
}
__device__ __forceinline__ int first_round(const Item& it, int x) {
  return it.split ? x : (x == 0 ? it.qa.lo : it.qb.lo) - it.lo;
}

// kFp8: qn and kn are e4m3 (scores on tcgen05 kind::f8f6f4); otherwise bf16 (kind::f16).  P and V are bf16 in both.
template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmVt,
                    const __grid_constant__ CUtensorMap tmO, const Params p) {
  using L = Smem<kFp8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sO = smem + L::kOffO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* k_full = bars + kBarKFull;        // [kKStages]  TMA -> MMA
  uint64_t* k_empty = bars + kBarKEmpty;      // [kKStages]  MMA -> TMA
  uint64_t* v_full = bars + kBarVFull;        // [kVStages]  TMA -> MMA
  uint64_t* v_empty = bars + kBarVEmpty;      // [kVStages]  MMA -> TMA
  uint64_t* q_full = bars + kBarQFull;        // [2]  Q_A, Q_B of the current item               TMA -> MMA
  uint64_t* q_empty = bars + kBarQEmpty;      //      every S of the item complete               MMA -> TMA
  uint64_t* s_full = bars + kBarSFull;        // [2]  S_X written                                MMA -> softmax X
  uint64_t* p_full = bars + kBarPFull;        // [2]  P_X written (one arrival per softmax warp) softmax -> MMA
  uint64_t* o_done = bars + kBarODone;        // [2]  P_X V product complete                     MMA -> softmax X
  uint64_t* o_free = bars + kBarOFree;        // [2]  O_X read by the epilogue (one per warp)    softmax -> MMA
  uint64_t* sched_full = bars + kBarSchedFull;    // [2]  work item published                     TMA -> all
  uint64_t* sched_empty = bars + kBarSchedEmpty;  // [2]  work item read (2 MMA warps + the softmax warps)
  uint64_t* mma_final = bars + kBarMmaFinal;
  float* xch = reinterpret_cast<float*>(smem + L::kOffXch);
  int* misc = reinterpret_cast<int*>(smem + L::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;
  int* sched = misc + 2;            // [2] work-item ring

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned long long lim = p.wait_limit_ns;
  if (static_cast<int>(smem - smem_raw) > kAlignSlack) {  // uniform: every thread sees the same base
    if (threadIdx.x == 0) raise_status(NC_DEV_SMEM_BASE);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 2);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(q_full + x, 1);
      mbar_init(s_full + x, 1);
      mbar_init(p_full + x, kSoftWarps);
      mbar_init(o_done + x, 1);
      mbar_init(o_free + x, kSoftWarps);
      mbar_init(sched_full + x, 1);
      mbar_init(sched_empty + x, 3);
    }
    mbar_init(q_empty, 2);
    mbar_init(mma_final + 0, 1);
    mbar_init(mma_final + 1, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x < 256 && p.G * p.P < 128) {
    // Rows of the Q tiles that TMA never fills (128 is not a multiple of G): zero them once so they stay finite.
    const int x = threadIdx.x >> 7, r = threadIdx.x & 127;
    if (r >= p.G * p.P) {
      uint4* r0 = reinterpret_cast<uint4*>(sQ + x * L::kQKBytes + r * 128);
      for (int i = 0; i < 8; ++i) r0[i] = make_uint4(0, 0, 0, 0);
      if (!kFp8) {
        uint4* r1 = reinterpret_cast<uint4*>(sQ + x * L::kQKBytes + kHalfBytes + r * 128);
        for (int i = 0; i < 8; ++i) r1[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  // Everything above ran concurrently with the tail of the prologue kernel; qn, kn and the work counter are read
  // only after it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // one Q tile: box {64, G, P, 1} x 2 in bf16, {128, G, P, 1} in e4m3
  const uint32_t q_bytes = (kFp8 ? 1u : 2u) * 128u * static_cast<uint32_t>(p.G * p.P);
  if (warp >= 8) {
    warpgroup_reg_dec<kRegsOther>();
    if (warp == kProducerWarp && lane == 0) {
      // ---------------------------------------------------------------- scheduler + TMA producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      if (p.pos0 != nullptr) tma_prefetch_desc(&tmVt);
      // Items fetched so far live in a 2-slot ring (the same slots the consumers read).  Three cursors walk the
      // item sequence: Q (item iq), K (item ik, round jk), V (item iv, round jv); kt / vt count the K / V tiles
      // loaded over all items (ring positions).
      Item items[2];
      int nfetched = 0;
      bool done = false;          // the counter ran past the last item
      int iq = 0, ik = 0, iv = 0, jk = 0, jv = 0, kt = 0, vt = 0;
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      bool ok = true;
      while (ok) {
        bool progress = false;
        // fetch the next item once the K cursor needs it and its slot has been read by every consumer
        if (!done && ik == nfetched && nfetched - min(iq, iv) < 2 &&
            (nfetched < 2 || mbar_test(sched_empty + (nfetched & 1), ((nfetched >> 1) - 1) & 1))) {
          const int slot = nfetched & 1;
          const int item = static_cast<int>(atomicAdd(p.item_ctr, 1u));
          sched[slot] = item < p.n_items ? item : -1;
          mbar_arrive(sched_full + slot);
          if (item >= p.n_items) {
            done = true;
          } else {
            items[slot] = decode_item(p, item);
            jk = 0;
            if (nfetched == iv) jv = 0;
            ++nfetched;
          }
          progress = true;
        }
        // Q tiles of item iq, once every S of item iq - 1 has completed
        if (iq < nfetched && (iq == 0 || mbar_test(q_empty, (iq - 1) & 1))) {
          const Item& it = items[iq & 1];
          // past T the box reads as zeros (still full bytes)
#pragma unroll
          for (int x = 0; x < 2; ++x) {  // a split item's two chains use the same Q tile
            const int t0 = x == 0 || it.split ? it.qa.t0 : it.qb.t0;
            mbar_arrive_expect_tx(q_full + x, q_bytes);
            tma_load_4d(sQ + x * L::kQKBytes, &tmQ, q_full + x, 0, it.g * p.G, t0, it.b);
            if (!kFp8) tma_load_4d(sQ + x * L::kQKBytes + kHalfBytes, &tmQ, q_full + x, 64, it.g * p.G, t0, it.b);
          }
          ++iq;
          progress = true;
        }
        // next K tile
        if (ik < nfetched && (kt < kKStages || mbar_test(k_empty + kt % kKStages, ((kt / kKStages) - 1) & 1))) {
          const Item& it = items[ik & 1];
          const int st = kt % kKStages;
          uint8_t* dk = sK + st * L::kQKBytes;
          const int row = round_tile(it, jk) * kBlockN;
          mbar_arrive_expect_tx(k_full + st, L::kQKBytes);
          tma_load_4d(dk, &tmK, k_full + st, 0, it.g, row, it.b);
          if (!kFp8) tma_load_4d(dk + kHalfBytes, &tmK, k_full + st, 64, it.g, row, it.b);
          ++kt;
          if (++jk == n_rounds(it)) ++ik;  // the next item's first round is set when it is fetched
          progress = true;
        }
        // next V tile
        if (iv < ik || (iv == ik && iv < nfetched && jv < jk)) {
          if (vt < kVStages || mbar_test(v_empty + vt % kVStages, ((vt / kVStages) - 1) & 1)) {
            const Item& it = items[iv & 1];
            const int st = vt % kVStages;
            uint8_t* dv = sV + st * kTileBytes;
            mbar_arrive_expect_tx(v_full + st, kTileBytes);
            // the tile holding the last key of a chunked prefill comes from its zero-padded copy: cache rows past
            // the chunk may hold anything, and P = 0 times a NaN would still poison O
            const int jt = round_tile(it, jv);
            const bool from_tail = jt == it.tail;
            const CUtensorMap* mv = from_tail ? &tmVt : &tmV;
            const int row = from_tail ? 0 : jt * kBlockN;
            tma_load_4d(dv, mv, v_full + st, 0, it.g, row, it.b);
            tma_load_4d(dv + kHalfBytes, mv, v_full + st, 64, it.g, row, it.b);
            ++vt;
            if (++jv == n_rounds(it)) {
              ++iv;
              jv = 0;
            }
            progress = true;
          }
        }
        if (done && iv == nfetched && iq == nfetched) break;
        if (progress) {
          spins = 0;
          continue;
        }
        // Bounded idle: give up (and stop the other roles) when nothing became ready for the wait limit.
        if ((++spins & 63u) == 0) {
          if (*abort_flag) break;
          const uint64_t now = global_timer_ns();
          if (spins == 64) {
            t_idle = now;
          } else if (now - t_idle > lim) {
            raise_status(NC_DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
      // Every copy this CTA started must land before the CTA exits (already true on the normal path).
      for (int t = max(0, kt - kKStages); t < kt; ++t) mbar_wait(k_full + t % kKStages, (t / kKStages) & 1, lim, nullptr);
      for (int t = max(0, vt - kVStages); t < vt; ++t) mbar_wait(v_full + t % kVStages, (t / kVStages) & 1, lim, nullptr);
      for (int i2 = max(0, iq - 1); i2 < iq; ++i2) {
        mbar_wait(q_full + 0, i2 & 1, lim, nullptr);
        mbar_wait(q_full + 1, i2 & 1, lim, nullptr);
      }
    } else if (warp == kMmaWarp || warp == kMmaWarpB) {
      // ---------------------------------------------------------------- MMA issuer of Q tile x
      // The whole warp walks the schedule and waits together (converged); lane 0 issues the MMAs and commits.
      // Every shared-memory descriptor is built once; a K step of an MMA only adds a constant to the start-address
      // field (addresses stay below 256 KB, so the 14-bit field never carries).
      const int x = warp == kMmaWarp ? 0 : 1;
      const bool leader = lane == 0;
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      // Buffers of one kind are equally spaced: the descriptor of buffer i is the one of buffer 0 plus i times the
      // buffer size >> 4.
      constexpr uint64_t kTileDesc = kTileBytes >> 4, kQKDesc = L::kQKBytes >> 4;
      const uint64_t dq = sdesc_sw128(aQ, 16, 1024) + x * kQKDesc, dk0 = sdesc_sw128(aK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(aV, kHalfBytes, 1024);
      const uint32_t tS = tbase + kColS + x * 128, tO = tbase + kColO + x * 128;
      auto issue_s = [&](int st) {  // S_X = Q_X K^T (K from stage st)
        if (leader) {
          if constexpr (kFp8) {
            // four K = 32 steps of 32 bytes along the 128-byte rows (kind::f8f6f4)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss_f8(tS, dq + kk * 2, dk0 + st * kQKDesc + kk * 2, kIdescQK8, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
              umma_ss(tS, dq + off, dk0 + st * kQKDesc + off, kIdescQK, kk > 0 ? 1u : 0u);
            }
          }
          umma_commit(s_full + x);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int st, uint32_t acc0) {  // O_X (+)= P_X V (V from stage st)
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // P of keys [16 kk, 16 kk + 16): columns 64 (kk / 4) + 8 (kk % 4)
            umma_ts(tO, tS + (kk >> 2) * 64 + (kk & 3) * 8,
                    dv0 + st * kTileDesc + static_cast<uint64_t>((kk * 2048) >> 4), kIdescPV, kk > 0 ? 1u : acc0);
          umma_commit(o_done + x);
        }
        __syncwarp();
      };
      auto commit = [&](uint64_t* bar) {
        if (leader) umma_commit(bar);
        __syncwarp();
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, lim, abort_flag));
      };
      int kv = 0;    // KV tiles of the item sequence passed so far (ring positions)
      int ns = 0;    // S / P.V products of Q tile x so far (phase of s_full / p_full / o_done)
      int nit = 0;   // items in which Q tile x was active (phase of o_free)
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!(ok = wait(sched_full + slot, (k >> 1) & 1))) break;
        const int item = sched[slot];
        __syncwarp();
        if (leader) mbar_arrive(sched_empty + slot);
        if (item < 0) break;
        const Item it = decode_item(p, item);
        const bool active = chain_active(it, x);
        const int first = first_round(it, x), nr = n_rounds(it);
        // Both issuers wait for every Q, K and V buffer of the item to land -- also the ones their own tile does not
        // use -- before releasing it: the release barriers count one commit from each issuer per fill, and an
        // issuer that ran ahead would otherwise commit twice within one fill.
        if (!(ok = wait(q_full + x, k & 1))) break;
        if (!(ok = wait(k_full + kv % kKStages, (kv / kKStages) & 1))) break;
        if (in_chain(it, x, 0)) {
          tc_fence_after_sync();
          issue_s(kv % kKStages);
        }
        commit(k_empty + kv % kKStages);
        for (int i = 0; ok && i < nr; ++i, ++kv) {
          const int vst = kv % kVStages, kst1 = (kv + 1) % kKStages;
          const bool more = i + 1 < nr;
          const bool pv = in_chain(it, x, i);
          const bool s_next = more && in_chain(it, x, i + 1);
          if (it.split && !pv) {
            // The other chain's round of a split item: this chain's next S goes in as soon as its K tile has landed;
            // the V tile of the round, which only the other chain reads, is waited for (the release barrier counts
            // one commit per issuer and fill) and released afterwards.
            if (more) {
              if (!(ok = wait(k_full + kst1, ((kv + 1) / kKStages) & 1))) break;
              tc_fence_after_sync();
              if (s_next) issue_s(kst1);
              commit(k_empty + kst1);
            }
            if (!(ok = wait(v_full + vst, (kv / kVStages) & 1))) break;
            commit(v_empty + vst);
            continue;
          }
          // Every wait of the round comes first, so that P.V and the next S go into the tensor core back to back (a
          // gap between them lets its pipeline drain).  The next K tile has normally landed a round earlier.
          if (!(ok = wait(v_full + vst, (kv / kVStages) & 1))) break;
          if (more && !(ok = wait(k_full + kst1, ((kv + 1) / kKStages) & 1))) break;
          // A tile this issuer does not read is released at once (its commit tracks only earlier products), not
          // after this round's P.V: in a split item the chain's softmax would otherwise hold the other chain's K tile.
          if (!pv) commit(v_empty + vst);
          if (more && !s_next) commit(k_empty + kst1);
          if (pv) {
            if (i == first && nit > 0 && !(ok = wait(o_free + x, (nit - 1) & 1))) break;
            if (!(ok = wait(p_full + x, ns & 1))) break;
          }
          tc_fence_after_sync();
          if (pv) {  // O_X += P_X V (the key tile of round i)
            issue_pv(vst, i > first ? 1u : 0u);
            ++ns;
          }
          if (s_next) issue_s(kst1);  // S_X = Q_X K^T (the key tile of round i + 1)
          if (pv) commit(v_empty + vst);
          if (s_next) commit(k_empty + kst1);
        }
        if (!ok) break;
        commit(q_empty);
        nit += active ? 1 : 0;
      }
      if (leader) umma_commit(mma_final + x);  // all issued MMAs complete before TMEM is released
      __syncwarp();
      mbar_wait(mma_final + x, 0, lim, nullptr);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-7)
    warpgroup_reg_inc<kRegsSoftmax>();
    const int r = threadIdx.x & 127;   // row of the Q tiles = TMEM lane
    const int h = warp >> 2;           // column half: columns [64 h, 64 h + 64) of S and O
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int tpos = r / p.G;
    constexpr uint32_t kBarAll = 1;    // named barrier of the 256 softmax threads
    int ns[2] = {0, 0};   // S tiles of Q tile X consumed so far (all items)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      ok = mbar_wait(sched_full + slot, (k >> 1) & 1, lim, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!named_bar_and(kBarAll, 2 * kSoftThreads, ok)) break;
      const int item = sched[slot];
      named_bar_sync(kBarAll, 2 * kSoftThreads);
      if (threadIdx.x == 0) mbar_arrive(sched_empty + slot);
      if (item < 0) break;
      const Item it = decode_item(p, item);
      float l[2] = {0.f, 0.f};  // this half's running softmax denominator (sum of 2^S)
      // Failure discipline: a failed wait only sets `fail`; every warp runs the same loop trip counts and reaches
      // every barrier of the 256 softmax threads, each barrier ANDs the threads' status, and the warps leave the
      // loops together, right after a barrier, when any of them failed.
      bool fail = false;
      const int nr = n_rounds(it);
      for (int i = 0; ok && i < nr; ++i) {
        const int j = round_tile(it, i);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!in_chain(it, x, i)) continue;
          const QRange q = x == 0 || it.split ? it.qa : it.qb;
          const uint32_t tS = tbase + lane_base + kColS + x * 128;
          const int t = q.a0 + tpos;  // position of this row's query
          if (!fail) fail = !mbar_wait(s_full + x, ns[x] & 1, lim, abort_flag);
          fail = !__all_sync(0xffffffffu, !fail);
          if (fail) continue;  // nothing more this round; the barrier after the rounds decides for everyone
          tc_fence_after_sync();
          uint32_t sv[2][32];
          tmem_ld32(tS + 64 * h, sv[0]);
          tmem_ld32(tS + 64 * h + 32, sv[1]);
          tmem_ld_wait(sv[0]);
          tmem_ld_wait(sv[1]);
          const int s0 = j * kBlockN + 64 * h;  // key of this thread's first column
          const bool full_tile = (j * kBlockN + kBlockN - 1 <= q.a0) &&
                                 (p.window < 0 || q.a_last - j * kBlockN <= p.window);
          if (!full_tile) {
            // visible columns form the interval [lo_c, hi_c]: key <= t, and t - key <= window
            const int hi_c = t - s0;
            const int lo_c = p.window < 0 ? -64 : hi_c - p.window;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int a = lo_c - 32 * c2, b = hi_c - 32 * c2;  // the interval within these 32 columns
              const uint32_t m_hi = b >= 31 ? ~0u : (b < 0 ? 0u : (2u << b) - 1u);
              const uint32_t m_lo = a <= 0 ? ~0u : (a > 31 ? 0u : ~((1u << a) - 1u));
              const uint32_t vis = m_hi & m_lo;
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((vis >> c) & 1u)) sv[c2][c] = __float_as_uint(-INFINITY);
            }
          }
          // P = 2^S rounded to bf16, written over this half's part of the S row (keys [64 h, 64 h + 64) -> packed
          // P columns [64 h, 64 h + 32), which only this thread reads as S).  All 32 pairs are computed before the two TMEM stores (which the compiler
          // cannot move code across) so that the exponentials of the whole half row interleave.  The row sum adds
          // the bf16 values the P.V product uses, so that O / l weighs every key exactly as the product does (a row
          // with one visible key returns that key's value exactly).
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[2][16];
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const uint32_t pp = pack_bf16x2(ex2_approx(__uint_as_float(sv[c2][2 * c])),
                                              ex2_approx(__uint_as_float(sv[c2][2 * c + 1])));
              pk[c2][c] = pp;
              rs[c & 3] = add_bf16x2_to_f32(pp, rs[c & 3]);
            }
          }
          tmem_st16(tS + 64 * h, pk[0]);
          tmem_st16(tS + 64 * h + 16, pk[1]);
          l[x] += (rs[0] + rs[1]) + (rs[2] + rs[3]);
          tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full + x);
          ++ns[x];
        }
      }
      // All 256 threads agree on the item's outcome before the epilogues use the exchange area.
      if (!named_bar_and(kBarAll, 2 * kSoftThreads, ok && !fail)) break;
      // ---- epilogues: O / l once the last P.V of each Q tile has completed; a split item has one epilogue,
      // (O_A + O_B) / (l_A + l_B)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (!chain_active(it, x) || (it.split && x == 1)) continue;
        const QRange q = x == 0 ? it.qa : it.qb;
        const bool merge = it.split && it.nb > 0;  // add chain B's partial sums
        const uint32_t tO = tbase + lane_base + kColO + x * 128;
        const uint32_t tOB = tbase + lane_base + kColO + 128;
        const bool row_in_box = r < p.G * p.P;  // rows past G * P belong to no query
        fail = !mbar_wait(o_done + x, (ns[x] - 1) & 1, lim, abort_flag);
        if (merge && !fail) fail = !mbar_wait(o_done + 1, (ns[1] - 1) & 1, lim, abort_flag);
        fail = !__all_sync(0xffffffffu, !fail);
        float* lx = xch;  // [2 halves][128] row sums
        if (!fail) lx[h * 128 + r] = merge ? l[0] + l[1] : l[x];
        // the staging tile is free once the previous tile's TMA store has read it
        if (threadIdx.x == 0) bulk_wait_read_all();
        if (!named_bar_and(kBarAll, 2 * kSoftThreads, !fail)) { ok = false; break; }
        const float l_row = lx[r] + lx[128 + r];
        const float inv_l = 1.f / l_row;
        tc_fence_after_sync();
        // Backward-pass statistics: this row's query position and head, and its part of rowsum(dout * O).
        const int t_row = q.t0 + r / p.G;
        const bool stats_row = row_in_box && t_row < p.T;
        const __nv_bfloat16* dorow =
            p.drow != nullptr && stats_row
                ? p.dout + ((static_cast<size_t>(it.b) * p.T + t_row) * p.Hq + it.g * p.G + r % p.G) * 128 + 64 * h
                : nullptr;
        float dpart = 0.f;
        // O / l in bf16 into the staging tile: this thread's 64 columns are one 128-byte row of half h, laid out
        // with the 128-byte swizzle of the output map (16-byte chunk c of row r at chunk position c ^ (r % 8)).
        uint8_t* srow = sO + h * kHalfBytes + r * 128;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t ov[32];
          tmem_ld32(tO + 64 * h + 32 * c2, ov);
          if (merge) {
            uint32_t ob[32];
            tmem_ld32(tOB + 64 * h + 32 * c2, ob);
            tmem_ld_wait(ov);
            tmem_ld_wait(ob);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) + __uint_as_float(ob[c]));
          } else {
            tmem_ld_wait(ov);
          }
          if (dorow != nullptr) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint4 d4 = __ldg(reinterpret_cast<const uint4*>(dorow + 32 * c2) + w);
              const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                dpart = fmaf(__uint_as_float(ov[8 * w + 2 * e]) * inv_l, bf16_lo(dw[e]), dpart);
                dpart = fmaf(__uint_as_float(ov[8 * w + 2 * e + 1]) * inv_l, bf16_hi(dw[e]), dpart);
              }
            }
          }
          if (row_in_box && p.store_out) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint32_t q4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                q4[e] = pack_bf16x2(__uint_as_float(ov[8 * w + 2 * e]) * inv_l,
                                    __uint_as_float(ov[8 * w + 2 * e + 1]) * inv_l);
              const int c = c2 * 4 + w;
              *reinterpret_cast<uint4*>(srow + ((c ^ (r & 7)) << 4)) = make_uint4(q4[0], q4[1], q4[2], q4[3]);
            }
          }
        }
        fence_proxy_async_smem();  // the generic-proxy writes above become visible to the TMA store
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {  // the MMA may start the next item's P.V into O_X (and O_B)
          mbar_arrive(o_free + x);
          if (merge) mbar_arrive(o_free + 1);
        }
        if (p.drow != nullptr) xch[256 + h * 128 + r] = dpart;
        named_bar_sync(kBarAll, 2 * kSoftThreads);  // staging tile written; the row-sum area is free again
        if (p.lse != nullptr && h == 0) {
          // Every row of the tile is written, the rows that hold no query with zeros.  The next tile's epilogue
          // writes the exchange area only after a barrier this thread has not reached yet.
          const size_t ri = ((static_cast<size_t>(it.b) * p.Hkv + it.g) * p.n_qtiles + q.t0 / p.P) * 128 + r;
          p.lse[ri] = stats_row ? log2f(l_row) : 0.f;
          if (p.drow != nullptr) p.drow[ri] = stats_row ? xch[256 + r] + xch[384 + r] : 0.f;
        }
        if (threadIdx.x == 0 && it.valid && p.store_out) {  // rows past T fall outside the tensor and are not written
          tma_store_4d(&tmO, sO, 0, it.g * p.G, q.t0, it.b);
          tma_store_4d(&tmO, sO + kHalfBytes, 64, it.g * p.G, q.t0, it.b);
          bulk_commit_group();
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (threadIdx.x == 0) bulk_wait_all();  // the output stores have read (and written) everything
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
