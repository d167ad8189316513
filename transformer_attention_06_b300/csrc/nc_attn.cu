// C-ABI entry points of the attention library: host-side validation, TMA descriptor encoding, launch
// configuration and workspace layout.  One translation unit holds every kernel, so that the device status word is
// a single symbol without relocatable device code.
//
// Nothing here falls back to the CPU or to another implementation: an unsupported request returns an error code.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "nc_attn.h"

#include "common.cuh"
#include "prologue.cuh"
#include "attn_fwd.cuh"
#include "attn_decode.cuh"
#include "attn_bwd.cuh"

namespace {

using nc::RopeTable;

constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s per bounded wait

// ---------------------------------------------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// A 4-D view [d3][d2][d1][d0] (d0 innermost, contiguous) of bf16 elements (or of bytes when `bytes` is set: e4m3
// codes), 128-byte swizzle, zero fill out of bounds.
bool make_map_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                 uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3, bool bytes = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t es = bytes ? 1 : 2;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * es, d0 * d1 * es, d0 * d1 * d2 * es};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  return fn(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------------------------------------------
RopeTable rope_table(float base) {
  // theta_i = base^(-2i/D) for D = 128, in fp64, split into an fp32 value and its fp32 residual.
  RopeTable t;
  for (int i = 0; i < 64; ++i) {
    const double th = std::pow(static_cast<double>(base), -2.0 * i / 128.0);
    t.hi[i] = static_cast<float>(th);
    t.lo[i] = static_cast<float>(th - static_cast<double>(t.hi[i]));
  }
  return t;
}

float scale_log2_for_d128() { return static_cast<float>(1.4426950408889634 / std::sqrt(128.0)); }

// Per-tensor scales of the e4m3 qn and kn: s_q = 4 g log2(e) / sqrt(128) and s_k = 1/4.  Every element of a unit-RMS
// vector lies within +-sqrt(128), so both stay far inside e4m3's +-448 for gains up to 4; their product makes the
// e4m3 product a base-2 logit; the factors 4 and 1/4 keep typical elements of both operands in e4m3's normal range.
constexpr float kFp8KScale = 0.25f;
float fp8_q_scale(float qk_gain) { return 4.0f * scale_log2_for_d128() * qk_gain; }

// Largest accepted gain on the logits.  The prefill kernel takes exponentials without a running maximum: with unit-RMS
// qn, kn its base-2 logits are bounded by 16.5 times the gain, so a gain of at most 4 keeps 2^S within [2^-66, 2^66]
// and any row sum below 2^97 (fp32 and bf16 hold both).
constexpr float kMaxQkGain = 4.0f;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool rope_base_ok(float base) { return std::isfinite(base) && base > 0.f; }

// Checks shared by the forward and the prologue.  Returns NC_OK or the error to report.
nc_status check_fwd_shapes(int B, int T, int Hq, int Hkv, int D) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1) return NC_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return NC_ERR_INVALID_ARG;
  if (D != 128) return NC_ERR_UNSUPPORTED;
  if (T >= (1 << 24)) return NC_ERR_UNSUPPORTED;  // positions must be exact in fp32
  // Token indices are 32-bit in the prologue kernels, including the block rounding of the token count.
  if (static_cast<long long>(B) * T > 0x7fffffffLL - nc::kPrologueTokensPerBlock) return NC_ERR_UNSUPPORTED;
  const long double elems = static_cast<long double>(B) * T * Hq * D;
  if (elems > 9.0e15L) return NC_ERR_INVALID_ARG;
  return NC_OK;
}

template <typename F>
void set_smem_attr_once(F* kernel, int bytes, int slot) {
  static bool done[16][32] = {};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 16) dev = 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev][slot]) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    done[dev][slot] = true;
  }
}

nc_status launch_status() { return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA; }

int sm_count();

// Slices per token for the prologue kernels: as many as keep the grid within one wave of lane groups (64 resident
// groups per SM: two blocks of 256 threads at 128 registers), so short inputs spread over every SM (a chunk of 2048
// tokens: 4 slices) while a partial second wave never appears (8192 tokens: 1 slice), at most kMaxSlices and at most
// one per q/k head.
int prologue_slices(long long tokens, int H) {
  const long long wave = static_cast<long long>(std::max(sm_count(), 1)) * 64;
  const long long s = wave / std::max(tokens, 1LL);
  return static_cast<int>(std::max(1LL, std::min<long long>({s, nc::kMaxSlices, H})));
}

// fp8: qn, kn written as e4m3 codes times q_scale, k_scale (else bf16, kn unscaled).
nc_status launch_prologue(const void* q, const void* k, void* qn, void* kn, int B, int T, int Hq, int Hkv,
                          const RopeTable& tab, float q_scale, unsigned* zero_word, cudaStream_t stream,
                          const void* v = nullptr, const void* ve = nullptr, const void* ve_gate = nullptr,
                          void* vmix = nullptr, bool fp8 = false, float k_scale = 1.0f) {
  const int BT = B * T;
  const int ns = prologue_slices(BT, Hq + Hkv);
  const long long groups = static_cast<long long>(BT) * ns;
  if (groups > 0x7fffffffLL - nc::kPrologueTokensPerBlock) return NC_ERR_UNSUPPORTED;
  const int blocks = static_cast<int>((groups + nc::kPrologueTokensPerBlock - 1) / nc::kPrologueTokensPerBlock);
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  if (fp8) {
    nc::qk_prologue_kernel<uint8_t><<<blocks, nc::kPrologueThreads, 0, stream>>>(
        qb, kb, static_cast<uint8_t*>(qn), static_cast<uint8_t*>(kn), BT, T, Hq, Hkv, tab, q_scale, k_scale,
        zero_word, nullptr, nullptr, nullptr, nullptr, ns);
  } else {
    nc::qk_prologue_kernel<__nv_bfloat16><<<blocks, nc::kPrologueThreads, 0, stream>>>(
        qb, kb, static_cast<__nv_bfloat16*>(qn), static_cast<__nv_bfloat16*>(kn), BT, T, Hq, Hkv, tab, q_scale,
        k_scale, zero_word, static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(ve),
        static_cast<const __nv_bfloat16*>(ve_gate), static_cast<__nv_bfloat16*>(vmix), ns);
  }
  return launch_status();
}

// Resident CTAs per device for the persistent kernels: one per SM.
int sm_count() {
  static int cached[16] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// ---- library-held workspaces for the entry points without a workspace argument -------------------------------
struct HeldBuffer {
  void* ptr = nullptr;
  size_t bytes = 0;
  long long tag = -1;  // decode: B * Hkv of the last call (its counter region); -1 = freshly zeroed
};

std::mutex g_ws_mu;
HeldBuffer g_fwd_ws[16];
HeldBuffer g_dec_ws[16];
HeldBuffer g_chunk_ws[16];

// Returns a buffer of at least `bytes` for the current device, grown in stream order; `zero` clears a new buffer.
// `tag` / `clear_bytes`: when a reused buffer was last used with another tag, its first `clear_bytes` are cleared
// (decode: a call with another B * Hkv may have left split partials where this call's arrival counters live).
void* held_workspace(HeldBuffer* table, size_t bytes, bool zero, long long tag, size_t clear_bytes,
                     cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return nullptr;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  HeldBuffer& hb = table[dev];
  if (hb.bytes < bytes) {
    if (hb.ptr != nullptr) cudaFreeAsync(hb.ptr, stream);
    hb.ptr = nullptr;
    hb.bytes = 0;
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) return nullptr;
    if (zero && cudaMemsetAsync(p, 0, bytes, stream) != cudaSuccess) return nullptr;
    hb.ptr = p;
    hb.bytes = bytes;
    hb.tag = tag;
  } else if (hb.tag != tag) {
    if (clear_bytes > 0 && cudaMemsetAsync(hb.ptr, 0, clear_bytes, stream) != cudaSuccess) return nullptr;
    hb.tag = tag;
  }
  return hb.ptr;
}

// ---- decode workspace layout ------------------------------------------------------------------------------------
// [B * Hkv arrival counters][(m, l) of 2 partials per CTA and head][128-float partial outputs of the same].
struct DecodeLayout {
  size_t off_cnt, off_ml, off_o, total;
};

DecodeLayout decode_layout(int B, int Hq, int Hkv) {
  DecodeLayout L;
  const size_t G = static_cast<size_t>(Hq / Hkv);
  const size_t slots = static_cast<size_t>(nc::dec::kMaxParts) * 2 * G;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  L.off_cnt = 0;
  L.off_ml = up(static_cast<size_t>(B) * Hkv * sizeof(unsigned));
  L.off_o = L.off_ml + up(slots * 2 * sizeof(float));
  L.total = L.off_o + up(slots * 128 * sizeof(float));
  return L;
}

// The decode kernel is launched with programmatic dependent launch: its CTAs may start (barriers, TMEM, operand
// padding) while the previous kernel in the stream drains, and wait for it (griddepcontrol.wait) before reading any
// input.  A launch failure is left for the caller's cudaGetLastError check.
template <int G>
void launch_decode_g(int grid, const CUtensorMap& mk, const CUtensorMap& mv, const RopeTable& tab,
                     const nc::dec::Params& prm, cudaStream_t stream) {
  set_smem_attr_once(nc::dec::attn_decode_kernel<G>, nc::dec::kSmemBytes, G);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(nc::dec::kThreads);
  cfg.dynamicSmemBytes = nc::dec::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, nc::dec::attn_decode_kernel<G>, mk, mv, tab, prm);
}

// Resident CTAs of the decode kernel on the current device: one per SM, at most kMaxParts.
int decode_grid() {
  const int n = sm_count();
  return n < nc::dec::kMaxParts ? n : nc::dec::kMaxParts;
}

nc_status check_decode_args(const void* q, const void* kcache, const void* vcache, const int* cache_lens,
                            const void* out, const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D,
                            int Tcap, int window, float rope_base) {
  if (q == nullptr || kcache == nullptr || vcache == nullptr || cache_lens == nullptr || out == nullptr)
    return NC_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return NC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out)) return NC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return NC_ERR_INVALID_ARG;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return NC_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || Tcap < 1) return NC_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return NC_ERR_INVALID_ARG;
  if (window < -1) return NC_ERR_INVALID_ARG;
  if (!rope_base_ok(rope_base)) return NC_ERR_INVALID_ARG;
  if (D != 128) return NC_ERR_UNSUPPORTED;
  if (Hq / Hkv > nc::dec::kMaxG) return NC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv * 4 > (1ll << 40)) return NC_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535 || Tcap >= (1 << 24)) return NC_ERR_UNSUPPORTED;
  return NC_OK;
}

// Launches the attention kernel after a prologue on the same stream, with programmatic dependent launch: the CTAs
// may start (and set up barriers and TMEM) while the prologue drains; they wait on the prologue grid
// (griddepcontrol.wait) before touching anything it writes.
nc_status launch_attention(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mvt,
                           const CUtensorMap& mo, const nc::fwd::Params& prm, int n_sm, cudaStream_t stream,
                           bool fp8 = false) {
  auto* kernel = fp8 ? nc::fwd::attn_fwd_kernel<true> : nc::fwd::attn_fwd_kernel<false>;
  const int smem = fp8 ? nc::fwd::kSmemBytesFp8 : nc::fwd::kSmemBytes;
  set_smem_attr_once(kernel, smem, fp8 ? 17 : 0);
  const int grid = std::min(n_sm, prm.n_items);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(nc::fwd::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mvt, mo, prm) != cudaSuccess) {
    (void)cudaGetLastError();  // clear it: the failure is reported here
    return NC_ERR_CUDA;
  }
  return launch_status();
}

// Work split of the attention kernel over T query rows: P = 128 / G positions per Q tile; two tiles per item
// (they share every K/V tile), or one tile per item when pairs would not give every SM of the GPU an item.
// n_pairs is the number of items per (b, kv head).
bool fwd_split(int B, int T, int Hq, int Hkv, int n_sm, int& G, int& P, int& n_pairs, int& tiles_per_item) {
  G = Hq / Hkv;
  if (G > 128) return false;
  P = 128 / G;
  const int n_qtiles = (T + P - 1) / P;
  tiles_per_item = static_cast<long long>(B) * Hkv * ((n_qtiles + 1) / 2) < n_sm ? 1 : 2;
  n_pairs = tiles_per_item == 2 ? (n_qtiles + 1) / 2 : n_qtiles;
  return static_cast<long long>(B) * Hkv * n_pairs <= 0x7fffffffLL;
}

template <bool kDQ>
nc_status launch_bwd(const CUtensorMap& mq, const CUtensorMap& mdo, const CUtensorMap& mk, const CUtensorMap& mv,
                            const nc::bwd::Params& prm, int n_sm, cudaStream_t stream) {
  set_smem_attr_once(nc::bwd::bwd_kernel<kDQ>, nc::bwd::kSmemBytes, kDQ ? 19 : 18);
  const int grid = std::min(n_sm, prm.n_items);
  nc::bwd::bwd_kernel<kDQ><<<grid, nc::bwd::kThreads, nc::bwd::kSmemBytes, stream>>>(mq, mdo, mk, mv, prm);
  return launch_status();
}

}  // namespace

// =================================================================================================================
extern "C" {

size_t nc_attn_fwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D) {
  if (check_fwd_shapes(B, T, Hq, Hkv, D) != NC_OK && !(D > 0 && D != 128)) return 0;
  return 2ull * static_cast<size_t>(B) * T * (Hq + Hkv) * D + 256;
}

nc_status nc_attn_qk_prologue(const void* q, const void* k, void* qn, void* kn, int B, int T, int Hq, int Hkv,
                              int D, float rope_base, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || qn == nullptr || kn == nullptr) return NC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(qn) || !aligned16(kn)) return NC_ERR_INVALID_ARG;
  if (!rope_base_ok(rope_base)) return NC_ERR_INVALID_ARG;
  const nc_status st = check_fwd_shapes(B, T, Hq, Hkv, D);
  if (st != NC_OK) return st;
  return launch_prologue(q, k, qn, kn, B, T, Hq, Hkv, rope_table(rope_base), 1.0f, nullptr, stream);
}

nc_status nc_attn_fwd_ws(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                         int D, int window, float rope_base, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  return nc_attn_fwd_ws_events(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, workspace, workspace_bytes,
                               nullptr, nullptr, nullptr, stream);
}

static nc_status fwd_impl(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                          int D, int window, float rope_base, float qk_gain, void* workspace,
                          size_t workspace_bytes, cudaEvent_t k1_begin, cudaEvent_t k2_begin, cudaEvent_t k2_end,
                          cudaStream_t stream, const void* ve = nullptr, const void* ve_gate = nullptr,
                          bool fp8 = false, float* lse_out = nullptr) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return NC_ERR_INVALID_ARG;
  if (lse_out != nullptr && (fp8 || ve != nullptr || (reinterpret_cast<uintptr_t>(lse_out) & 15u) != 0))
    return NC_ERR_INVALID_ARG;
  if (!(qk_gain > 0.f && qk_gain <= kMaxQkGain)) return NC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return NC_ERR_INVALID_ARG;
  if (window < -1 || !rope_base_ok(rope_base)) return NC_ERR_INVALID_ARG;
  nc_status st = check_fwd_shapes(B, T, Hq, Hkv, D);
  if (st != NC_OK) return st;
  int G = 0, P = 0, n_pairs = 0, tpi = 0;
  if (!fwd_split(B, T, Hq, Hkv, 0, G, P, n_pairs, tpi)) return NC_ERR_UNSUPPORTED;
  if ((ve == nullptr) != (ve_gate == nullptr)) return NC_ERR_INVALID_ARG;
  if (ve != nullptr && (!aligned16(ve) || (reinterpret_cast<uintptr_t>(ve_gate) & 1u) != 0)) return NC_ERR_INVALID_ARG;
  const size_t need = fp8 ? nc_attn_fwd_fp8_workspace_bytes(B, T, Hq, Hkv, D)
                          : ve != nullptr ? nc_attn_fwd_ve_workspace_bytes(B, T, Hq, Hkv, D)
                                          : nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return NC_ERR_WORKSPACE;

  // qn, kn (bf16, or e4m3 codes), then the work-item counter
  const size_t es = fp8 ? 1 : 2;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qn = ws;
  void* kn = ws + es * static_cast<size_t>(B) * T * Hq * D;
  unsigned* item_ctr = reinterpret_cast<unsigned*>(ws + es * static_cast<size_t>(B) * T * (Hq + Hkv) * D);
  // with a value embedding, the mixed values follow the counter (the fwd workspace size, a multiple of 256)
  void* vmix = ve != nullptr ? ws + nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D) : nullptr;
  const void* vsrc = ve != nullptr ? vmix : v;
  const int n_sm = sm_count();
  if (n_sm < 1) return NC_ERR_CUDA;
  if (!fwd_split(B, T, Hq, Hkv, n_sm, G, P, n_pairs, tpi)) return NC_ERR_UNSUPPORTED;

  // Q and K boxes: one 64-element half of a row in bf16 (two loads per tile), the whole 128-byte row in e4m3
  const uint32_t qk_box = fp8 ? 128 : 64;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map_4d(&mq, qn, 128, Hq, T, B, qk_box, G, P, 1, fp8) ||
      !make_map_4d(&mk, kn, 128, Hkv, T, B, qk_box, 1, 128, 1, fp8) ||
      !make_map_4d(&mv, vsrc, 128, Hkv, T, B, 64, 1, 128, 1) || !make_map_4d(&mo, out, 128, Hq, T, B, 64, G, P, 1))
    return NC_ERR_CUDA;

  if (k1_begin != nullptr && cudaEventRecord(k1_begin, stream) != cudaSuccess) return NC_ERR_CUDA;
  // qn leaves the prologue multiplied by log2(e) / sqrt(D): the attention kernel's scores are then base-2 logits.
  if (fp8)
    st = launch_prologue(q, k, qn, kn, B, T, Hq, Hkv, rope_table(rope_base), fp8_q_scale(qk_gain), item_ctr, stream,
                         nullptr, nullptr, nullptr, nullptr, true, kFp8KScale);
  else
    st = launch_prologue(q, k, qn, kn, B, T, Hq, Hkv, rope_table(rope_base), scale_log2_for_d128() * qk_gain,
                         item_ctr, stream, v, ve, ve_gate, vmix);
  if (st != NC_OK) return st;
  if (k2_begin != nullptr && cudaEventRecord(k2_begin, stream) != cudaSuccess) return NC_ERR_CUDA;

  nc::fwd::Params prm;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.B = B;
  prm.T = T;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = G;
  prm.P = P;
  prm.n_pairs = n_pairs;
  prm.n_items = B * Hkv * n_pairs;
  prm.tiles_per_item = tpi;
  prm.item_ctr = item_ctr;
  prm.pos0 = nullptr;
  prm.Tk = T;
  prm.window = window;
  prm.wait_limit_ns = kWaitLimitNs;
  prm.lse = lse_out;  // with it: every query row's base-2 log-sum-exp, for a backward that reuses it
  prm.drow = nullptr;
  prm.dout = nullptr;
  prm.n_qtiles = (T + P - 1) / P;
  prm.store_out = 1;
  st = launch_attention(mq, mk, mv, mv, mo, prm, n_sm, stream, fp8);
  if (st == NC_OK && k2_end != nullptr && cudaEventRecord(k2_end, stream) != cudaSuccess) return NC_ERR_CUDA;
  return st;
}

size_t nc_attn_fwd_fp8_workspace_bytes(int B, int T, int Hq, int Hkv, int D) {
  if (check_fwd_shapes(B, T, Hq, Hkv, D) != NC_OK) return 0;
  return static_cast<size_t>(B) * T * (Hq + Hkv) * D + 256;
}

nc_status nc_attn_fwd_fp8_events(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq,
                                 int Hkv, int D, int window, float rope_base, float qk_gain, void* workspace,
                                 size_t workspace_bytes, cudaEvent_t k1_begin, cudaEvent_t k2_begin,
                                 cudaEvent_t k2_end, cudaStream_t stream) {
  return fwd_impl(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace, workspace_bytes, k1_begin,
                  k2_begin, k2_end, stream, nullptr, nullptr, true);
}

nc_status nc_attn_fwd_fp8(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                          int D, int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  return fwd_impl(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace, workspace_bytes, nullptr,
                  nullptr, nullptr, stream, nullptr, nullptr, true);
}

nc_status nc_attn_qk_prologue_fp8(const void* q, const void* k, void* qn8, void* kn8, int B, int T, int Hq, int Hkv,
                                  int D, float rope_base, float qk_gain, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || qn8 == nullptr || kn8 == nullptr) return NC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(qn8) || !aligned16(kn8)) return NC_ERR_INVALID_ARG;
  if (!rope_base_ok(rope_base) || !(qk_gain > 0.f && qk_gain <= kMaxQkGain)) return NC_ERR_INVALID_ARG;
  const nc_status st = check_fwd_shapes(B, T, Hq, Hkv, D);
  if (st != NC_OK) return st;
  return launch_prologue(q, k, qn8, kn8, B, T, Hq, Hkv, rope_table(rope_base), fp8_q_scale(qk_gain), nullptr, stream,
                         nullptr, nullptr, nullptr, nullptr, true, kFp8KScale);
}

nc_status nc_attn_fwd_ws_events(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq,
                                int Hkv, int D, int window, float rope_base, void* workspace,
                                size_t workspace_bytes, cudaEvent_t k1_begin, cudaEvent_t k2_begin,
                                cudaEvent_t k2_end, cudaStream_t stream) {
  return fwd_impl(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, 1.0f, workspace, workspace_bytes, k1_begin,
                  k2_begin, k2_end, stream);
}

size_t nc_attn_fwd_ve_workspace_bytes(int B, int T, int Hq, int Hkv, int D) {
  const size_t base = nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D);
  return base == 0 ? 0 : base + 2ull * static_cast<size_t>(B) * T * Hkv * D;
}

nc_status nc_attn_fwd_ve(const void* q, const void* k, const void* v, const void* ve, const void* ve_gate, void* out,
                         int B, int T, int Hq, int Hkv, int D, int window, float rope_base, float qk_gain,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (ve == nullptr || ve_gate == nullptr) return NC_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace, workspace_bytes, nullptr,
                  nullptr, nullptr, stream, ve, ve_gate);
}

nc_status nc_attn_fwd_ex(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                         int D, int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  return fwd_impl(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace, workspace_bytes, nullptr,
                  nullptr, nullptr, stream);
}

nc_status nc_attn_fwd_lse_ws(const void* q, const void* k, const void* v, void* out, float* lse, int B, int T, int Hq,
                             int Hkv, int D, int window, float rope_base, float qk_gain, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  if (lse == nullptr) return NC_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace, workspace_bytes, nullptr,
                  nullptr, nullptr, stream, nullptr, nullptr, false, lse);
}

nc_status nc_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv, int D,
                      int window, float rope_base, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return NC_ERR_INVALID_ARG;
  const nc_status st = check_fwd_shapes(B, T, Hq, Hkv, D);
  if (st != NC_OK) return st;
  const size_t need = nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D);
  void* ws = held_workspace(g_fwd_ws, need, false, -1, 0, stream);
  if (ws == nullptr) return NC_ERR_CUDA;
  return nc_attn_fwd_ws(q, k, v, out, B, T, Hq, Hkv, D, window, rope_base, ws, need, stream);
}

size_t nc_attn_prefill_chunk_workspace_bytes(int B, int Tq, int Hq, int Hkv, int D) {
  if (check_fwd_shapes(B, Tq, Hq, Hkv, D) != NC_OK) return 0;
  // qn [B, Tq, Hq, D], the V tail copies [B, 128, Hkv, D] (bf16), then the work-item counter
  return 2ull * static_cast<size_t>(B) * Tq * Hq * D + 2ull * static_cast<size_t>(B) * 128 * Hkv * D + 256;
}

static nc_status chunk_impl(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                            const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D, int Tcap,
                            int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream, const void* ve_new = nullptr, const void* ve_gate = nullptr) {
  if (!(qk_gain > 0.f && qk_gain <= kMaxQkGain)) return NC_ERR_INVALID_ARG;
  if (q == nullptr || k_new == nullptr || v_new == nullptr || kcache == nullptr || vcache == nullptr ||
      cache_lens == nullptr || out == nullptr)
    return NC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(kcache) || !aligned16(vcache) ||
      !aligned16(out))
    return NC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return NC_ERR_INVALID_ARG;
  if (window < -1 || !rope_base_ok(rope_base)) return NC_ERR_INVALID_ARG;
  if ((ve_new == nullptr) != (ve_gate == nullptr)) return NC_ERR_INVALID_ARG;
  if (ve_new != nullptr && (!aligned16(ve_new) || (reinterpret_cast<uintptr_t>(ve_gate) & 1u) != 0))
    return NC_ERR_INVALID_ARG;
  nc_status st = check_fwd_shapes(B, Tq, Hq, Hkv, D);
  if (st != NC_OK) return st;
  if (Tcap < Tq) return NC_ERR_INVALID_ARG;
  st = check_fwd_shapes(B, Tcap, Hkv, Hkv, D);  // cache positions exact in fp32, sizes in range
  if (st != NC_OK) return st;
  int G = 0, P = 0, n_pairs = 0, tpi = 0;
  if (!fwd_split(B, Tq, Hq, Hkv, 0, G, P, n_pairs, tpi)) return NC_ERR_UNSUPPORTED;
  const size_t need = nc_attn_prefill_chunk_workspace_bytes(B, Tq, Hq, Hkv, D);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return NC_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qn = ws;
  void* vtail = ws + 2ull * static_cast<size_t>(B) * Tq * Hq * D;
  unsigned* item_ctr = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(vtail) + 2ull * static_cast<size_t>(B) * 128 * Hkv * D);
  const int n_sm = sm_count();
  if (n_sm < 1) return NC_ERR_CUDA;
  if (!fwd_split(B, Tq, Hq, Hkv, n_sm, G, P, n_pairs, tpi)) return NC_ERR_UNSUPPORTED;

  CUtensorMap mq, mk, mv, mvt, mo;
  if (!make_map_4d(&mq, qn, 128, Hq, Tq, B, 64, G, P, 1) ||
      !make_map_4d(&mk, kcache, 128, Hkv, Tcap, B, 64, 1, 128, 1) ||
      !make_map_4d(&mv, vcache, 128, Hkv, Tcap, B, 64, 1, 128, 1) ||
      !make_map_4d(&mvt, vtail, 128, Hkv, 128, B, 64, 1, 128, 1) ||
      !make_map_4d(&mo, out, 128, Hq, Tq, B, 64, G, P, 1))
    return NC_ERR_CUDA;

  const int ns = prologue_slices(static_cast<long long>(B) * Tq, Hq + Hkv);
  const long long groups = static_cast<long long>(B) * Tq * ns;
  if (groups > 0x7fffffffLL - nc::kPrologueTokensPerBlock) return NC_ERR_UNSUPPORTED;
  const int tok_blocks = static_cast<int>((groups + nc::kPrologueTokensPerBlock - 1) / nc::kPrologueTokensPerBlock);
  const int tail_blocks = (B * 128 + nc::kPrologueTokensPerBlock - 1) / nc::kPrologueTokensPerBlock;
  nc::chunk_prologue_kernel<<<tok_blocks + tail_blocks, nc::kPrologueThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
      static_cast<const __nv_bfloat16*>(v_new), static_cast<__nv_bfloat16*>(qn), static_cast<__nv_bfloat16*>(kcache),
      static_cast<__nv_bfloat16*>(vcache), static_cast<__nv_bfloat16*>(vtail), static_cast<__nv_bfloat16*>(out),
      cache_lens, B, Tq, Hq, Hkv, Tcap, tok_blocks, rope_table(rope_base), scale_log2_for_d128() * qk_gain,
      item_ctr, static_cast<const __nv_bfloat16*>(ve_new), static_cast<const __nv_bfloat16*>(ve_gate), ns);
  st = launch_status();
  if (st != NC_OK) return st;

  nc::fwd::Params prm;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.B = B;
  prm.T = Tq;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = G;
  prm.P = P;
  prm.n_pairs = n_pairs;
  prm.n_items = B * Hkv * n_pairs;
  prm.tiles_per_item = tpi;
  prm.item_ctr = item_ctr;
  prm.pos0 = cache_lens;
  prm.Tk = Tcap;
  prm.window = window;
  prm.wait_limit_ns = kWaitLimitNs;
  prm.lse = nullptr;
  prm.drow = nullptr;
  prm.dout = nullptr;
  prm.n_qtiles = (Tq + P - 1) / P;
  prm.store_out = 1;
  return launch_attention(mq, mk, mv, mvt, mo, prm, n_sm, stream);
}

nc_status nc_attn_prefill_chunk_ws(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                                   const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D,
                                   int Tcap, int window, float rope_base, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  return chunk_impl(q, k_new, v_new, kcache, vcache, cache_lens, out, B, Tq, Hq, Hkv, D, Tcap, window, rope_base,
                    1.0f, workspace, workspace_bytes, stream);
}

nc_status nc_attn_prefill_chunk_ex(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                                   const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D,
                                   int Tcap, int window, float rope_base, float qk_gain, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  return chunk_impl(q, k_new, v_new, kcache, vcache, cache_lens, out, B, Tq, Hq, Hkv, D, Tcap, window, rope_base,
                    qk_gain, workspace, workspace_bytes, stream);
}

nc_status nc_attn_prefill_chunk_ve(const void* q, const void* k_new, const void* v_new, const void* ve_new,
                                   const void* ve_gate, void* kcache, void* vcache, const int* cache_lens, void* out,
                                   int B, int Tq, int Hq, int Hkv, int D, int Tcap, int window, float rope_base,
                                   float qk_gain, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (ve_new == nullptr || ve_gate == nullptr) return NC_ERR_INVALID_ARG;
  return chunk_impl(q, k_new, v_new, kcache, vcache, cache_lens, out, B, Tq, Hq, Hkv, D, Tcap, window, rope_base,
                    qk_gain, workspace, workspace_bytes, stream, ve_new, ve_gate);
}

nc_status nc_attn_prefill_chunk(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                                const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D, int Tcap,
                                int window, float rope_base, cudaStream_t stream) {
  const nc_status st = check_fwd_shapes(B, Tq, Hq, Hkv, D);
  if (st != NC_OK) return st;
  const size_t need = nc_attn_prefill_chunk_workspace_bytes(B, Tq, Hq, Hkv, D);
  void* ws = held_workspace(g_chunk_ws, need, false, -1, 0, stream);
  if (ws == nullptr) return NC_ERR_CUDA;
  return nc_attn_prefill_chunk_ws(q, k_new, v_new, kcache, vcache, cache_lens, out, B, Tq, Hq, Hkv, D, Tcap, window,
                                  rope_base, ws, need, stream);
}

// Backward workspace: qn' and kn (bf16, as the forward writes them), three work-item counters (forward statistics,
// dK/dV, dQ), then the per-row base-2 log-sum-exp and rowsum(dO * O) in the padded Q-tile layout
// [B, Hkv, n_qtiles, 128]; each region 256-byte aligned.
struct BwdLayout {
  size_t qn, kn, ctr, lse, drow, total;
  int G, P, n_qtiles;
};

static BwdLayout bwd_layout(int B, int T, int Hq, int Hkv) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  BwdLayout L;
  L.G = Hq / Hkv;
  L.P = 128 / L.G;
  L.n_qtiles = (T + L.P - 1) / L.P;
  const size_t rows = static_cast<size_t>(B) * Hkv * L.n_qtiles * 128;
  L.qn = 0;
  L.kn = up(L.qn + static_cast<size_t>(B) * T * Hq * 128 * 2);
  L.ctr = up(L.kn + static_cast<size_t>(B) * T * Hkv * 128 * 2);
  L.lse = up(L.ctr + 16);
  L.drow = up(L.lse + rows * 4);
  L.total = up(L.drow + rows * 4);
  return L;
}

size_t nc_attn_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D) {
  if (check_fwd_shapes(B, T, Hq, Hkv, D) != NC_OK || Hq / Hkv > 128) return 0;
  return bwd_layout(B, T, Hq, Hkv).total;
}

size_t nc_attn_lse_bytes(int B, int T, int Hq, int Hkv) {
  if (check_fwd_shapes(B, T, Hq, Hkv, 128) != NC_OK || Hq / Hkv > 128) return 0;
  const BwdLayout L = bwd_layout(B, T, Hq, Hkv);
  return L.drow - L.lse;  // the row-statistics block of the backward workspace: rows * 4 bytes, rounded up
}

// The backward of nc_attn_bwd_ws; with `out` and `lse_in` (the forward's output and its nc_attn_fwd_lse_ws
// statistics) the forward is not run again: rowsum(dout * out) comes from the kept output.
static nc_status bwd_impl(const void* q, const void* k, const void* v, const void* dout, float* dq, float* dk,
                          float* dv, int B, int T, int Hq, int Hkv, int D, int window, float rope_base, float qk_gain,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream, const void* out = nullptr,
                          const float* lse_in = nullptr) {
  if (q == nullptr || k == nullptr || v == nullptr || dout == nullptr || dq == nullptr || dk == nullptr ||
      dv == nullptr)
    return NC_ERR_INVALID_ARG;
  if ((out == nullptr) != (lse_in == nullptr)) return NC_ERR_INVALID_ARG;
  if (out != nullptr && (!aligned16(out) || (reinterpret_cast<uintptr_t>(lse_in) & 15u) != 0))
    return NC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return NC_ERR_INVALID_ARG;
  if (!(qk_gain > 0.f && qk_gain <= kMaxQkGain)) return NC_ERR_INVALID_ARG;
  if (window < -1 || !rope_base_ok(rope_base)) return NC_ERR_INVALID_ARG;
  nc_status st = check_fwd_shapes(B, T, Hq, Hkv, D);
  if (st != NC_OK) return st;
  if (Hq / Hkv > 128) return NC_ERR_UNSUPPORTED;
  const BwdLayout L = bwd_layout(B, T, Hq, Hkv);
  if (static_cast<long long>(B) * Hkv * L.n_qtiles > 0x7fffffffLL) return NC_ERR_UNSUPPORTED;
  // the rowsum kernel's one-dimensional grid: 32 packed rows per block
  if (lse_in != nullptr && static_cast<long long>(B) * Hkv * L.n_qtiles * 4 > 0x7fffffffLL) return NC_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < L.total || !aligned16(workspace)) return NC_ERR_WORKSPACE;
  const int n_sm = sm_count();
  if (n_sm < 1) return NC_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qn = ws + L.qn;
  void* kn = ws + L.kn;
  unsigned* ctr = reinterpret_cast<unsigned*>(ws + L.ctr);
  float* lse = reinterpret_cast<float*>(ws + L.lse);
  float* drow = reinterpret_cast<float*>(ws + L.drow);
  const int G = L.G, P = L.P;
  const int w_eff = (window < 0 || window >= T - 1) ? -1 : window;  // windows >= T - 1 are plain causal

  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_4d(&mq, qn, 128, Hq, T, B, 64, G, P, 1) || !make_map_4d(&mk, kn, 128, Hkv, T, B, 64, 1, 128, 1) ||
      !make_map_4d(&mv, v, 128, Hkv, T, B, 64, 1, 128, 1) || !make_map_4d(&mdo, dout, 128, Hq, T, B, 64, G, P, 1))
    return NC_ERR_CUDA;
  if (cudaMemsetAsync(ctr + 1, 0, 2 * sizeof(unsigned), stream) != cudaSuccess) return NC_ERR_CUDA;

  // 1. qn' = qn log2(e) qk_gain / sqrt(D) and kn, as in the forward (zeroes the forward's work counter)
  const RopeTable tab = rope_table(rope_base);
  st = launch_prologue(q, k, qn, kn, B, T, Hq, Hkv, tab, scale_log2_for_d128() * qk_gain, ctr, stream);
  if (st != NC_OK) return st;
  // 2. the forward's row statistics: kept from the forward (rowsum(dout * out) from its output), or recomputed by
  // the attention kernel in its statistics mode (no output written: the output map points at qn', which has its
  // shape)
  if (lse_in != nullptr) {
    lse = const_cast<float*>(lse_in);
    const long long n_rows = static_cast<long long>(B) * Hkv * L.n_qtiles * 128;
    const long long blocks = (n_rows + nc::bwd::kDrowThreads / 8 - 1) / (nc::bwd::kDrowThreads / 8);
    nc::bwd::drow_kernel<<<static_cast<unsigned>(blocks), nc::bwd::kDrowThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), drow, T, Hq, Hkv, G, P,
        L.n_qtiles, n_rows);
    st = launch_status();
    if (st != NC_OK) return st;
  }
  int n_pairs = 0, tpi = 0, G2 = 0, P2 = 0;
  if (!fwd_split(B, T, Hq, Hkv, n_sm, G2, P2, n_pairs, tpi)) return NC_ERR_UNSUPPORTED;
  nc::fwd::Params fp;
  fp.out = static_cast<__nv_bfloat16*>(qn);
  fp.item_ctr = ctr;
  fp.pos0 = nullptr;
  fp.B = B;
  fp.T = T;
  fp.Hq = Hq;
  fp.Hkv = Hkv;
  fp.G = G;
  fp.P = P;
  fp.n_pairs = n_pairs;
  fp.n_items = B * Hkv * n_pairs;
  fp.window = window;
  fp.tiles_per_item = tpi;
  fp.Tk = T;
  fp.wait_limit_ns = kWaitLimitNs;
  fp.lse = lse;
  fp.drow = drow;
  fp.dout = static_cast<const __nv_bfloat16*>(dout);
  fp.n_qtiles = L.n_qtiles;
  fp.store_out = 0;
  if (lse_in == nullptr) {
    st = launch_attention(mq, mk, mv, mv, mq, fp, n_sm, stream);
    if (st != NC_OK) return st;
  }
  // 3. dK (w.r.t. kn) and dV;  4. dQ (w.r.t. qn)
  nc::bwd::Params bp;
  bp.lse = lse;
  bp.drow = drow;
  bp.B = B;
  bp.T = T;
  bp.Hq = Hq;
  bp.Hkv = Hkv;
  bp.G = G;
  bp.P = P;
  bp.n_qtiles = L.n_qtiles;
  bp.n_ktiles = (T + 127) / 128;
  bp.window = w_eff;
  bp.wait_limit_ns = kWaitLimitNs;
  bp.dst_a = dk;
  bp.dst_b = dv;
  bp.item_ctr = ctr + 1;
  bp.n_items = B * Hkv * bp.n_ktiles;
  bp.scale_a = static_cast<float>(std::log(2.0));
  st = launch_bwd<false>(mq, mdo, mk, mv, bp, n_sm, stream);
  if (st != NC_OK) return st;
  bp.dst_a = dq;
  bp.dst_b = nullptr;
  bp.item_ctr = ctr + 2;
  bp.n_items = B * Hkv * L.n_qtiles;
  bp.scale_a = static_cast<float>(static_cast<double>(qk_gain) / std::sqrt(128.0));
  st = launch_bwd<true>(mq, mdo, mk, mv, bp, n_sm, stream);
  if (st != NC_OK) return st;
  // 5. the RMSNorm and RoPE backward of every q and k row, in place
  const int BT = B * T;  // at most 2^31 - 33 (check_fwd_shapes)
  const int blocks = (BT + nc::bwd::kPostTokensPerBlock - 1) / nc::bwd::kPostTokensPerBlock;
  nc::bwd::bwd_norm_rope_kernel<<<blocks, nc::bwd::kPostThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), dq, dk, BT, T, Hq, Hkv, tab);
  return launch_status();
}

nc_status nc_attn_bwd_ws(const void* q, const void* k, const void* v, const void* dout, float* dq, float* dk,
                         float* dv, int B, int T, int Hq, int Hkv, int D, int window, float rope_base, float qk_gain,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(q, k, v, dout, dq, dk, dv, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace,
                  workspace_bytes, stream);
}

nc_status nc_attn_bwd_saved_ws(const void* q, const void* k, const void* v, const void* out, const void* dout,
                               const float* lse, float* dq, float* dk, float* dv, int B, int T, int Hq, int Hkv,
                               int D, int window, float rope_base, float qk_gain, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  if (out == nullptr || lse == nullptr) return NC_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, dout, dq, dk, dv, B, T, Hq, Hkv, D, window, rope_base, qk_gain, workspace,
                  workspace_bytes, stream, out, lse);
}

size_t nc_attn_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int Tcap, int window) {
  if (B < 1 || Hq < 1 || Hkv < 1 || D != 128 || Tcap < 1 || Hq % Hkv != 0 || window < -1) return 0;
  if (Hq / Hkv > nc::dec::kMaxG) return 0;
  return decode_layout(B, Hq, Hkv).total;
}

static nc_status decode_impl(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                             const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap,
                             int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream, const void* ve_new = nullptr, const void* ve_gate = nullptr) {
  if (!(qk_gain > 0.f && qk_gain <= kMaxQkGain)) return NC_ERR_INVALID_ARG;
  const nc_status st =
      check_decode_args(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window, rope_base);
  if (st != NC_OK) return st;
  if ((ve_new == nullptr) != (ve_gate == nullptr)) return NC_ERR_INVALID_ARG;
  if (ve_new != nullptr &&
      (k_new == nullptr || !aligned16(ve_new) || (reinterpret_cast<uintptr_t>(ve_gate) & 1u) != 0))
    return NC_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(B, Hq, Hkv);
  if (workspace == nullptr || workspace_bytes < L.total || !aligned16(workspace)) return NC_ERR_WORKSPACE;
  const int grid = decode_grid();
  if (grid < 1) return NC_ERR_CUDA;

  CUtensorMap mk, mv;
  if (!make_map_4d(&mk, kcache, 128, Hkv, Tcap, B, 64, 1, nc::dec::kRows, 1) ||
      !make_map_4d(&mv, vcache, 128, Hkv, Tcap, B, 64, 1, nc::dec::kRows, 1))
    return NC_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  nc::dec::Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.kcache = static_cast<__nv_bfloat16*>(kcache);
  prm.vcache = static_cast<__nv_bfloat16*>(vcache);
  prm.cache_lens = cache_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.k_new = static_cast<const __nv_bfloat16*>(k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(v_new);
  prm.ve_new = static_cast<const __nv_bfloat16*>(ve_new);
  prm.ve_gate = static_cast<const __nv_bfloat16*>(ve_gate);
  prm.ws_cnt = reinterpret_cast<unsigned*>(ws + L.off_cnt);
  prm.ws_ml = reinterpret_cast<float*>(ws + L.off_ml);
  prm.ws_o = reinterpret_cast<float*>(ws + L.off_o);
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = Hq / Hkv;
  prm.Tcap = Tcap;
  prm.window = window;
  prm.scale_log2 = scale_log2_for_d128() * qk_gain;
  prm.wait_limit_ns = kWaitLimitNs;
  const RopeTable tab = rope_table(rope_base);
  switch (prm.G) {
    case 1: launch_decode_g<1>(grid, mk, mv, tab, prm, stream); break;
    case 2: launch_decode_g<2>(grid, mk, mv, tab, prm, stream); break;
    case 3: launch_decode_g<3>(grid, mk, mv, tab, prm, stream); break;
    case 4: launch_decode_g<4>(grid, mk, mv, tab, prm, stream); break;
    case 5: launch_decode_g<5>(grid, mk, mv, tab, prm, stream); break;
    case 6: launch_decode_g<6>(grid, mk, mv, tab, prm, stream); break;
    case 7: launch_decode_g<7>(grid, mk, mv, tab, prm, stream); break;
    case 8: launch_decode_g<8>(grid, mk, mv, tab, prm, stream); break;
    case 9: launch_decode_g<9>(grid, mk, mv, tab, prm, stream); break;
    case 10: launch_decode_g<10>(grid, mk, mv, tab, prm, stream); break;
    case 11: launch_decode_g<11>(grid, mk, mv, tab, prm, stream); break;
    case 12: launch_decode_g<12>(grid, mk, mv, tab, prm, stream); break;
    case 13: launch_decode_g<13>(grid, mk, mv, tab, prm, stream); break;
    case 14: launch_decode_g<14>(grid, mk, mv, tab, prm, stream); break;
    case 15: launch_decode_g<15>(grid, mk, mv, tab, prm, stream); break;
    case 16: launch_decode_g<16>(grid, mk, mv, tab, prm, stream); break;
    default: return NC_ERR_UNSUPPORTED;
  }
  return launch_status();
}

nc_status nc_attn_decode_ws(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                            const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap,
                            int window, float rope_base, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  return decode_impl(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window, rope_base, 1.0f,
                     workspace, workspace_bytes, stream);
}

nc_status nc_attn_decode_ex(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                            const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap,
                            int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  return decode_impl(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window, rope_base,
                     qk_gain, workspace, workspace_bytes, stream);
}

nc_status nc_attn_decode_ve(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                            const void* k_new, const void* v_new, const void* ve_new, const void* ve_gate, int B,
                            int Hq, int Hkv, int D, int Tcap, int window, float rope_base, float qk_gain,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (ve_new == nullptr || ve_gate == nullptr || k_new == nullptr) return NC_ERR_INVALID_ARG;
  return decode_impl(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window, rope_base,
                     qk_gain, workspace, workspace_bytes, stream, ve_new, ve_gate);
}

nc_status nc_attn_decode(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                         const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap, int window,
                         float rope_base, cudaStream_t stream) {
  const nc_status st =
      check_decode_args(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window, rope_base);
  if (st != NC_OK) return st;
  const DecodeLayout L = decode_layout(B, Hq, Hkv);
  const size_t need = L.total;
  void* ws = held_workspace(g_dec_ws, need, true, static_cast<long long>(B) * Hkv, L.off_ml, stream);
  if (ws == nullptr) return NC_ERR_CUDA;
  return nc_attn_decode_ws(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window,
                           rope_base, ws, need, stream);
}

const char* nc_attn_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "NC_OK: success";
    case NC_ERR_INVALID_ARG: return "NC_ERR_INVALID_ARG: null or misaligned pointer, bad size, window or rope base";
    case NC_ERR_UNSUPPORTED: return "NC_ERR_UNSUPPORTED: valid request outside what this library implements";
    case NC_ERR_CUDA: return "NC_ERR_CUDA: a CUDA call or kernel launch failed";
    case NC_ERR_DEVICE_TIMEOUT: return "NC_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel ran out";
    case NC_ERR_DEVICE_BAD_INPUT: return "NC_ERR_DEVICE_BAD_INPUT: a kernel found a cache length outside the cache";
    case NC_ERR_WORKSPACE: return "NC_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case NC_ERR_SCRATCH_LIMIT:
      return "NC_ERR_SCRATCH_LIMIT: the request needs more than the fixed no-allocation scratch array "
             "(NC_ATTN_DECODE_NOALLOC_MAX_BYTES)";
  }
  return "unknown nc_status";
}

nc_status nc_attn_get_device_status(cudaStream_t stream, int clear) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return NC_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, nc::g_status, sizeof(v)) != cudaSuccess) return NC_ERR_CUDA;
  if (clear && v != 0) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(nc::g_status, &z, sizeof(z)) != cudaSuccess) return NC_ERR_CUDA;
  }
  if (v & nc::NC_DEV_TIMEOUT) return NC_ERR_DEVICE_TIMEOUT;
  if (v & nc::NC_DEV_BAD_CACHE_LEN) return NC_ERR_DEVICE_BAD_INPUT;
  if (v & nc::NC_DEV_SMEM_BASE) return NC_ERR_UNSUPPORTED;
  return NC_OK;
}

}  // extern "C"

namespace nc {
// One warp waits on a barrier that nothing completes; the bounded wait gives up and raises NC_DEV_TIMEOUT.
__global__ void selftest_wait_timeout_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, limit_ns, &abort_flag);
}
}  // namespace nc

extern "C" nc_status nc_attn_selftest_wait_timeout(int limit_us, cudaStream_t stream) {
  if (limit_us < 1 || limit_us > 2000000) return NC_ERR_INVALID_ARG;
  nc::selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(limit_us) * 1000ull);
  return launch_status();
}

// =================================================================================================================
// Decode without any allocation: the split partials and arrival counters go to a fixed array in device memory,
// declared here at file scope, instead of a workspace.  For callers that may not allocate (a host framework's plugin
// hook that owns the memory budget; serving loops that forbid cudaMalloc / cudaFree after start-up because those
// calls can synchronize the device).  Every GPU that loads the library holds the array until the process exits.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[NC_ATTN_DECODE_NOALLOC_MAX_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[16] = {};

// Device address of the scratch array on the current device.  In host code `g_decode_noalloc_scratch` names a
// host-side stand-in, not device memory, so the address is looked up once per device (with that device current)
// and kept.  Returns nullptr when the lookup fails.
void* noalloc_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_noalloc_addr[dev] = ptr;
  }
  return g_noalloc_addr[dev];
}

}  // namespace

extern "C" nc_status nc_attn_decode_noalloc(const void* q, void* kcache, void* vcache, const int* cache_lens,
                                            void* out, const void* k_new, const void* v_new, int B, int Hq,
                                            int Hkv, int D, int Tcap, int window, float rope_base,
                                            cudaStream_t stream) {
  const nc_status st =
      check_decode_args(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window, rope_base);
  if (st != NC_OK) return st;
  const DecodeLayout L = decode_layout(B, Hq, Hkv);
  if (L.total > static_cast<size_t>(NC_ATTN_DECODE_NOALLOC_MAX_BYTES)) return NC_ERR_SCRATCH_LIMIT;
  void* scratch = noalloc_scratch_address();
  if (scratch == nullptr) return NC_ERR_CUDA;
  // The arrival counters at the start of the array must read zero.  A previous call with another B * Hkv may have
  // left split partials there, so clear the whole counter region in stream order before the kernel.
  if (cudaMemsetAsync(scratch, 0, L.off_ml, stream) != cudaSuccess) return NC_ERR_CUDA;
  return nc_attn_decode_ws(q, kcache, vcache, cache_lens, out, k_new, v_new, B, Hq, Hkv, D, Tcap, window,
                           rope_base, scratch, NC_ATTN_DECODE_NOALLOC_MAX_BYTES, stream);
}
