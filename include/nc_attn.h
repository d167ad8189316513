/* nc_attn -- the nanochat attention block on one B300 GPU (sm_103a), behind a plain C ABI.
 *
 * The block: half-split RoPE (base 100000) on q and k, then weightless RMSNorm of every q and k head vector
 * (QK-norm), then causal grouped-query attention with an optional sliding window, scale 1/sqrt(D).
 *   - "nanochat Admin & Developer Guide", section 3 "The GPT Model (Internals)": RoPE base theta 100000,
 *     QK-norm, RMSNorm without learnable parameters, GQA with n_kv_head <= n_head, per-layer sliding windows
 *     (window_pattern, passed to Flash Attention as (left, right) tuples).
 *   - same guide, section 6 "Attention: FA3 with SDPA Fallback": the three masking cases (full causal,
 *     single-token decode over a sliced KV window, windowed attention) and GQA.
 *   - same guide, section 7 "The Inference Engine & Tool Use", "KV cache": cache tensors laid out
 *     (B, T, H, D), positions tracked per row with an int32 cache_seqlens, new keys appended in place.
 *   - "nanochat (Fucina port)", section "Architecture": half-split RoPE with an inverse-built table,
 *     no-weight RMSNorm, grouped causal attention.
 *
 * Entry points: the prefill forward (nc_attn_fwd*; nc_attn_fwd_fp8* with e4m3 score operands), the chunked prefill
 * against a KV cache (nc_attn_prefill_chunk*),
 * the single-token decode (nc_attn_decode*), the same three with a QK-norm gain on the logits (*_ex), the backward
 * pass of the prefill (nc_attn_bwd_ws), the RoPE + norm kernel alone (nc_attn_qk_prologue), and status helpers.
 *
 * Conventions for every entry point
 *   - Tensors are bfloat16 (passed as void*, 16-bit storage), contiguous, row-major, in DEVICE memory owned by
 *     the caller, and 16-byte aligned (the backward's gradients are fp32).  cache_lens is a device int32 array.
 *   - D (head dim) must be 128; otherwise NC_ERR_UNSUPPORTED.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) and never synchronizes.  Arguments are
 *     checked on the host before anything is launched; an error return means nothing was launched.
 *   - RoPE: element i of a head vector is paired with element i + D/2; theta_i = rope_base^(-2i/D); at
 *     position t the pair is mapped to (x_i cos a + x_{i+D/2} sin a, -x_i sin a + x_{i+D/2} cos a), a = t theta_i.
 *   - RMSNorm: y / sqrt(mean(y^2) + 1e-6), no weight, computed in fp32.
 *   - window: -1 means unbounded (plain causal).  window >= 0 means key position j is visible to query position
 *     i iff 0 <= i - j <= window (window + 1 keys including the query's own position).
 *   - Arithmetic: bf16 operands, fp32 accumulation and softmax; the softmax probabilities are rounded to bf16
 *     before the P.V product; outputs are rounded to bf16 (round to nearest even).  The backward pass computes in
 *     fp32 throughout.
 *   - Device-side problems never trap.  They set a sticky device status word that nc_attn_get_device_status()
 *     returns: a bounded wait that ran out (NC_ERR_DEVICE_TIMEOUT) or a cache length outside the cache
 *     (NC_ERR_DEVICE_BAD_INPUT; that row's output is written as zeros).
 */
#ifndef NC_ATTN_H
#define NC_ATTN_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NC_OK = 0,
  NC_ERR_INVALID_ARG = 1,      /* null / misaligned pointer, bad size, bad window or rope base */
  NC_ERR_UNSUPPORTED = 2,      /* valid but not implemented here (D != 128, group size too large) */
  NC_ERR_CUDA = 3,             /* a CUDA runtime / driver call or a kernel launch failed */
  NC_ERR_DEVICE_TIMEOUT = 4,   /* a bounded wait inside a kernel ran out (see nc_attn_get_device_status) */
  NC_ERR_DEVICE_BAD_INPUT = 5, /* a kernel found an invalid cache length (see nc_attn_get_device_status) */
  NC_ERR_WORKSPACE = 6,        /* the caller's workspace is null or smaller than the *_workspace_bytes value */
  NC_ERR_SCRATCH_LIMIT = 7     /* nc_attn_decode_noalloc: the request needs more than its fixed scratch array */
} nc_status;

/* ---- prefill / training forward ------------------------------------------------------------------------------
 * q:[B,T,Hq,D]  k,v:[B,T,Hkv,D]  out:[B,T,Hq,D].  Token t of every sequence is at position t (0..T-1).
 * Query head h uses kv head h / (Hq/Hkv).  Requires Hq % Hkv == 0, Hq/Hkv <= 128, T < 2^24.
 *
 * nc_attn_fwd_ws takes a caller-owned device workspace of at least nc_attn_fwd_workspace_bytes(...) bytes,
 * 16-byte aligned, with no initial contents required; it holds the roped + normed q and k (bf16) between the
 * two kernels and must not be used by another call until this one has finished on `stream`.
 * nc_attn_fwd (the same call without a workspace argument) uses a workspace owned by the library, grown on
 * demand with cudaMallocAsync on `stream`; it is for one stream at a time per device and must not be first
 * called while `stream` is being captured into a CUDA graph.
 */
size_t nc_attn_fwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D);

nc_status nc_attn_fwd_ws(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                         int D, int window, float rope_base, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

nc_status nc_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                      int D, int window, float rope_base, cudaStream_t stream);

/* Same as nc_attn_fwd_ws, and records CUDA events on `stream` around the two kernels it launches: `k1_begin`
 * before the RoPE + QK-norm prologue, `k2_begin` between the prologue and the attention kernel, `k2_end` after the
 * attention kernel.  Any event may be NULL.  Used to time each kernel with CUDA events on its own stream. */
nc_status nc_attn_fwd_ws_events(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq,
                                int Hkv, int D, int window, float rope_base, void* workspace,
                                size_t workspace_bytes, cudaEvent_t k1_begin, cudaEvent_t k2_begin,
                                cudaEvent_t k2_end, cudaStream_t stream);

/* ---- the fused RoPE + QK-norm prologue alone -----------------------------------------------------------------
 * qn = norm(rope(q)), kn = norm(rope(k)) at positions 0..T-1, bf16, same layouts as q and k.  This is the first
 * kernel of nc_attn_fwd, exported so that the normalised vectors can be checked on their own.
 */
nc_status nc_attn_qk_prologue(const void* q, const void* k, void* qn, void* kn, int B, int T, int Hq, int Hkv,
                              int D, float rope_base, cudaStream_t stream);

/* ---- prefill forward with e4m3 (fp8) score operands -----------------------------------------------------------
 * ("nanochat Admin & Developer Guide", section 6: the fast attention kernel takes bf16 or fp8 operands; section 5
 * "Precision", FP8 training: operands of a product quantised to float8_e4m3fn with one scale per tensor, fp32
 * accumulation, the scales removed from the result.)  Same inputs, output, positions, window and grouping as
 * nc_attn_fwd_ex (qk_gain in (0, 4] multiplies every logit).  The difference: the roped + normed qn and kn are
 * rounded to e4m3 as qn * s_q and kn * s_k, with s_q = 4 qk_gain log2(e) / sqrt(D) and s_k = 1/4 (unit-RMS vectors
 * bound every element by sqrt(D), so these fixed per-tensor scales keep both inside e4m3's +-448), and the score
 * contraction runs on the tensor cores' 8-bit path; its result divided by s_q s_k and times qk_gain / sqrt(D) is the
 * logit.  The probabilities and v stay bf16 (P.V in bf16 with fp32 accumulation), the output is bf16.
 *
 * workspace: caller-owned device memory of at least nc_attn_fwd_fp8_workspace_bytes(...) bytes, 16-byte aligned,
 * no initial contents required (the e4m3 qn and kn and a counter); not to be shared by calls that overlap on the GPU.
 * nc_attn_fwd_fp8_events additionally records `k1_begin`, `k2_begin`, `k2_end` around the two kernels it launches
 * (any may be NULL), as nc_attn_fwd_ws_events does.
 * nc_attn_qk_prologue_fp8 runs the first kernel alone: qn8 [B,T,Hq,D] and kn8 [B,T,Hkv,D] receive the e4m3 codes
 * (one byte per element, round to nearest even) of qn * s_q and kn * s_k.
 */
size_t nc_attn_fwd_fp8_workspace_bytes(int B, int T, int Hq, int Hkv, int D);

nc_status nc_attn_fwd_fp8(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                          int D, int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

nc_status nc_attn_fwd_fp8_events(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq,
                                 int Hkv, int D, int window, float rope_base, float qk_gain, void* workspace,
                                 size_t workspace_bytes, cudaEvent_t k1_begin, cudaEvent_t k2_begin,
                                 cudaEvent_t k2_end, cudaStream_t stream);

nc_status nc_attn_qk_prologue_fp8(const void* q, const void* k, void* qn8, void* kn8, int B, int T, int Hq, int Hkv,
                                  int D, float rope_base, float qk_gain, cudaStream_t stream);

/* ---- Chunked prefill against a KV cache ------------------------------------------------------------------------
 * ("nanochat Admin & Developer Guide", section 6: the SDPA fallback's third case, chunked / sliding-window
 * inference, where the queries of a chunk attend to the cache plus the chunk; section 7 "KV cache": FA3 layout
 * (B, T, H, D), per-row cache_seqlens, in-place append.)  Tq new tokens per sequence b, at positions
 * p_b + t (t < Tq) with p_b = cache_lens[b].
 *   q:[B,Tq,Hq,D]                 raw queries of the chunk (roped at p_b + t and normed inside the call)
 *   k_new,v_new:[B,Tq,Hkv,D]      raw keys and values of the chunk; norm(rope(k_new[b,t], p_b + t)) and v_new[b,t]
 *                                 are written to cache row p_b + t (in place)
 *   kcache,vcache:[B,Tcap,Hkv,D]  rows 0..p_b-1 are used as given (already roped and normed); rows at or past
 *                                 p_b + Tq are never read into the result (they may hold anything)
 *   cache_lens: device int32[B]   read only; the caller advances it by Tq after the call
 *   out:[B,Tq,Hq,D]
 * Query t of sequence b sees cache rows j <= p_b + t with p_b + t - j <= window (window -1 = all); the result
 * equals rows p_b .. p_b+Tq-1 of nc_attn_fwd over the whole sequence.  A p_b outside [0, Tcap - Tq] gives zero
 * output rows for that sequence, leaves its cache untouched and sets NC_ERR_DEVICE_BAD_INPUT in the device status
 * word.  Requires Tcap >= Tq and Hq % Hkv == 0, D == 128.
 *
 * nc_attn_prefill_chunk_ws takes a caller-owned, 16-byte aligned device workspace of at least
 * nc_attn_prefill_chunk_workspace_bytes(...) bytes (normed queries, a zero-padded copy of each sequence's last V
 * tile, a counter); it needs no initialisation.  nc_attn_prefill_chunk uses a workspace owned by the library
 * (same growth and stream rules as nc_attn_fwd).  Two calls that share a workspace must not overlap on the GPU.
 * The pages have no such entry point under this name; it is the chunked case of their attention call.
 */
size_t nc_attn_prefill_chunk_workspace_bytes(int B, int Tq, int Hq, int Hkv, int D);

nc_status nc_attn_prefill_chunk_ws(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                                   const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D,
                                   int Tcap, int window, float rope_base, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

nc_status nc_attn_prefill_chunk(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                                const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D, int Tcap,
                                int window, float rope_base, cudaStream_t stream);

/* ---- QK-norm gain ----------------------------------------------------------------------------------------------
 * ("nanochat Admin & Developer Guide", section 3, QK-norm bullet: after the norm, q and k carry a combined factor
 * of 1.2 that sharpens the attention.)  The _ex entry points take that factor as `qk_gain`: every logit is
 * qk_gain * qn.kn / sqrt(D).  qk_gain = 1 is the plain forms above; 1.2 is nanochat's.  Accepted range (0, 4]: the
 * prefill kernel's softmax takes exponentials without a running maximum, which the bound |logit| <= 16.5 qk_gain
 * (in base 2, for unit-RMS q and k) keeps within fp32 and bf16 up to a gain of 4; NC_ERR_INVALID_ARG otherwise.
 * All other arguments, layouts, workspaces and errors as for the corresponding _ws entry point.
 */
nc_status nc_attn_fwd_ex(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                         int D, int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

nc_status nc_attn_prefill_chunk_ex(const void* q, const void* k_new, const void* v_new, void* kcache, void* vcache,
                                   const int* cache_lens, void* out, int B, int Tq, int Hq, int Hkv, int D,
                                   int Tcap, int window, float rope_base, float qk_gain, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

nc_status nc_attn_decode_ex(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                            const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap,
                            int window, float rope_base, float qk_gain, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* ---- Gated value embedding -------------------------------------------------------------------------------------
 * (The catalog pages list value embeddings with a sigmoid gate, in the ResFormer manner, among nanochat's
 * architectural additions.  The pages give no formula; the reading taken: v' = v + sigmoid(g) * ve, one gate logit g
 * per token and kv head.)  As nc_attn_fwd_ex with the attention run on v' instead of v:
 *   ve:[B,T,Hkv,D]   value embedding, bf16, 16-byte aligned
 *   ve_gate:[B,T,Hkv] gate logits, bf16 (2-byte aligned)
 * v' is formed in fp32 and rounded to bf16 inside the call (in the workspace, which must hold
 * nc_attn_fwd_ve_workspace_bytes(...) bytes).  Both ve and ve_gate are required (NC_ERR_INVALID_ARG otherwise).
 */
size_t nc_attn_fwd_ve_workspace_bytes(int B, int T, int Hq, int Hkv, int D);

nc_status nc_attn_fwd_ve(const void* q, const void* k, const void* v, const void* ve, const void* ve_gate, void* out,
                         int B, int T, int Hq, int Hkv, int D, int window, float rope_base, float qk_gain,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The same value embedding for the new tokens on the cache paths: the values appended to the cache (and attended
 * to) are v_new' = v_new + sigmoid(ve_gate) * ve_new, formed in fp32 and rounded to bf16 once, as in nc_attn_fwd_ve.
 *   nc_attn_prefill_chunk_ve: as nc_attn_prefill_chunk_ex, with ve_new:[B,Tq,Hkv,D] and ve_gate:[B,Tq,Hkv]
 *     (the chunk's tokens); workspace as for nc_attn_prefill_chunk_ws.
 *   nc_attn_decode_ve: as nc_attn_decode_ex with a new key and value (k_new, v_new required), with ve_new:[B,Hkv,D]
 *     and ve_gate:[B,Hkv]; workspace as for nc_attn_decode_ws.
 * ve tensors bf16 and 16-byte aligned, gates bf16 (2-byte aligned); both required (NC_ERR_INVALID_ARG otherwise).
 */
nc_status nc_attn_prefill_chunk_ve(const void* q, const void* k_new, const void* v_new, const void* ve_new,
                                   const void* ve_gate, void* kcache, void* vcache, const int* cache_lens, void* out,
                                   int B, int Tq, int Hq, int Hkv, int D, int Tcap, int window, float rope_base,
                                   float qk_gain, void* workspace, size_t workspace_bytes, cudaStream_t stream);

nc_status nc_attn_decode_ve(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                            const void* k_new, const void* v_new, const void* ve_new, const void* ve_gate, int B,
                            int Hq, int Hkv, int D, int Tcap, int window, float rope_base, float qk_gain,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- Backward pass of the prefill forward -----------------------------------------------------------------------
 * ("nanochat Admin & Developer Guide", section 3: the model trains through this block.)  Gradients of
 * sum(dout * out), out = nc_attn_fwd_ex(q, k, v, window, rope_base, qk_gain), with respect to the raw q, k, v:
 *   q:[B,T,Hq,D] k,v:[B,T,Hkv,D] dout:[B,T,Hq,D]  bf16, 16-byte aligned device memory
 *   dq:[B,T,Hq,D] dk,dv:[B,T,Hkv,D]               fp32, written (not accumulated)
 * through the RoPE, the weightless RMSNorm and the banded GQA softmax, in fp32 on the CUDA cores.  The workspace
 * (16-byte aligned, nc_attn_bwd_workspace_bytes(...) bytes, no initialisation) holds the normed vectors and row
 * statistics.  Errors as nc_attn_fwd_ws (qk_gain in (0, 4]).  The pages have no such entry point; autograd
 * computes the same gradients there.
 */
size_t nc_attn_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D);

nc_status nc_attn_bwd_ws(const void* q, const void* k, const void* v, const void* dout, float* dq, float* dk,
                         float* dv, int B, int T, int Hq, int Hkv, int D, int window, float rope_base, float qk_gain,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- training: forward that keeps its row statistics, backward that reuses them ------------------------------
 * A training step normally keeps the forward's output and the log-sum-exp of every score row for the backward, so
 * that the backward does not run the forward again ("nanochat Admin & Developer Guide", section 3: the model trains
 * through this block).
 *
 * nc_attn_fwd_lse_ws: nc_attn_fwd_ex plus `lse`, a device float buffer of nc_attn_lse_bytes(B, T, Hq, Hkv) bytes,
 * 16-byte aligned, into which it writes the base-2 log-sum-exp log2(sum_j 2^s_j) of every query row's logits
 * s_j = qk_gain log2(e) qn . kn_j / sqrt(D), in the layout the backward reads: float[B][Hkv][ceil(T / P)][128]
 * with P = floor(128 / G), G = Hq / Hkv; entry r of block m of (b, kv head g) belongs to query position m P + r / G
 * of query head g G + r % G, and entries that hold no query are 0.  Not with a value embedding or e4m3 operands.
 *
 * nc_attn_bwd_saved_ws: the gradients of nc_attn_bwd_ws from the same inputs plus that forward's `out` [B,T,Hq,D]
 * (bf16) and `lse`; it skips the forward's recomputation and forms rowsum(dout * out) from the kept output.  Same
 * workspace (nc_attn_bwd_workspace_bytes) and the same window, rope_base and qk_gain as the forward's.  Returns 0
 * bytes / NC_ERR_INVALID_ARG for the shapes and pointers nc_attn_bwd_ws rejects, and for a null or misaligned
 * out or lse.
 */
size_t nc_attn_lse_bytes(int B, int T, int Hq, int Hkv);

nc_status nc_attn_fwd_lse_ws(const void* q, const void* k, const void* v, void* out, float* lse, int B, int T, int Hq,
                             int Hkv, int D, int window, float rope_base, float qk_gain, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

nc_status nc_attn_bwd_saved_ws(const void* q, const void* k, const void* v, const void* out, const void* dout,
                               const float* lse, float* dq, float* dk, float* dv, int B, int T, int Hq, int Hkv,
                               int D, int window, float rope_base, float qk_gain, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/* ---- KV-cache single-token decode ------------------------------------------------------------------------------
 * One new query token per sequence b, at position p_b = cache_lens[b].
 *   q:[B,Hq,D]            raw query of the new token (roped at position p_b, then normed, inside the call)
 *   kcache,vcache:[B,Tcap,Hkv,D]  rows 0..p_b-1 are used as given (already roped and normed)
 *   cache_lens: device int32[B]   read only; the caller advances it after the call
 *   k_new,v_new:[B,Hkv,D] or both NULL.  When given, norm(rope(k_new, p_b)) and v_new are written to cache
 *                         row p_b (in place) and attended to; then p_b must be <= Tcap-1.
 *   out:[B,Hq,D]
 * Visible keys are j in [max(0, p_b - window), L_b) with L_b = p_b (+1 with a new key); window -1 = all.
 * An empty visible set (p_b = 0 and no new key) gives a zero output row and no error.  A p_b outside the cache
 * gives a zero output row and NC_ERR_DEVICE_BAD_INPUT in the device status word.  Requires Hq/Hkv <= 16.
 *
 * nc_attn_decode_ws takes a caller-owned device workspace of at least nc_attn_decode_workspace_bytes(...) bytes,
 * 16-byte aligned.  It holds B*Hkv arrival counters at its start, then the split partial results.  The counters
 * must be zero when a call starts: zero the workspace before its first use (e.g. a zero-filled allocation) and
 * again before any call whose B*Hkv differs from that of the previous call on the same workspace (that call's
 * partials may lie where the new counters go).  A call leaves its own counters zero, so calls with the same B and
 * Hkv can reuse the workspace as is.  Two calls that share a workspace must not overlap on the GPU.
 * nc_attn_decode uses a workspace owned by the library (same growth and stream rules as nc_attn_fwd).
 */
size_t nc_attn_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int Tcap, int window);

nc_status nc_attn_decode_ws(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                            const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap,
                            int window, float rope_base, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

nc_status nc_attn_decode(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                         const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap, int window,
                         float rope_base, cudaStream_t stream);

/* ---- decode that allocates nothing ----------------------------------------------------------------------------
 * Not a step of the attention block itself (the pages have no counterpart): an extra way to call the decode step
 * for callers that may not allocate device memory at all.  Examples: code that runs inside another framework's
 * plugin or enqueue hook, where the host framework owns the whole memory budget and forbids allocation on the hot
 * path; serving loops that reserve every byte at start-up, because cudaMalloc and cudaFree can synchronize the
 * device and stall the other streams.  Such a caller can pass neither a workspace nor let nc_attn_decode grow one.
 *
 * Same arguments and results as nc_attn_decode.  The split partials and arrival counters live in one array of
 * NC_ATTN_DECODE_NOALLOC_MAX_BYTES bytes that the library declares in device memory at file scope; every GPU that
 * loads the library holds that array until the process exits.  A request fits when
 * nc_attn_decode_workspace_bytes(B, Hq, Hkv, D, Tcap, window) <= NC_ATTN_DECODE_NOALLOC_MAX_BYTES (the 64-sequence,
 * Hq 12, Hkv 4 decode needs about 0.8 MiB; the size grows with B * Hkv and the group size); a larger one returns
 * NC_ERR_SCRATCH_LIMIT and launches nothing.  The call never runs cudaMalloc, cudaFree or any other allocating routine.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with that device
 *     current) and keeps it; make that first call before any stream capture begins.
 *   - Each call clears the counter region of the array on `stream` (cudaMemsetAsync) before its kernel, so the
 *     previous call's leftovers do not matter.
 *   - All calls on a device share the one array: two calls that overlap on the GPU (different streams without
 *     ordering between them) race on it and give wrong results.  Order them on one stream, or use nc_attn_decode_ws
 *     with a workspace per stream.
 */
#define NC_ATTN_DECODE_NOALLOC_MAX_BYTES (8u * 1024u * 1024u)

nc_status nc_attn_decode_noalloc(const void* q, void* kcache, void* vcache, const int* cache_lens, void* out,
                                 const void* k_new, const void* v_new, int B, int Hq, int Hkv, int D, int Tcap,
                                 int window, float rope_base, cudaStream_t stream);

/* ---- status ------------------------------------------------------------------------------------------------------ */
/* Static description of a status code (never NULL). */
const char* nc_attn_status_string(nc_status s);

/* Synchronizes `stream`, then returns the sticky device status of the current device (NC_OK when clean,
 * NC_ERR_DEVICE_TIMEOUT or NC_ERR_DEVICE_BAD_INPUT otherwise; timeout wins; NC_ERR_UNSUPPORTED if a kernel found
 * its dynamic shared memory less aligned than it can use, in which case it wrote nothing) and, when `clear` is
 * non-zero, resets it.  Returns NC_ERR_CUDA when the synchronization or the read fails. */
nc_status nc_attn_get_device_status(cudaStream_t stream, int clear);

/* Self-test of the bounded waits: launches one tiny kernel whose threads wait on a barrier that nothing ever
 * completes, giving up after `limit_us` microseconds (1..2000000).  The kernel then returns normally and the
 * device status reads NC_ERR_DEVICE_TIMEOUT.  Used by the tests to show that a stuck pipeline ends its kernel
 * and leaves the context usable. */
nc_status nc_attn_selftest_wait_timeout(int limit_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NC_ATTN_H */
