"""FP8 (e4m3) variant of the prefill forward, in fp64 -- test infrastructure only (called by ``tests/`` and never by
the product path).

The pages: the fast attention kernel the project uses supports bf16 and fp8 operands ("nanochat Admin & Developer
Guide", section 6 "Attention: FA3 with SDPA Fallback"), and the project's own fp8 training recipe quantises the
operands of a matrix product to float8_e4m3fn in the forward pass with one scale per tensor, multiplies them with
fp32 accumulation and removes the scales from the result (same guide, section 5 "Precision", "FP8 training").  They
do not say which operands of attention are quantised or how the scales are chosen.  Readings taken here:

* The score contraction S = qn kn^T runs on e4m3 operands: qn and kn (after RoPE and the weightless RMSNorm) are
  quantised with per-tensor scales s_q and s_k, and the product is divided by s_q s_k.
* The scales are fixed by the QK-norm rather than measured: every element of a unit-RMS vector of D = 128 entries
  lies within +-sqrt(128), so no data-dependent maximum is needed to stay inside e4m3's range (+-448).  s_q =
  4 g log2(e) / sqrt(D) and s_k = 1/4, with g the QK-norm gain on the logits: the dequantisation factor 1 / (s_q s_k)
  times the logit scale g / sqrt(D) is then ln 2, so the quantised product is directly a base-2 logit, and the
  factors 4 and 1/4 put typical elements of both operands (|x| ~ 1 times g log2(e) / sqrt(D), resp. ~ 1) well
  inside e4m3's normal range (smallest normal 2^-6).
* The probabilities and the values stay as in the bf16 path (the P V contraction is not quantised): softmax without
  a running maximum gives probabilities spread over 2^(+-16.5 g), far more octaves than e4m3 holds, and the tensor
  core's kinds take both operands of a product in one type.
* Rounding to e4m3 is round-to-nearest, ties to even; nothing here goes out of range (a value beyond 448 raises).

Everything else (positions, window, grouping, softmax, value product) is ``oracle.ref.attn_fwd``.
"""

import math

import numpy as np

from oracle import ref

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9


def e4m3_decode(code):
    """Value of an 8-bit float8_e4m3fn code: sign bit 7, exponent bits 6-3 (bias 7), mantissa bits 2-0.  Exponent
    field 0 encodes subnormals m * 2^-9; the all-ones pattern S.1111.111 is NaN (the format has no infinities)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_round(x):
    """Rounds fp64 values to the nearest float8_e4m3fn value (ties to even), returned as fp64.  Raises on NaN or
    |x| > 448 (the scales above keep every operand in range)."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e4m3_round: non-finite input")
    a = np.abs(x)
    if np.any(a > E4M3_MAX):
        raise ValueError(f"e4m3_round: |x| = {a.max()} beyond the e4m3 range 448")
    # quantum of the binade of |x|: 2^(e - 3) with e = floor(log2 |x|), and 2^-9 throughout the subnormal range
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    r = np.rint(a / quantum) * quantum          # np.rint rounds halves to even: the even multiple of the quantum
    return np.copysign(r, x)


def fp8_scales(qk_gain=1.0, D=128):
    """Per-tensor scales (s_q, s_k) of the quantised qn and kn."""
    s_q = 4.0 * qk_gain * math.log2(math.e) / math.sqrt(D)
    return s_q, 0.25


def attn_fwd_fp8(q, k, v, window, rope_base=ref.ROPE_BASE, eps=ref.RMS_EPS, chunk=128, qk_gain=1.0):
    """Prefill forward with the score contraction on e4m3 operands (readings above).

    q: [B, T, Hq, D], k and v: [B, T, Hkv, D].  Returns out [B, T, Hq, D] fp64.  Blocked over query chunks like
    ``ref.attn_fwd``: only the keys of a chunk's band are scored, then the exact mask is applied.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    pos = np.broadcast_to(np.arange(T), (B, T))
    s_q, s_k = fp8_scales(qk_gain, D)
    q8 = e4m3_round(ref.qk_prologue(q, pos, rope_base, eps) * s_q)
    k8 = e4m3_round(ref.qk_prologue(k, pos, rope_base, eps) * s_k)
    logit = qk_gain / np.sqrt(D)
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i0 in range(0, T, chunk):
                i1 = min(T, i0 + chunk)
                j0 = 0 if window < 0 else max(0, i0 - window)
                s = (q8[b, i0:i1, h] @ k8[b, j0:i1, g].T) / (s_q * s_k) * logit
                mask = ref.visible(np.arange(i0, i1)[:, None], np.arange(j0, i1)[None, :], window)
                s = np.where(mask, s, -np.inf)
                m = s.max(axis=-1, keepdims=True)
                p = np.exp(s - m)
                out[b, i0:i1, h] = (p / p.sum(axis=-1, keepdims=True)) @ v[b, j0:i1, g]
    return out
