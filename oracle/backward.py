"""Backward pass of the attention block in fp64 -- test infrastructure only (called by ``tests/``; never by the
product path, which has no CPU implementation).

What is differentiated is the forward of ``oracle.ref.attn_fwd``: out = attention(norm(rope(q)), norm(rope(k)), v)
with the causal / window mask, the 1/sqrt(D) scale times the QK-norm gain, and GQA grouping ("nanochat Admin &
Developer Guide", section 3; the model trains through it with autograd).  The gradients are written out from the
chain rule, step by step in the forward's order reversed:

* attention, per (b, query head h, kv head g = h // G), with P = softmax(S), O = P V:
  dV_g += P^T dO,  dP = dO V_g^T,  dS = P * (dP - rowsum(P * dP)),  dqn_h = c dS kn_g,  dkn_g += c dS^T qn_h,
  where c = qk_gain / sqrt(D) and masked entries have P = 0 (so dS = 0 there);
* weightless RMSNorm y = x / r, r = sqrt(mean(x^2) + eps):  dx = dy / r - x (dy . x) / (D r^3);
* RoPE is a rotation of each pair (i, i + D/2) by t theta_i, so its backward is the rotation by -t theta_i.

Pinned against central finite differences of the forward oracle (``tests/test_oracle_backward.py``).
"""

import numpy as np

from oracle import ref


def rope_bwd(dy, pos, base=ref.ROPE_BASE):
    """Gradient through ``ref.rope`` at the given positions: the transposed rotation, i.e. RoPE at -pos."""
    return ref.rope(dy, -np.asarray(pos, dtype=np.float64), base)


def rms_norm_bwd(dy, x, eps=ref.RMS_EPS):
    """Gradient through ``ref.rms_norm`` (over the last axis) for upstream gradient dy at input x."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    D = x.shape[-1]
    r2 = np.mean(x * x, axis=-1, keepdims=True) + eps
    r = np.sqrt(r2)
    return dy / r - x * np.sum(dy * x, axis=-1, keepdims=True) / (D * r2 * r)


def attn_fwd_bwd(q, k, v, dout, window, rope_base=ref.ROPE_BASE, eps=ref.RMS_EPS, qk_gain=1.0):
    """Forward output and gradients of sum(dout * out) with respect to q, k, v.

    q: [B, T, Hq, D], k and v: [B, T, Hkv, D], dout: [B, T, Hq, D].  Returns (out, dq, dk, dv), all fp64.
    Dense over T (full score matrices): for the small cases the tests use.
    """
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    pos = np.broadcast_to(np.arange(T), (B, T))
    qr, kr = ref.rope(q, pos, rope_base), ref.rope(k, pos, rope_base)
    qn, kn = ref.rms_norm(qr, eps), ref.rms_norm(kr, eps)
    c = qk_gain / np.sqrt(D)
    mask = ref.visible(np.arange(T)[:, None], np.arange(T)[None, :], window)
    out = np.zeros_like(q)
    dqn = np.zeros_like(q)
    dkn = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = np.where(mask, (qn[b, :, h] @ kn[b, :, g].T) * c, -np.inf)
            p = np.exp(s - s.max(axis=-1, keepdims=True))
            p /= p.sum(axis=-1, keepdims=True)
            out[b, :, h] = p @ v[b, :, g]
            do = dout[b, :, h]
            dv[b, :, g] += p.T @ do
            dp = do @ v[b, :, g].T
            ds = p * (dp - np.sum(p * dp, axis=-1, keepdims=True))
            dqn[b, :, h] = c * (ds @ kn[b, :, g])
            dkn[b, :, g] += c * (ds.T @ qn[b, :, h])
    dq = rope_bwd(rms_norm_bwd(dqn, qr, eps), pos, rope_base)
    dk = rope_bwd(rms_norm_bwd(dkn, kr, eps), pos, rope_base)
    return out, dq, dk, dv
