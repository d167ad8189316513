"""GPU parity of the backward pass (through the C ABI) against the fp64 backward oracle, which is pinned by finite
differences.

The tensor-core kernels take their operands in bf16, as the forward does: the roped + normed q and k (rounded once),
the probabilities P and dS = P (dP - rowsum(dO O)) (rounded before each product); every sum is accumulated in fp32.
Each rounding moves its value by at most 2^-9 relatively, and a gradient element sums products carrying a few of them,
so its error stays within a few 2^-9 of the gradient's own scale (measured: 0.3-0.45 % of max |ref| at most, 0.3 % of
mean |ref| on average).  The bar: max-abs <= 2^-6 max |ref| + 1e-4 and mean-abs <= 2^-7 mean |ref| + 1e-5 per
gradient.  A wrong or missing term (the rowsum, the norm's projection, the RoPE direction) moves the gradients by
tens of percent.
"""

import numpy as np
import pytest
import torch

from oracle import backward
from seeded_inputs import bwd_inputs
from tests.parity import f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_attention_06_b300 import nc_attn
    nc_attn.nc_attn_get_device_status(clear=True)
    yield nc_attn
    assert nc_attn.nc_attn_get_device_status(clear=True) == nc_attn.NC_OK


def check(got, exp, what):
    g = got.detach().double().cpu().numpy()
    assert np.isfinite(g).all(), what
    d = np.abs(g - exp)
    mx, mn = 2.0 ** -6 * np.abs(exp).max() + 1e-4, 2.0 ** -7 * np.abs(exp).mean() + 1e-5
    assert d.max() <= mx and d.mean() <= mn, f"{what}: max-abs {d.max():.3e} (<= {mx:.2e}), mean {d.mean():.3e} (<= {mn:.2e})"


# (B, T, Hq, Hkv, window, gain)
CASES = [
    (1, 37, 4, 2, -1, 1.0),
    (2, 130, 6, 2, 50, 1.0),
    (1, 200, 8, 8, 0, 1.0),      # window 0: dq = dk = 0 exactly
    (1, 260, 12, 4, -1, 1.2),
    (1, 150, 16, 1, 20, 1.0),
    (1, 300, 3, 1, 100, 1.0),    # group of 3: 126 of the 128 packed rows hold queries
    (1, 129, 10, 2, 128, 4.0),   # group of 5, window = T - 1, largest gain
    (2, 1, 4, 4, -1, 1.0),       # one token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}_T{c[1]}_Hq{c[2]}_Hkv{c[3]}_W{c[4]}_g{c[5]}")
def test_bwd_matches_oracle(nc, case):
    B, T, Hq, Hkv, W, gain = case
    q, k, v, dout = bwd_inputs(B, T, Hq, Hkv, 128, seed=T + Hq)
    dq, dk, dv = nc.nc_attn_bwd(q.cuda(), k.cuda(), v.cuda(), dout.cuda(), window=W, qk_gain=gain)
    torch.cuda.synchronize()
    _, rq, rk, rv = backward.attn_fwd_bwd(f64(q), f64(k), f64(v), f64(dout), W, qk_gain=gain)
    check(dq, rq, f"dq {case}")
    check(dk, rk, f"dk {case}")
    check(dv, rv, f"dv {case}")


@pytest.mark.parametrize("W", [1024, 2048])
def test_bwd_full_size_is_linear_and_independent_of_the_schedule(nc, W):
    """The depth-12 layer (B=4, T=2048, Hq=Hkv=6) as the bench times it: finite gradients, linear in dout, and every
    sequence's gradients bit-identical to a call on that sequence alone (each gradient row is accumulated by one CTA in
    a fixed order, whichever CTA takes the item), so the full-size result is the oracle-checked one-sequence result."""
    q, k, v, dout = (t.cuda() for t in bwd_inputs(4, 2048, 6, 6, 128, seed=0))
    g1 = nc.nc_attn_bwd(q, k, v, dout, window=W)
    g1 = [x.clone() for x in g1]
    g2 = nc.nc_attn_bwd(q, k, v, (2 * dout.float()).to(torch.bfloat16), window=W)   # exact doubling in bf16
    for a, b in zip(g1, g2):
        assert torch.isfinite(a).all()
        torch.testing.assert_close(b, 2 * a, rtol=1e-5, atol=1e-6)
    for b in range(4):
        one = nc.nc_attn_bwd(*(x[b:b + 1].contiguous() for x in (q, k, v, dout)), window=W)
        for a, o in zip(g1, one):
            assert torch.equal(a[b:b + 1], o)


@pytest.mark.parametrize("Hq,Hkv,W", [(6, 6, 1024), (16, 4, 2048)])
def test_bwd_full_length_one_sequence_matches_oracle(nc, Hq, Hkv, W):
    """T = 2048 on one sequence with the depth-12 (Hq = Hkv = 6, window 1024) and the GQA (Hq = 16, Hkv = 4, full
    causal) head layouts, every gradient element against the dense oracle."""
    q, k, v, dout = bwd_inputs(1, 2048, Hq, Hkv, 128, seed=0)
    dq, dk, dv = nc.nc_attn_bwd(q.cuda(), k.cuda(), v.cuda(), dout.cuda(), window=W)
    torch.cuda.synchronize()
    _, rq, rk, rv = backward.attn_fwd_bwd(f64(q), f64(k), f64(v), f64(dout), W)
    check(dq, rq, f"dq Hq={Hq} Hkv={Hkv} W={W}")
    check(dk, rk, f"dk Hq={Hq} Hkv={Hkv} W={W}")
    check(dv, rv, f"dv Hq={Hq} Hkv={Hkv} W={W}")


# ---- training path: a forward that keeps its row statistics, a backward that reuses them -------------------------
SAVED_CASES = [
    (1, 37, 4, 2, -1, 1.0),
    (2, 130, 6, 2, 50, 1.2),
    (1, 300, 3, 1, 100, 1.0),    # group of 3: 126 of the 128 packed rows hold queries
    (1, 129, 10, 2, 128, 4.0),   # group of 5, window = T - 1, largest gain
    (1, 2048, 6, 6, 1024, 1.0),  # a depth-12 layer's sequence at full length
]


def oracle_lse2(q, k, W, gain):
    """Base-2 log-sum-exp of every query row's logits gain qn . kn_j / sqrt(D) over its visible keys, [B, T, Hq]."""
    from oracle import ref
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    pos = np.broadcast_to(np.arange(T), (B, T))
    qn, kn = ref.qk_prologue(f64(q), pos), ref.qk_prologue(f64(k), pos)
    mask = ref.visible(np.arange(T)[:, None], np.arange(T)[None, :], W)
    out = np.empty((B, T, Hq))
    for b in range(B):
        for h in range(Hq):
            s = np.where(mask, qn[b, :, h] @ kn[b, :, h // G].T * gain / np.sqrt(D), -np.inf)
            m = s.max(axis=1, keepdims=True)
            out[b, :, h] = (np.log(np.exp(s - m).sum(axis=1)) + m[:, 0]) / np.log(2.0)
    return out


def unpack_lse(lse, B, T, Hq, Hkv):
    """[B, T, Hq] view of the packed statistics, and the entries of rows that hold no query (must be zero)."""
    G = Hq // Hkv
    P = 128 // G
    nt = (T + P - 1) // P
    a = lse[: B * Hkv * nt * 128].view(B, Hkv, nt, 128).double().cpu().numpy()
    rows = np.empty((B, T, Hq))
    pad = []
    for r in range(128):
        t_off, j = divmod(r, G)
        for m in range(nt):
            t = m * P + t_off
            if r < G * P and t < T:
                rows[:, t, np.arange(Hkv) * G + j] = a[:, :, m, r]
            else:
                pad.append(a[:, :, m, r])
    return rows, (np.concatenate([x.ravel() for x in pad]) if pad else np.zeros(0))


@pytest.mark.parametrize("case", SAVED_CASES, ids=lambda c: f"B{c[0]}_T{c[1]}_Hq{c[2]}_Hkv{c[3]}_W{c[4]}_g{c[5]}")
def test_saved_statistics_forward_and_backward_match_oracle(nc, case):
    B, T, Hq, Hkv, W, gain = case
    q, k, v, dout = bwd_inputs(B, T, Hq, Hkv, 128, seed=T + Hq + 1)
    qc, kc, vc, dc = (x.cuda() for x in (q, k, v, dout))
    out, lse = nc.nc_attn_fwd_lse(qc, kc, vc, window=W, qk_gain=gain)
    torch.cuda.synchronize()
    # the statistics: the logits come from qn, kn rounded to bf16 (2^-9 relative each), so their error, and that of
    # the log-sum-exp the largest of them dominate, grows with the logits, i.e. with the gain (|s| <= 16.5 gain in
    # log2 units); the probabilities' own bf16 rounding adds < 0.006.  The bar scales with the gain as the output's
    # does.
    rows, pad = unpack_lse(lse, B, T, Hq, Hkv)
    ref_lse = oracle_lse2(q, k, W, gain)
    assert np.abs(rows - ref_lse).max() < 2e-2 * max(1.0, gain / 1.2)
    assert (pad == 0).all()
    # the kept output is the forward's output
    ro, rq, rk, rv = backward.attn_fwd_bwd(f64(q), f64(k), f64(v), f64(dout), W, qk_gain=gain)
    o = out.double().cpu().numpy()
    assert np.abs(o - ro).max() <= 2e-2 * max(1.0, gain / 1.2)
    dq, dk, dv = nc.nc_attn_bwd_saved(qc, kc, vc, out, dc, lse, window=W, qk_gain=gain)
    torch.cuda.synchronize()
    check(dq, rq, f"saved dq {case}")
    check(dk, rk, f"saved dk {case}")
    check(dv, rv, f"saved dv {case}")
