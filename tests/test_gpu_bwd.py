"""GPU parity of the backward pass (through the C ABI) against the fp64 backward oracle, which is pinned by finite
differences.

The kernels compute in fp32 from the same bf16 inputs the oracle reads exactly, so the gradients agree to fp32
rounding accumulated over a row's keys: the bar is max-abs <= 1e-3 (1 + max |ref|) and mean-abs <= 1e-4
(1 + mean |ref|) per gradient, two orders above that rounding and far below what a wrong or missing term gives.
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
    mx, mn = 1e-3 * (1 + np.abs(exp).max()), 1e-4 * (1 + np.abs(exp).mean())
    assert d.max() <= mx and d.mean() <= mn, f"{what}: max-abs {d.max():.3e} (<= {mx:.2e}), mean {d.mean():.3e} (<= {mn:.2e})"


# (B, T, Hq, Hkv, window, gain)
CASES = [
    (1, 37, 4, 2, -1, 1.0),
    (2, 130, 6, 2, 50, 1.0),
    (1, 200, 8, 8, 0, 1.0),
    (1, 260, 12, 4, -1, 1.2),
    (1, 150, 16, 1, 20, 1.0),
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


def test_bwd_full_size_is_finite_and_linear(nc):
    """The depth-12 layer (B=4, T=2048, Hq=Hkv=6, window 1024): finite gradients, linear in dout."""
    q, k, v, dout = (t.cuda() for t in bwd_inputs(4, 2048, 6, 6, 128, seed=0))
    g1 = nc.nc_attn_bwd(q, k, v, dout, window=1024)
    g2 = nc.nc_attn_bwd(q, k, v, (2 * dout.float()).to(torch.bfloat16), window=1024)   # exact doubling in bf16
    for a, b in zip(g1, g2):
        assert torch.isfinite(a).all()
        torch.testing.assert_close(b, 2 * a, rtol=1e-5, atol=1e-6)


def test_bwd_depth12_layer_one_sequence_matches_oracle(nc):
    """The depth-12 layer shapes (T=2048, Hq=Hkv=6, window 1024) on one sequence, every gradient element against the
    dense oracle."""
    q, k, v, dout = bwd_inputs(1, 2048, 6, 6, 128, seed=0)
    dq, dk, dv = nc.nc_attn_bwd(q.cuda(), k.cuda(), v.cuda(), dout.cuda(), window=1024)
    torch.cuda.synchronize()
    _, rq, rk, rv = backward.attn_fwd_bwd(f64(q), f64(k), f64(v), f64(dout), 1024)
    check(dq, rq, "dq depth-12 layer")
    check(dk, rk, "dk depth-12 layer")
    check(dv, rv, "dv depth-12 layer")
