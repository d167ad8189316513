"""Pins for the fp64 backward oracle (CPU only): central finite differences of the forward oracle.

L(q, k, v) = sum(dout * attn_fwd(q, k, v)) is differentiated numerically with h = 1e-5 (error ~1e-10 at these sizes)
and compared with ``oracle.backward.attn_fwd_bwd``.  A dropped term of the softmax backward, a missing sum over the
heads of a GQA group, the RMSNorm backward's second term, the rotation direction of the RoPE backward or the gain
would each fail a check; the window-0 case pins dv exactly and dq = dk = 0.
"""

import numpy as np
import pytest

from oracle import backward, ref

H = 1e-5


def loss(q, k, v, dout, W, gain):
    return float(np.sum(dout * ref.attn_fwd(q, k, v, W, qk_gain=gain)))


def inputs(B, T, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D))
    k = rng.standard_normal((B, T, Hkv, D))
    v = rng.standard_normal((B, T, Hkv, D))
    dout = rng.standard_normal((B, T, Hq, D))
    return q, k, v, dout


@pytest.mark.parametrize("W,gain", [(-1, 1.0), (2, 1.0), (-1, 1.2), (1, 3.0)])
def test_every_coordinate_against_central_differences(W, gain):
    q, k, v, dout = inputs(1, 5, 4, 2, 4, seed=W + 10)
    out, dq, dk, dv = backward.attn_fwd_bwd(q, k, v, dout, W, qk_gain=gain)
    np.testing.assert_allclose(out, ref.attn_fwd(q, k, v, W, qk_gain=gain), rtol=0, atol=1e-13)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += H
            xm[idx] -= H
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"], dout, W, gain) -
                        loss(args_m["q"], args_m["k"], args_m["v"], dout, W, gain)) / (2 * H)
        np.testing.assert_allclose(grad, num, rtol=0, atol=2e-8, err_msg=f"d{name} W={W} gain={gain}")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_directional_derivatives_at_head_dim_128(seed):
    """Full head dim, GQA, a window: the gradient against random directions."""
    q, k, v, dout = inputs(2, 9, 6, 2, 128, seed=seed)
    W = 4
    _, dq, dk, dv = backward.attn_fwd_bwd(q, k, v, dout, W)
    rng = np.random.default_rng(100 + seed)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        d = rng.standard_normal(x.shape)
        args = {"q": q, "k": k, "v": v}
        ap, am = dict(args), dict(args)
        ap[name], am[name] = x + H * d, x - H * d
        num = (loss(ap["q"], ap["k"], ap["v"], dout, W, 1.0) - loss(am["q"], am["k"], am["v"], dout, W, 1.0)) / (2 * H)
        assert abs(np.sum(grad * d) - num) <= 1e-7 * max(1.0, abs(num)), name


def test_window_zero():
    """Each query sees only its own key: out_t = v_t, so dv_t is the sum of dout over the group and dq = dk = 0."""
    q, k, v, dout = inputs(2, 6, 6, 2, 8, seed=5)
    out, dq, dk, dv = backward.attn_fwd_bwd(q, k, v, dout, 0)
    np.testing.assert_allclose(out, np.repeat(v, 3, axis=2), rtol=0, atol=1e-15)
    np.testing.assert_allclose(dv, dout.reshape(2, 6, 2, 3, 8).sum(axis=3), rtol=0, atol=1e-14)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
