"""GPU parity of the prefill with e4m3 score operands (``nc_attn_fwd_fp8``, through the C ABI) against the fp8 oracle
(``oracle.fp8``), which quantises the same real numbers qn * s_q and kn * s_k to e4m3.

The kernels form qn * s_q in fp32, the oracle in fp64; the two round to the same e4m3 code except where the fp32
value lies within ~1e-7 (relative) of a rounding midpoint, i.e. for a few elements per million, each then one code
apart.  The prologue test checks exactly that.  Past the quantisation both sides do what the bf16 path does (P rounded
to bf16, fp32 accumulation), so the outputs are held to the same bar as the bf16 path: max-abs 2e-2, mean-abs 2e-3,
element by element, the full-size workloads included.
"""

import numpy as np
import pytest
import torch

from oracle import fp8, ref
from seeded_inputs import DEPTH12, GQA, LONG, TINY, fwd_inputs
from tests.parity import MAX_ABS, MEAN_ABS, assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_attention_06_b300 import nc_attn
    nc_attn.nc_attn_get_device_status(clear=True)
    yield nc_attn
    assert nc_attn.nc_attn_get_device_status(clear=True) == nc_attn.NC_OK


def cuda(*ts):
    return [t.cuda() for t in ts]


def e4m3_values(codes):
    """Decoded values of a uint8 tensor of e4m3 codes (torch's float8_e4m3fn view of the same bytes)."""
    return codes.cpu().view(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("gain", [1.0, 1.2, 4.0])
def test_prologue_codes_match_the_oracle_quantisation(nc, gain):
    B, T, Hq, Hkv = 2, 700, 12, 4
    q, k, _ = fwd_inputs(B, T, Hq, Hkv, 128, seed=11)
    qn8, kn8 = nc.nc_attn_qk_prologue_fp8(*cuda(q, k), qk_gain=gain)
    torch.cuda.synchronize()
    s_q, s_k = fp8.fp8_scales(gain)
    pos = np.broadcast_to(np.arange(T), (B, T))
    finite = np.array(sorted({x for x in map(fp8.e4m3_decode, range(256)) if x == x}))   # the 253 distinct values
    for got8, x, s in ((qn8, q, s_q), (kn8, k, s_k)):
        exact = ref.qk_prologue(f64(x), pos) * s
        exp = fp8.e4m3_round(exact)
        got = e4m3_values(got8)
        bad = got != exp
        assert bad.mean() < 1e-4, f"{bad.sum()} of {bad.size} codes differ"
        if bad.any():
            # a differing code is the other neighbour of a value that sits at a rounding midpoint
            lo = finite[np.searchsorted(finite, exact[bad], side="right") - 1]
            hi = finite[np.searchsorted(finite, exact[bad], side="left")]
            assert np.all((got[bad] == lo) | (got[bad] == hi))
            assert np.all(np.abs(np.abs(exact[bad] - lo) - np.abs(hi - exact[bad])) <= 1e-6 * np.abs(exact[bad]))


@pytest.mark.parametrize("W", TINY.windows)
def test_fwd_fp8_tiny_config(nc, W):
    w = TINY
    q, k, v = fwd_inputs(w.B, w.T, w.Hq, w.Hkv, w.D, seed=0)
    out = nc.nc_attn_fwd_fp8(*cuda(q, k, v), window=W)
    assert_close(out, fp8.attn_fwd_fp8(f64(q), f64(k), f64(v), W), f"fp8 tiny W={W}")


ODD = [  # (B, T, Hq, Hkv, W, gain): ragged tails, group sizes, windows, gains
    (1, 1, 1, 1, -1, 1.0),
    (2, 7, 2, 1, -1, 1.0),
    (1, 130, 3, 1, 5, 1.0),
    (2, 300, 8, 2, 127, 1.2),
    (1, 257, 12, 4, 0, 1.0),
    (1, 384, 16, 4, 200, 4.0),
    (1, 33, 128, 1, -1, 1.0),
    (2, 77, 10, 2, 30, 1.0),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,W,gain", ODD)
def test_fwd_fp8_odd_shapes(nc, B, T, Hq, Hkv, W, gain):
    q, k, v = fwd_inputs(B, T, Hq, Hkv, 128, seed=T + Hq)
    out = nc.nc_attn_fwd_fp8(*cuda(q, k, v), window=W, qk_gain=gain)
    exp = fp8.attn_fwd_fp8(f64(q), f64(k), f64(v), W, qk_gain=gain)
    # as on the bf16 path, the rounding carried by the logits grows with the gain, and so does the bar
    f = max(1.0, gain / 1.2)
    assert_close(out, exp, f"fp8 B{B} T{T} Hq{Hq} Hkv{Hkv} W{W} g{gain}", max_abs=MAX_ABS * f, mean_abs=MEAN_ABS * f)


FULL = [(DEPTH12, li, W) for li, W in enumerate(DEPTH12.windows)] + \
       [(GQA, li, W) for li, W in enumerate(GQA.windows)] + [(LONG, li, W) for li, W in enumerate(LONG.windows)]


@pytest.mark.parametrize("wl,seed,W", FULL, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_fwd_fp8_full_size_every_element(nc, wl, seed, W):
    q, k, v = fwd_inputs(wl.B, wl.T, wl.Hq, wl.Hkv, wl.D, seed=seed)
    out = nc.nc_attn_fwd_fp8(*cuda(q, k, v), window=W)
    torch.cuda.synchronize()
    g = f64(out)
    exp = fp8.attn_fwd_fp8(f64(q), f64(k), f64(v), W)
    d = np.abs(g - exp)
    worst = np.unravel_index(int(np.argmax(d)), d.shape)[:3]
    assert np.isfinite(g).all()
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (
        f"{wl.name} W={W}: max-abs {d.max():.3e} at (b, t, h) = {tuple(int(x) for x in worst)}, mean {d.mean():.3e}")


def test_fp8_window_at_least_T_minus_1_equals_full_causal_and_position_0(nc):
    q, k, v = cuda(*fwd_inputs(2, 515, 6, 2, 128, seed=5))
    full = nc.nc_attn_fwd_fp8(q, k, v, window=-1).clone()
    for W in (514, 100000):
        assert torch.equal(nc.nc_attn_fwd_fp8(q, k, v, window=W), full)
    for h in range(6):
        assert torch.equal(full[:, 0, h], v[:, 0, h // 3])
