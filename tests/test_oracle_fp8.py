"""Pins for the fp8 (e4m3) variant of the oracle (CPU only).

The e4m3 rounding is pinned three ways that share nothing with its own arithmetic: the code table written out from
the format's bit layout, an exhaustive nearest-value search with ties to even (``oracle.brute``), and torch's own
float8_e4m3fn conversion (a library routine).  The quantised attention is pinned by brute force on tiny inputs, by
the invariants that survive quantisation exactly (position 0, window >= T - 1, GQA = repeated-KV MHA), and by its
distance to the unquantised oracle, which a wrong dequantisation scale would blow far past.
"""

import math

import numpy as np
import pytest
import torch

from oracle import fp8, ref
from oracle.brute import attn_fwd_fp8_brute, e4m3_nearest
from seeded_inputs import fwd_inputs


def f64(t):
    return t.to(torch.float64).numpy()


def test_e4m3_code_table_closed_form():
    vals = [fp8.e4m3_decode(c) for c in range(256)]
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    assert sum(not math.isnan(x) for x in vals) == 254
    assert vals[0x7E] == 448.0 and vals[0xFE] == -448.0            # largest finite: 1.75 * 2^8
    assert vals[0x01] == 2.0 ** -9                                  # smallest subnormal
    assert vals[0x07] == 7 * 2.0 ** -9                              # largest subnormal
    assert vals[0x08] == 2.0 ** -6                                  # smallest normal
    assert vals[0x38] == 1.0 and vals[0x39] == 1.125 and vals[0xB8] == -1.0
    pos = sorted(x for x in vals[:0x7F])
    assert all(b > a for a, b in zip(pos, pos[1:]))                 # codes 0..0x7E increase strictly


def test_e4m3_round_trips_every_finite_code():
    for c in range(256):
        x = fp8.e4m3_decode(c)
        if not math.isnan(x):
            assert fp8.e4m3_round(np.array([x]))[0] == x


def test_e4m3_round_matches_exhaustive_search_and_ties_go_to_even():
    finite = sorted({fp8.e4m3_decode(c) for c in range(256) if not math.isnan(fp8.e4m3_decode(c))})
    mids = [(a + b) / 2 for a, b in zip(finite, finite[1:])]          # every tie
    rng = np.random.default_rng(0)
    rand = list(rng.uniform(-448, 448, 300)) + list(rng.uniform(-0.05, 0.05, 300))
    xs = np.array(mids + rand)
    got = fp8.e4m3_round(xs)
    exp = np.array([e4m3_nearest(x) for x in xs])
    np.testing.assert_array_equal(got, exp)


def test_e4m3_round_matches_torch_float8_cast():
    rng = np.random.default_rng(1)
    x = rng.uniform(-448, 448, 200000) * rng.choice([1, 1e-1, 1e-2, 1e-3, 1e-4], 200000)
    np.testing.assert_array_equal(fp8.e4m3_round(x), torch.tensor(x).to(torch.float8_e4m3fn).double().numpy())


def test_e4m3_round_rejects_out_of_range():
    with pytest.raises(ValueError):
        fp8.e4m3_round(np.array([449.0]))
    with pytest.raises(ValueError):
        fp8.e4m3_round(np.array([np.nan]))


def test_scales_turn_the_quantised_product_into_base2_logits():
    for g in (1.0, 1.2, 4.0):
        s_q, s_k = fp8.fp8_scales(g)
        assert g / math.sqrt(128) / (s_q * s_k) == pytest.approx(math.log(2), rel=1e-15)
        # the largest possible element of a unit-RMS vector, sqrt(128), stays inside e4m3's range
        assert math.sqrt(128) * s_q < fp8.E4M3_MAX and math.sqrt(128) * s_k < fp8.E4M3_MAX


@pytest.mark.parametrize("T,Hq,Hkv,W", [(1, 1, 1, -1), (7, 2, 1, -1), (9, 4, 2, 3), (12, 2, 2, 0)])
def test_fp8_oracle_matches_brute_force(T, Hq, Hkv, W):
    q, k, v = fwd_inputs(1, T, Hq, Hkv, 128, seed=T * 7 + Hq)
    s_q, s_k = fp8.fp8_scales()
    exp = np.array(attn_fwd_fp8_brute(f64(q), f64(k), f64(v), W, s_q, s_k))
    np.testing.assert_allclose(fp8.attn_fwd_fp8(f64(q), f64(k), f64(v), W), exp, rtol=0, atol=1e-12)


def test_fp8_invariants_hold_exactly():
    q, k, v = (f64(t) for t in fwd_inputs(2, 150, 8, 2, 128, seed=3))
    full = fp8.attn_fwd_fp8(q, k, v, -1)
    np.testing.assert_array_equal(fp8.attn_fwd_fp8(q, k, v, 149), full)       # window >= T - 1: full causal
    for h in range(8):
        np.testing.assert_allclose(full[:, 0, h], v[:, 0, h // 4], rtol=0, atol=1e-15)   # position 0 sees v_0
    mha = fp8.attn_fwd_fp8(q, np.repeat(k, 4, axis=2), np.repeat(v, 4, axis=2), 40)
    np.testing.assert_allclose(fp8.attn_fwd_fp8(q, k, v, 40), mha, rtol=0, atol=1e-13)


def test_fp8_oracle_stays_near_the_exact_result_and_a_wrong_scale_does_not():
    """Quantising qn, kn to e4m3 (3 mantissa bits) moves the outputs by ~5e-3 on average; a dequantisation off by a
    factor 2 either way (a plausible slip: the logits' temperature halved or doubled) moves them by far more."""
    q, k, v = (f64(t) for t in fwd_inputs(1, 256, 4, 2, 128, seed=4))
    exact = ref.attn_fwd(q, k, v, 128)
    d = np.abs(fp8.attn_fwd_fp8(q, k, v, 128) - exact)
    assert 1e-4 < d.mean() < 1e-2 and d.max() < 0.1
    for wrong in (0.5, 2.0):
        dw = np.abs(ref.attn_fwd(q, k, v, 128, qk_gain=wrong) - exact)
        assert dw.mean() > 5 * d.mean()
