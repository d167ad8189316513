"""Pins for the fp64 oracle (CPU only).

The pages print no worked numeric example for RoPE, the norm or attention, so the oracle is pinned by
closed forms written out by hand, by brute force on tiny inputs (``oracle.brute``) and by invariants of the
mathematics.  Each test names the plausible mistake it would catch.
"""

import math

import numpy as np
import pytest
import torch

from oracle import ref
from oracle.brute import attn_decode_brute, attn_fwd_brute
from seeded_inputs import TINY, decode_inputs, fwd_inputs

GPU_MAX_ABS = 2e-2   # tolerance of the GPU parity tests (bf16 outputs, fp32 accumulation)


def f64(t):
    return t.to(torch.float64).numpy()


# ----------------------------------------------------------------------------------------------------------
# RoPE: closed forms
# ----------------------------------------------------------------------------------------------------------

def test_inv_freq_closed_form():
    th = ref.inv_freq(128, 100000.0)
    assert th.shape == (64,)
    assert th[0] == 1.0
    assert th[32] == pytest.approx(0.0031622776601683794, rel=1e-15)        # 1e5^(-1/2)
    assert th[63] == pytest.approx(100000.0 ** (-126.0 / 128.0), rel=1e-15)
    assert np.all(np.diff(th) < 0)                                          # strictly decreasing


@pytest.mark.parametrize("t", [0, 1, 3, 2047, 8191])
def test_rope_basis_vectors_closed_form(t):
    """Half-split pairing (i, i+D/2), frequency base^(-2i/D), and the rotation sign, on basis vectors (D=4).

    Catches: interleaved pairing, a wrong frequency exponent, a transposed rotation.
    """
    D = 4
    th1 = 100000.0 ** (-0.5)
    a0, a1 = t * 1.0, t * th1
    E = np.eye(D)[:, None, :]                          # [4 tokens, 1 head, D]: token r holds e_r
    pos = np.full((D,), t)
    y = ref.rope(E, pos)[:, 0, :]                      # row r = rope(e_r)
    exp = np.zeros((D, D))
    exp[0] = [math.cos(a0), 0, -math.sin(a0), 0]       # e_0 -> (cos a, 0, -sin a, 0)
    exp[2] = [math.sin(a0), 0, math.cos(a0), 0]        # e_2 -> (sin a, 0,  cos a, 0)
    exp[1] = [0, math.cos(a1), 0, -math.sin(a1)]
    exp[3] = [0, math.sin(a1), 0, math.cos(a1)]
    np.testing.assert_allclose(y, exp, atol=1e-12)


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((3, 5, 2, 128))
    y = ref.rope(x, np.zeros((3, 5)))
    np.testing.assert_array_equal(y, x)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 64, 3, 128))
    pos = np.broadcast_to(np.arange(64) * 97, (2, 64))
    y = ref.rope(x, pos)
    np.testing.assert_allclose(y[..., :64] ** 2 + y[..., 64:] ** 2, x[..., :64] ** 2 + x[..., 64:] ** 2,
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shift", [1, 17, 4000])
def test_rope_relative_position(shift):
    """rope(q, m) . rope(k, n) depends only on m - n."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    for m, n in [(5, 2), (100, 0), (2048, 1024)]:
        d0 = float(ref.rope(q, np.array([m]))[0, 0] @ ref.rope(k, np.array([n]))[0, 0])
        d1 = float(ref.rope(q, np.array([m + shift]))[0, 0] @ ref.rope(k, np.array([n + shift]))[0, 0])
        assert d0 == pytest.approx(d1, abs=1e-9)


# ----------------------------------------------------------------------------------------------------------
# RMSNorm (QK-norm): closed form and invariants
# ----------------------------------------------------------------------------------------------------------

def test_rms_norm_closed_form():
    x = np.array([3.0, 4.0, 0.0, 0.0])
    y = ref.rms_norm(x)
    np.testing.assert_allclose(y, x / math.sqrt(25.0 / 4.0 + 1e-6), rtol=1e-15)
    c = np.full(128, -2.5)
    np.testing.assert_allclose(ref.rms_norm(c), -2.5 / math.sqrt(6.25 + 1e-6), rtol=1e-15)


def test_unit_rms_after_norm():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 32, 6, 128))
    y = ref.qk_prologue(x, np.broadcast_to(np.arange(32), (4, 32)))
    rms = np.sqrt(np.mean(y * y, axis=-1))
    assert np.max(np.abs(rms - 1.0)) < 1e-6


def test_norm_and_rope_commute():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 16, 3, 128))
    pos = np.broadcast_to(np.arange(16) * 511, (2, 16))
    a = ref.rms_norm(ref.rope(x, pos))
    b = ref.rope(ref.rms_norm(x), pos)
    np.testing.assert_allclose(a, b, atol=1e-12)


# ----------------------------------------------------------------------------------------------------------
# Attention: closed forms
# ----------------------------------------------------------------------------------------------------------

def test_two_key_attention_closed_form():
    """D=2, T=2: all of RoPE, the norm, the 1/sqrt(D) scale and the softmax written out by hand.

    q_1 = k_0 = k_1 = (1, 0).  After RoPE at positions 1, 0, 1 and the norm (mean square 1/2):
      qn_1 = (cos 1, -sin 1)/r,  kn_0 = (1, 0)/r,  kn_1 = (cos 1, -sin 1)/r,  r^2 = 1/2 + eps.
      s_0 = cos(1) / r^2 / sqrt(2),  s_1 = 1 / r^2 / sqrt(2),  p_1 = 1 / (1 + exp(s_0 - s_1)).
    """
    eps = 1e-6
    q = np.zeros((1, 2, 1, 2))
    k = np.zeros((1, 2, 1, 2))
    q[0, 1, 0] = [1, 0]
    q[0, 0, 0] = [0.3, -0.7]
    k[0, 0, 0] = [1, 0]
    k[0, 1, 0] = [1, 0]
    v = np.array([[[[1.5, -2.0]], [[0.25, 4.0]]]])
    r2 = 0.5 + eps
    s0 = math.cos(1.0) / r2 / math.sqrt(2.0)
    s1 = 1.0 / r2 / math.sqrt(2.0)
    p1 = 1.0 / (1.0 + math.exp(s0 - s1))
    exp1 = (1 - p1) * v[0, 0, 0] + p1 * v[0, 1, 0]
    out = ref.attn_fwd(q, k, v, window=-1)
    np.testing.assert_allclose(out[0, 1, 0], exp1, rtol=1e-13)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 0], rtol=0, atol=0)
    # window 0: only the diagonal is visible
    np.testing.assert_allclose(ref.attn_fwd(q, k, v, window=0)[0, 1, 0], v[0, 1, 0], atol=0)
    # the same closed form through the one-row path
    np.testing.assert_allclose(ref.attn_fwd_rows(q, k, v, -1, [(0, 1, 0)])[0], exp1, rtol=1e-13)


@pytest.mark.parametrize("gain", [1.2, 0.5, 3.0])
def test_qk_gain_closed_form(gain):
    """The QK-norm gain (1.2 in the Guide) multiplies both logits of the two-key case above: p_1 =
    1 / (1 + exp(gain (s_0 - s_1))), through the prefill, one-row, decode and chunk paths."""
    eps = 1e-6
    q = np.zeros((1, 2, 1, 2))
    k = np.zeros((1, 2, 1, 2))
    q[0, 1, 0] = [1, 0]
    q[0, 0, 0] = [0.3, -0.7]
    k[0, 0, 0] = [1, 0]
    k[0, 1, 0] = [1, 0]
    v = np.array([[[[1.5, -2.0]], [[0.25, 4.0]]]])
    r2 = 0.5 + eps
    s0 = math.cos(1.0) / r2 / math.sqrt(2.0)
    s1 = 1.0 / r2 / math.sqrt(2.0)
    p1 = 1.0 / (1.0 + math.exp(gain * (s0 - s1)))
    exp1 = (1 - p1) * v[0, 0, 0] + p1 * v[0, 1, 0]
    np.testing.assert_allclose(ref.attn_fwd(q, k, v, -1, qk_gain=gain)[0, 1, 0], exp1, rtol=1e-13)
    np.testing.assert_allclose(ref.attn_fwd_rows(q, k, v, -1, [(0, 1, 0)], qk_gain=gain)[0], exp1, rtol=1e-13)
    # decode of position 1 against a cache holding key 0 (roped at 0 = itself, normed) plus key 1 as the new key
    kc = np.zeros((1, 2, 1, 2))
    kc[0, 0, 0] = np.array([1.0, 0.0]) / math.sqrt(r2)
    vc = np.zeros((1, 2, 1, 2))
    vc[0, 0] = v[0, 0]
    dec, _ = ref.attn_decode(q[:, 1], kc, vc, np.array([1]), -1, k_new=k[:, 1], v_new=v[:, 1], qk_gain=gain)
    np.testing.assert_allclose(dec[0, 0], exp1, rtol=1e-12)
    out, _ = ref.attn_prefill_chunk(q[:, 1:], k[:, 1:], v[:, 1:], kc, vc, [1], -1, qk_gain=gain)
    np.testing.assert_allclose(out[0, 0, 0], exp1, rtol=1e-12)


def test_value_gate_by_linearity():
    """Attention is linear in v and the gate logit 0 gives the factor 1/2, so out(v, ve, g = 0) = out(v) + out(ve)/2;
    a gate logit of -60 leaves v as it is (factor ~1e-26), +60 adds ve in full."""
    q, k, v = (f64(t) for t in fwd_inputs(2, 40, 4, 2, 16, seed=6))
    ve = np.random.default_rng(1).standard_normal(v.shape)
    g0 = np.zeros(v.shape[:3])
    W = 7
    np.testing.assert_allclose(ref.attn_fwd(q, k, v, W, ve=ve, ve_gate=g0),
                               ref.attn_fwd(q, k, v, W) + 0.5 * ref.attn_fwd(q, k, ve, W), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ref.attn_fwd(q, k, v, W, ve=ve, ve_gate=g0 - 60), ref.attn_fwd(q, k, v, W), atol=1e-12)
    np.testing.assert_allclose(ref.attn_fwd(q, k, v, W, ve=ve, ve_gate=g0 + 60), ref.attn_fwd(q, k, v + ve, W),
                               atol=1e-12)


# ----------------------------------------------------------------------------------------------------------
# Attention: brute force on tiny inputs
# ----------------------------------------------------------------------------------------------------------

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("T", [1, 7, 64, 130])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_blocked_oracle_matches_brute_force(T, G):
    D = 8
    Hkv = 1 if T >= 64 else 2
    Hq = G * Hkv
    q = _rand((1, T, Hq, D), 10 + T)
    k = _rand((1, T, Hkv, D), 20 + T)
    v = _rand((1, T, Hkv, D), 30 + T)
    windows = sorted({-1, 0, 1, 5, 63, T - 1, T})
    if T >= 64:
        windows = [-1, 0, 5, 63]          # keep the scalar loops fast; small T covers the rest
    for W in windows:
        a = ref.attn_fwd(q, k, v, W, chunk=32)
        b = np.array(attn_fwd_brute(q, k, v, W))
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12, err_msg=f"T={T} G={G} W={W}")


def test_blocked_oracle_matches_brute_force_d128():
    q = _rand((1, 9, 4, 128), 1)
    k = _rand((1, 9, 2, 128), 2)
    v = _rand((1, 9, 2, 128), 3)
    for W in (-1, 3):
        np.testing.assert_allclose(ref.attn_fwd(q, k, v, W), np.array(attn_fwd_brute(q, k, v, W)),
                                   rtol=1e-11, atol=1e-12)


def test_rows_path_matches_full():
    q, k, v = (f64(t) for t in fwd_inputs(2, 300, 6, 2, 128, seed=7))
    for W in (-1, 100):
        full = ref.attn_fwd(q, k, v, W)
        rows = [(0, 0, 0), (1, 299, 5), (0, 150, 3), (1, 101, 2), (0, 128, 1)]
        got = ref.attn_fwd_rows(q, k, v, W, rows)
        for n, (b, i, h) in enumerate(rows):
            np.testing.assert_allclose(got[n], full[b, i, h], rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------------------------------------
# Attention: invariants
# ----------------------------------------------------------------------------------------------------------

def test_window_at_least_T_minus_1_is_full_causal():
    q, k, v = (f64(t) for t in fwd_inputs(1, 256, 4, 2, 128))
    full = ref.attn_fwd(q, k, v, -1)
    for W in (255, 256, 10000):
        np.testing.assert_array_equal(ref.attn_fwd(q, k, v, W), full)


def test_gqa_equals_mha_with_repeated_kv():
    """Contiguous grouping: query head h reads kv head h // G (catches h % G)."""
    q, k, v = (f64(t) for t in fwd_inputs(1, 96, 8, 2, 128, seed=3))
    G = 4
    kr = np.repeat(k, G, axis=2)
    vr = np.repeat(v, G, axis=2)
    for W in (-1, 17):
        np.testing.assert_allclose(ref.attn_fwd(q, k, v, W), ref.attn_fwd(q, kr, vr, W), rtol=0, atol=1e-15)
    # the other grouping (h % Hkv) gives a different answer
    kt = np.tile(k, (1, 1, G, 1))
    vt = np.tile(v, (1, 1, G, 1))
    assert np.max(np.abs(ref.attn_fwd(q, k, v, -1) - ref.attn_fwd(q, kt, vt, -1))) > 0.1


def test_position_zero_and_window_zero_return_v():
    q, k, v = (f64(t) for t in fwd_inputs(2, 64, 6, 3, 128, seed=4))
    out = ref.attn_fwd(q, k, v, -1)
    G = 2
    for h in range(6):
        np.testing.assert_array_equal(out[:, 0, h], v[:, 0, h // G])
    out0 = ref.attn_fwd(q, k, v, 0)
    for h in range(6):
        np.testing.assert_array_equal(out0[:, :, h], v[:, :, h // G])


@pytest.mark.parametrize("W", [-1, 10])
def test_causality_and_band(W):
    """Perturbing keys/values outside row i's band leaves row i bit-identical."""
    T = 80
    q, k, v = (f64(t) for t in fwd_inputs(1, T, 2, 1, 128, seed=5))
    base = ref.attn_fwd(q, k, v, W)
    i = 40
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1:] += 3.0
    v2[:, i + 1:] -= 5.0
    if W >= 0:
        k2[:, :i - W] *= -2.0
        v2[:, :i - W] += 7.0
    out = ref.attn_fwd(q, k2, v2, W)
    np.testing.assert_array_equal(out[:, i], base[:, i])
    # and perturbing inside the band does change it
    k3 = k.copy()
    k3[:, i] += 1.0
    assert np.max(np.abs(ref.attn_fwd(q, k3, v, W)[:, i] - base[:, i])) > 1e-4


def test_constant_values_give_constant_output():
    q, k, _ = (f64(t) for t in fwd_inputs(1, 100, 4, 2, 128, seed=6))
    c = np.random.default_rng(0).standard_normal(128)
    v = np.broadcast_to(c, (1, 100, 2, 128)).copy()
    for W in (-1, 7):
        out = ref.attn_fwd(q, k, v, W)
        np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=1e-12, atol=1e-12)


def test_scale_invariance_of_qk_norm():
    q, k, v = (f64(t) for t in fwd_inputs(1, 64, 2, 2, 128, seed=8))
    a = ref.attn_fwd(q, k, v, -1)
    b = ref.attn_fwd(3.0 * q, 0.5 * k, v, -1)
    assert np.max(np.abs(a - b)) < 1e-5


# ----------------------------------------------------------------------------------------------------------
# Decode
# ----------------------------------------------------------------------------------------------------------

def test_decode_matches_brute_force():
    d = decode_inputs(3, 4, 2, 8, 12, 0, 11, seed=9, with_new=True)
    cl = d["cache_lens"].numpy().copy()
    cl[0] = 0                      # empty cache
    args = [f64(d[n]) for n in ("q", "kcache", "vcache")]
    for W in (-1, 0, 3):
        for new in (False, True):
            kn = f64(d["k_new"]) if new else None
            vn = f64(d["v_new"]) if new else None
            a, _ = ref.attn_decode(*args, cl, W, kn, vn)
            b = np.array(attn_decode_brute(*args, cl, W, kn, vn))
            np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12, err_msg=f"W={W} new={new}")
            if not new:
                np.testing.assert_array_equal(a[0], 0.0)     # empty visible set -> zeros


def test_decode_equals_prefill_row():
    """Cache-vs-full self-consistency: decoding token p against a cache built from the prefill's roped+normed
    keys equals row p of the prefill."""
    B, T, Hq, Hkv, D = 2, 70, 6, 2, 128
    q, k, v = (f64(t) for t in fwd_inputs(B, T, Hq, Hkv, D, seed=11))
    pos = np.broadcast_to(np.arange(T), (B, T))
    kn = ref.qk_prologue(k, pos)
    for W in (-1, 9):
        full = ref.attn_fwd(q, k, v, W)
        for p in (0, 1, 37, 69):
            Tcap = T
            kc = np.zeros((B, Tcap, Hkv, D))
            vc = np.zeros((B, Tcap, Hkv, D))
            kc[:, :p] = kn[:, :p]
            vc[:, :p] = v[:, :p]
            lens = np.full(B, p)
            out, kn_new = ref.attn_decode(q[:, p], kc, vc, lens, W, k[:, p], v[:, p])
            np.testing.assert_allclose(out, full[:, p], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(kn_new, kn[:, p], rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------------------------------------
# Discriminators: the other readings would fail the GPU tolerance by a wide margin
# ----------------------------------------------------------------------------------------------------------

def _rope_variant(x, pos, kind, base=100000.0):
    D = x.shape[-1]
    th = base ** (-2.0 * np.arange(D // 2) / D)
    a = np.asarray(pos, dtype=np.float64)[..., None, None] * th
    c, s = np.cos(a), np.sin(a)
    if kind == "flipped_sign":
        x1, x2 = x[..., :D // 2], x[..., D // 2:]
        return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)
    if kind == "interleaved":
        x1, x2 = x[..., 0::2], x[..., 1::2]
        y = np.empty_like(x)
        y[..., 0::2] = x1 * c + x2 * s
        y[..., 1::2] = -x1 * s + x2 * c
        return y
    raise ValueError(kind)


def _dense_attn(qn, kn, v, W):
    B, T, Hq, D = qn.shape
    G = Hq // kn.shape[2]
    out = np.zeros_like(qn)
    ii, jj = np.arange(T)[:, None], np.arange(T)[None, :]
    mask = (jj <= ii) & ((W < 0) | (ii - jj <= W))
    for b in range(B):
        for h in range(Hq):
            s = qn[b, :, h] @ kn[b, :, h // G].T / math.sqrt(D)
            s = np.where(mask, s, -np.inf)
            p = np.exp(s - s.max(1, keepdims=True))
            out[b, :, h] = (p / p.sum(1, keepdims=True)) @ v[b, :, h // G]
    return out


@pytest.mark.parametrize("kind", ["flipped_sign", "interleaved"])
def test_rope_reading_discriminators(kind):
    w = TINY
    q, k, v = (f64(t) for t in fwd_inputs(w.B, w.T, w.Hq, w.Hkv, w.D))
    pos = np.broadcast_to(np.arange(w.T), (w.B, w.T))
    chosen = ref.attn_fwd(q, k, v, 128)
    alt = _dense_attn(ref.rms_norm(_rope_variant(q, pos, kind)), ref.rms_norm(_rope_variant(k, pos, kind)), v, 128)
    # sanity: the local dense attention reproduces the oracle with the chosen rope
    same = _dense_attn(ref.qk_prologue(q, pos), ref.qk_prologue(k, pos), v, 128)
    np.testing.assert_allclose(same, chosen, atol=1e-12)
    assert np.max(np.abs(alt - chosen)) > 10 * GPU_MAX_ABS
