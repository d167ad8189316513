"""Pins for the chunked-prefill oracle (CPU only).

``oracle.ref.attn_prefill_chunk`` is tied to the prefill and decode oracles, which are themselves pinned by brute
force and closed forms: a chunk with an empty cache is the prefill of the chunk; the second chunk of a sequence
split in two, against the first chunk's normed keys, is the tail of the whole sequence's prefill; a one-token chunk
is a decode step with a new key.  A slip in the chunk's positions (an offset dropped or added twice), its mask, its
key order or its cache handling breaks one of them.
"""

import numpy as np
import pytest
import torch

from oracle import ref
from seeded_inputs import chunk_inputs, fwd_inputs


def f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("W", [-1, 0, 3, 40])
def test_empty_cache_is_the_prefill_of_the_chunk(W):
    q, k, v = (f64(t) for t in fwd_inputs(2, 37, 4, 2, 128, seed=3))
    kc = np.full((2, 50, 2, 128), np.nan)   # never read: p_b = 0
    out, kn = ref.attn_prefill_chunk(q, k, v, kc, kc, [0, 0], W)
    np.testing.assert_allclose(out, ref.attn_fwd(q, k, v, W), rtol=0, atol=1e-12)
    pos = np.broadcast_to(np.arange(37), (2, 37))
    np.testing.assert_allclose(kn, ref.qk_prologue(k, pos), rtol=0, atol=1e-15)


@pytest.mark.parametrize("W", [-1, 5, 64, 200])
@pytest.mark.parametrize("T1", [1, 29, 64])
def test_second_chunk_is_the_tail_of_the_whole_prefill(W, T1):
    B, T, Hq, Hkv = 2, 90, 6, 2
    q, k, v = (f64(t) for t in fwd_inputs(B, T, Hq, Hkv, 128, seed=11))
    full = ref.attn_fwd(q, k, v, W)
    Tcap = 100
    kc = np.full((B, Tcap, Hkv, 128), np.nan)
    vc = np.full((B, Tcap, Hkv, 128), np.nan)
    kc[:, :T1] = ref.qk_prologue(k[:, :T1], np.broadcast_to(np.arange(T1), (B, T1)))
    vc[:, :T1] = v[:, :T1]
    out, _ = ref.attn_prefill_chunk(q[:, T1:], k[:, T1:], v[:, T1:], kc, vc, [T1, T1], W)
    np.testing.assert_allclose(out, full[:, T1:], rtol=0, atol=1e-12)


def test_sequences_at_different_offsets():
    """Each sequence's chunk is the tail of its own prefill, whatever the other sequences' offsets."""
    B, T, Hq, Hkv, W = 3, 60, 4, 4, 17
    q, k, v = (f64(t) for t in fwd_inputs(B, T, Hq, Hkv, 128, seed=5))
    full = ref.attn_fwd(q, k, v, W)
    p = [0, 13, 40]
    Tq = 20
    Tcap = 64
    kc = np.full((B, Tcap, Hkv, 128), np.nan)
    vc = np.full((B, Tcap, Hkv, 128), np.nan)
    qs, ks, vs = (np.zeros((B, Tq) + x.shape[2:]) for x in (q, k, v))
    for b in range(B):
        kc[b, :p[b]] = ref.qk_prologue(k[b:b + 1, :p[b]], np.arange(p[b])[None])[0]
        vc[b, :p[b]] = v[b, :p[b]]
        qs[b], ks[b], vs[b] = q[b, p[b]:p[b] + Tq], k[b, p[b]:p[b] + Tq], v[b, p[b]:p[b] + Tq]
    out, _ = ref.attn_prefill_chunk(qs, ks, vs, kc, vc, p, W)
    for b in range(B):
        np.testing.assert_allclose(out[b], full[b, p[b]:p[b] + Tq], rtol=0, atol=1e-12)


@pytest.mark.parametrize("W", [-1, 2, 30])
def test_one_token_chunk_is_a_decode_step(W):
    d = chunk_inputs(3, 1, 6, 3, 128, 40, seed=2)
    kc, vc, q, kn, vn = (f64(d[x]) for x in ("kcache", "vcache", "q", "k_new", "v_new"))
    lens = [0, 7, 39]
    out, kn_new = ref.attn_prefill_chunk(q, kn, vn, kc, vc, lens, W)
    dec, dec_kn = ref.attn_decode(q[:, 0], kc, vc, np.array(lens), W, k_new=kn[:, 0], v_new=vn[:, 0])
    np.testing.assert_allclose(out[:, 0], dec, rtol=0, atol=1e-12)
    np.testing.assert_allclose(kn_new[:, 0], dec_kn, rtol=0, atol=1e-15)


def test_out_of_range_cache_length_gives_zero_rows():
    d = chunk_inputs(3, 8, 4, 2, 128, 20, seed=4)
    kc, vc, q, kn, vn = (f64(d[x]) for x in ("kcache", "vcache", "q", "k_new", "v_new"))
    out, kn_new = ref.attn_prefill_chunk(q, kn, vn, kc, vc, [-1, 12, 13], -1)   # 12 + 8 = Tcap is the last valid
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.all(kn_new[2] == 0)
    assert np.isfinite(out[1]).all() and np.abs(out[1]).max() > 0


@pytest.mark.parametrize("W", [-1, 7])
def test_value_embedding_chunk_and_decode_agree_with_the_prefill(W):
    """The gated value embedding on the cache paths: a chunk against an empty cache is the prefill with the same
    embedding, and a one-token chunk is a decode step whose new value carries it."""
    B, T, Hq, Hkv = 2, 23, 4, 2
    q, k, v = (f64(t) for t in fwd_inputs(B, T, Hq, Hkv, 128, seed=17))
    rng = np.random.default_rng(5)
    ve = rng.standard_normal((B, T, Hkv, 128))
    gate = rng.standard_normal((B, T, Hkv)) * 2
    kc = np.full((B, 40, Hkv, 128), np.nan)
    out, _ = ref.attn_prefill_chunk(q, k, v, kc, kc, [0, 0], W, ve_new=ve, ve_gate_new=gate)
    np.testing.assert_allclose(out, ref.attn_fwd(q, k, v, W, ve=ve, ve_gate=gate), rtol=0, atol=1e-12)
    # one token at position p against a cache of the prefill's normed keys and mixed values
    p = 11
    pos = np.broadcast_to(np.arange(T), (B, T))
    kn = ref.qk_prologue(k, pos)
    vmix = ref.value_mix(v, ve, gate)
    kc2 = np.zeros((B, 40, Hkv, 128))
    vc2 = np.zeros((B, 40, Hkv, 128))
    kc2[:, :p], vc2[:, :p] = kn[:, :p], vmix[:, :p]
    full = ref.attn_fwd(q, k, v, W, ve=ve, ve_gate=gate)
    one, _ = ref.attn_prefill_chunk(q[:, p:p + 1], k[:, p:p + 1], v[:, p:p + 1], kc2, vc2, [p, p], W,
                                    ve_new=ve[:, p:p + 1], ve_gate_new=gate[:, p:p + 1])
    dec, _ = ref.attn_decode(q[:, p], kc2, vc2, np.array([p, p]), W, k[:, p], v[:, p], ve_new=ve[:, p],
                             ve_gate_new=gate[:, p])
    np.testing.assert_allclose(one[:, 0], full[:, p], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dec, full[:, p], rtol=0, atol=1e-12)
