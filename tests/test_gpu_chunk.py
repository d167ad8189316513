"""GPU parity of the chunked prefill against a KV cache (through the C ABI) with the fp64 oracle.

Same tolerance as the other GPU parity tests (max-abs 2e-2, mean-abs 2e-3 on bf16 outputs).  Small cases are
compared element by element, including the cache rows the call appends and the rows it must leave alone; the
full-size chunk workload is compared in full as well.  Edge cases: one-token chunks, a chunk that fills the
cache exactly, a chunk ending on a tile boundary, window 0, a group of 16 heads, garbage (NaN) in the cache rows past
the chunk, out-of-range cache lengths, and agreement with the plain prefill when a sequence arrives in two chunks.
"""

import numpy as np
import pytest
import torch

from oracle import ref
from seeded_inputs import CHUNK, chunk_inputs, fwd_inputs
from tests.parity import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_attention_06_b300 import nc_attn
    nc_attn.nc_attn_get_device_status(clear=True)
    yield nc_attn
    assert nc_attn.nc_attn_get_device_status(clear=True) == nc_attn.NC_OK


def run_chunk(nc, d, lens, W):
    """One call on device copies of the inputs; returns (out, kcache, vcache) after the call."""
    kc, vc = d["kcache"].cuda(), d["vcache"].cuda()
    q, kn, vn = d["q"].cuda(), d["k_new"].cuda(), d["v_new"].cuda()
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = nc.nc_attn_prefill_chunk(q, kn, vn, kc, vc, lt, window=W)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle(d, lens, W):
    return ref.attn_prefill_chunk(*(f64(d[x]) for x in ("q", "k_new", "v_new", "kcache", "vcache")), lens, W)


# (B, Tq, Hq, Hkv, Tcap, cache lengths, window)
CASES = [
    (2, 130, 6, 2, 700, [0, 300], -1),
    (2, 130, 6, 2, 700, [0, 300], 100),
    (3, 1, 8, 8, 300, [5, 128, 255], -1),       # one-token chunks
    (1, 300, 12, 4, 2048, [1500], 1024),
    (2, 257, 4, 4, 600, [343, 0], 0),           # 343 + 257 = Tcap: the chunk fills the cache; window 0
    (2, 200, 16, 1, 520, [320, 77], 63),        # group of 16 heads (P = 8 positions per tile)
    (1, 64, 3, 1, 192, [128], -1),              # the chunk ends on a key-tile boundary
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}_Tq{c[1]}_Hq{c[2]}_Hkv{c[3]}_p{c[5]}_W{c[6]}")
def test_chunk_matches_oracle(nc, case):
    B, Tq, Hq, Hkv, Tcap, lens, W = case
    d = chunk_inputs(B, Tq, Hq, Hkv, 128, Tcap, seed=7 * B + Tq)
    exp, kn_exp = oracle(d, lens, W)
    out, kc, vc = run_chunk(nc, d, lens, W)
    assert_close(out, exp, f"chunk {case}")
    kc, vc = kc.cpu(), vc.cpu()
    for b, p in enumerate(lens):
        # the chunk's normed keys and its values are appended in place; every other cache row is left as it was
        assert_close(kc[b, p:p + Tq], kn_exp[b], f"appended keys b={b}")
        assert torch.equal(vc[b, p:p + Tq], d["v_new"][b])
        for c, src in ((kc, d["kcache"]), (vc, d["vcache"])):
            assert torch.equal(c[b, :p], src[b, :p]) and torch.equal(c[b, p + Tq:], src[b, p + Tq:])


def test_chunk_ignores_garbage_past_the_chunk(nc):
    B, Tq, Hq, Hkv, Tcap = 2, 100, 4, 2, 512
    lens = [70, 200]                            # the chunks end inside key tiles 1 and 2
    d = chunk_inputs(B, Tq, Hq, Hkv, 128, Tcap, seed=3)
    clean, _, _ = run_chunk(nc, d, lens, -1)
    for b, p in enumerate(lens):
        d["kcache"][b, p + Tq:] = float("nan")
        d["vcache"][b, p + Tq:] = float("nan")
    dirty, _, _ = run_chunk(nc, d, lens, -1)
    assert torch.isfinite(dirty).all()
    assert torch.equal(dirty, clean)


@pytest.mark.parametrize("W", [-1, 200])
def test_two_chunks_equal_one_prefill(nc, W):
    """A sequence prefilled in two chunks against an initially empty cache gives the plain prefill's rows, and
    leaves in the cache exactly the keys the prologue computes."""
    B, T, Hq, Hkv, T1, Tcap = 2, 700, 6, 2, 333, 768
    q, k, v = (t.cuda() for t in fwd_inputs(B, T, Hq, Hkv, 128, seed=21))
    full = nc.nc_attn_fwd(q, k, v, window=W)
    kc = torch.zeros(B, Tcap, Hkv, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    lens0 = torch.zeros(B, dtype=torch.int32, device="cuda")
    lens1 = torch.full((B,), T1, dtype=torch.int32, device="cuda")
    o1 = nc.nc_attn_prefill_chunk(q[:, :T1].contiguous(), k[:, :T1].contiguous(), v[:, :T1].contiguous(), kc, vc,
                                  lens0, window=W)
    o2 = nc.nc_attn_prefill_chunk(q[:, T1:].contiguous(), k[:, T1:].contiguous(), v[:, T1:].contiguous(), kc, vc,
                                  lens1, window=W)
    assert_close(torch.cat([o1, o2], dim=1), f64(full), f"two chunks vs one prefill W={W}")
    _, kn = nc.nc_attn_qk_prologue(q, k)
    assert torch.equal(kc[:, :T], kn)
    assert torch.equal(vc[:, :T], v)


def test_chunk_bad_cache_length_sets_status_and_zero_rows(nc):
    B, Tq, Hq, Hkv, Tcap = 3, 40, 4, 2, 100
    lens = [-3, 60, 61]                         # 60 + 40 = Tcap is the last valid length
    d = chunk_inputs(B, Tq, Hq, Hkv, 128, Tcap, seed=8)
    out, kc, vc = run_chunk(nc, d, lens, -1)
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_ERR_DEVICE_BAD_INPUT
    out, kc, vc = out.cpu(), kc.cpu(), vc.cpu()
    for b in (0, 2):
        assert torch.all(out[b] == 0)
        assert torch.equal(kc[b], d["kcache"][b]) and torch.equal(vc[b], d["vcache"][b])
    exp, _ = oracle(d, lens, -1)
    assert_close(out[1], exp[1], "valid sequence beside invalid ones")
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_OK


@pytest.mark.parametrize("W", CHUNK.windows)
def test_chunk_full_size(nc, W):
    """The chunk workload (B=4, Tq=512 appended at 1536 to a 2048-row cache) in the launch configuration the
    bench times; every sequence against the oracle in full, outputs and appended keys."""
    w = CHUNK
    d = chunk_inputs(w.B, w.Tq, w.Hq, w.Hkv, w.D, w.Tcap, seed=0)
    lens = [w.p0] * w.B
    out, kc, vc = run_chunk(nc, d, lens, W)
    exp, kn_exp = oracle(d, lens, W)
    assert_close(out, exp, f"chunk workload W={W}")
    assert_close(kc[:, w.p0:w.p0 + w.Tq], kn_exp, f"chunk workload appended keys W={W}")
    assert torch.equal(vc[:, w.p0:w.p0 + w.Tq].cpu(), d["v_new"])
