"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded bf16 inputs.

Tolerance: max-abs 2e-2 and mean-abs 2e-3 on bf16 outputs.  Every case, the full-size workloads included, is
compared element by element in full, plus properties that hold at any size.
"""

import numpy as np
import pytest
import torch

from oracle import ref
from seeded_inputs import DECODE, DEPTH12, GQA, LONG, TINY, decode_inputs, fwd_inputs
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
    return [t.cuda() if t is not None else None for t in ts]


# ------------------------------------------------------------------------------------------------ prologue

def test_prologue_matches_oracle_and_has_unit_rms(nc):
    q, k, _ = fwd_inputs(2, 300, 6, 2, 128, seed=1)
    qd, kd = cuda(q, k)
    qn, kn = nc.nc_attn_qk_prologue(qd, kd)
    torch.cuda.synchronize()
    pos = np.broadcast_to(np.arange(300), (2, 300))
    for got, x in ((qn, q), (kn, k)):
        r = ref.qk_prologue(f64(x), pos)
        g = f64(got)
        # bf16 rounding of a value of size |r| costs at most 2^-9 |r|; allow 2^-8 |r| + 1e-3
        assert np.all(np.abs(g - r) <= np.abs(r) * 2.0 ** -8 + 1e-3)
        rms = np.sqrt(np.mean(g * g, axis=-1))
        assert np.max(np.abs(rms - 1.0)) < 2.0 ** -8


def test_prologue_rotation_is_accurate_at_large_positions(nc):
    """Positions up to 2^16 - 1 (angles up to 6.6e4 rad on the fastest pair): every element of qn and kn lies within
    one bf16 ulp of the exact fp64 value, plus 2^-17 for the values near zero, where the absolute error of the
    rotation (below 1e-6) can exceed an ulp.  A wrong angle reduction at large positions shows up as errors ~1e-2."""
    T = 1 << 16
    q, k, _ = fwd_inputs(1, T, 2, 1, 128, seed=7)
    qn, kn = nc.nc_attn_qk_prologue(*cuda(q, k))
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(T - 2048, T), rng.integers(0, T, 2048)]))
    for got, x in ((qn, q), (kn, k)):
        r = ref.qk_prologue(f64(x)[:, rows], rows[None, :])
        g = f64(got)[:, rows]
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
        err = np.abs(g - r) - ulp
        assert err.max() <= 2.0 ** -17, f"worst excess over one ulp {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"


def test_prologue_rotation_is_accurate_up_to_position_2_24(nc):
    """The largest positions the kernels take (T < 2^24), where the angle of the fastest pair exceeds 1.3e7 rad and
    its fp32 reduction needs the extra quarter turn: 4096 sampled rows of a (2^24 - 1)-token sequence (the other rows
    zero) carry seeded inputs, and each transformed row lies within one bf16 ulp of the fp64 oracle (plus 2^-17 near
    zero)."""
    T = (1 << 24) - 1
    rng = np.random.default_rng(24)
    rows = np.unique(np.concatenate([np.arange(T - 1024, T), rng.integers(1 << 23, T, 2048), rng.integers(0, T, 1024)]))
    qs, ks, _ = fwd_inputs(1, len(rows), 1, 1, 128, seed=24)
    dev = torch.device("cuda")
    idx = torch.from_numpy(rows).to(dev)
    qd = torch.zeros((1, T, 1, 128), dtype=torch.bfloat16, device=dev)
    kd = torch.zeros_like(qd)
    qd[0, idx] = qs[0].to(dev)
    kd[0, idx] = ks[0].to(dev)
    qn, kn = nc.nc_attn_qk_prologue(qd, kd)
    torch.cuda.synchronize()
    for got, x in ((qn, qs), (kn, ks)):
        r = ref.qk_prologue(f64(x), rows[None, :])
        g = f64(got[0, idx].cpu()[None])
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
        err = np.abs(g - r) - ulp
        assert err.max() <= 2.0 ** -17, f"worst excess over one ulp {err.max():.3e}"
    del qd, kd, qn, kn
    torch.cuda.empty_cache()


# ------------------------------------------------------------------------------------------------ prefill

@pytest.mark.parametrize("W", TINY.windows)
def test_fwd_tiny_config(nc, W):
    w = TINY
    q, k, v = fwd_inputs(w.B, w.T, w.Hq, w.Hkv, w.D, seed=0)
    out = nc.nc_attn_fwd(*cuda(q, k, v), window=W)
    assert_close(out, ref.attn_fwd(f64(q), f64(k), f64(v), W), f"tiny W={W}")


ODD = [  # (B, T, Hq, Hkv, W): T not a multiple of the tile, ragged tails, every group size the kernel packs
    (1, 1, 1, 1, -1),
    (2, 7, 2, 1, -1),
    (1, 130, 3, 1, 5),
    (2, 300, 8, 2, 127),
    (1, 257, 12, 4, 0),
    (1, 200, 6, 6, 1),
    (1, 384, 16, 4, 200),
    (1, 129, 5, 1, 64),
    (2, 160, 4, 4, 128),
    (1, 65, 32, 1, -1),
    (1, 700, 2, 2, 300),
    (1, 33, 128, 1, -1),     # largest group: one position per tile
    (1, 70, 64, 1, 20),
    (2, 77, 10, 2, 30),      # group of 5: 125 of the 128 tile rows in use
]


@pytest.mark.parametrize("B,T,Hq,Hkv,W", ODD)
def test_fwd_odd_shapes(nc, B, T, Hq, Hkv, W):
    q, k, v = fwd_inputs(B, T, Hq, Hkv, 128, seed=T + Hq)
    out = nc.nc_attn_fwd(*cuda(q, k, v), window=W)
    assert_close(out, ref.attn_fwd(f64(q), f64(k), f64(v), W), f"B{B} T{T} Hq{Hq} Hkv{Hkv} W{W}")


# Single-tile items (too few pairs to give every SM an item) run their key tiles as two chains whose partial sums the
# epilogue adds.  With G = 1 (128 positions per Q tile) and one sequence, Q tile m of a T = 640 layer has m + 1 key
# tiles under a causal mask: 1 to 5 rounds, i.e. chain B empty, one tile each, A one tile longer than B; the windows put
# a band edge in the first chain's tiles, in the second's, or in both.
SPLIT = [(1, 640, 1, 1, W) for W in (-1, 0, 100, 200, 300, 511)] + [(1, 600, 2, 2, 250), (1, 1000, 3, 3, -1)]


@pytest.mark.parametrize("B,T,Hq,Hkv,W", SPLIT)
def test_fwd_split_items(nc, B, T, Hq, Hkv, W):
    q, k, v = fwd_inputs(B, T, Hq, Hkv, 128, seed=3 * T + W)
    out = nc.nc_attn_fwd(*cuda(q, k, v), window=W)
    assert_close(out, ref.attn_fwd(f64(q), f64(k), f64(v), W), f"split items B{B} T{T} Hq{Hq} Hkv{Hkv} W{W}")


def assert_close_rows(got, exp, what):
    """Element-wise comparison of a whole [B, T, H, D] output; names the worst (b, t, h) row on failure."""
    g = f64(got)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    d = np.abs(g - exp)
    worst = np.unravel_index(int(np.argmax(d)), d.shape)[:3]
    mx, mn = float(d.max()), float(d.mean())
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (
        f"{what}: max-abs {mx:.3e} (<= {MAX_ABS}) at row (b, t, h) = {tuple(int(x) for x in worst)}, "
        f"mean-abs {mn:.3e} (<= {MEAN_ABS})")
    return mx, mn


# Every output element of the full-size prefill workloads against the oracle, on the inputs the bench times: call i of
# a workload's window list draws its q, k, v from seed i (the depth-12 SSSL step's four layers, both windows of the
# GQA and long-context workloads).
FULL = [(DEPTH12, li, W) for li, W in enumerate(DEPTH12.windows)] + \
       [(GQA, li, W) for li, W in enumerate(GQA.windows)] + [(LONG, li, W) for li, W in enumerate(LONG.windows)]


@pytest.mark.parametrize("wl,seed,W", FULL, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_fwd_full_size_every_element(nc, wl, seed, W):
    q, k, v = fwd_inputs(wl.B, wl.T, wl.Hq, wl.Hkv, wl.D, seed=seed)
    out = nc.nc_attn_fwd(*cuda(q, k, v), window=W)
    torch.cuda.synchronize()
    exp = ref.attn_fwd(f64(q), f64(k), f64(v), W)
    assert_close_rows(out, exp, f"{wl.name} seed={seed} W={W}")
    # position 0 sees only itself: the output is v_0 of the group's kv head
    G = wl.Hq // wl.Hkv
    o0, v0 = f64(out[:, 0]), f64(v[:, 0])
    for h in range(wl.Hq):
        assert np.max(np.abs(o0[:, h] - v0[:, h // G])) < 1e-6


def test_window_at_least_T_minus_1_equals_full_causal(nc):
    q, k, v = cuda(*fwd_inputs(2, 515, 6, 2, 128, seed=5))
    full = nc.nc_attn_fwd(q, k, v, window=-1).clone()
    for W in (514, 515, 100000):
        assert torch.equal(nc.nc_attn_fwd(q, k, v, window=W), full)


def test_gqa_equals_mha_with_repeated_kv(nc):
    q, k, v = fwd_inputs(1, 333, 8, 2, 128, seed=6)
    qd, kd, vd = cuda(q, k, v)
    a = nc.nc_attn_fwd(qd, kd, vd, window=50).clone()
    b = nc.nc_attn_fwd(qd, kd.repeat_interleave(4, dim=2).contiguous(), vd.repeat_interleave(4, dim=2).contiguous(),
                       window=50)
    assert_close(a, f64(b), "GQA vs repeated-KV MHA (GPU vs GPU)")


@pytest.mark.parametrize("W", [-1, 40])
def test_causality_and_band_on_gpu(nc, W):
    q, k, v = fwd_inputs(1, 400, 4, 2, 128, seed=7)
    qd, kd, vd = cuda(q, k, v)
    base = nc.nc_attn_fwd(qd, kd, vd, window=W).clone()
    i = 200
    k2, v2 = kd.clone(), vd.clone()
    k2[:, i + 1:] *= -3
    v2[:, i + 1:] += 5
    if W >= 0:
        k2[:, :i - W] *= 2
        v2[:, :i - W] -= 7
    out = nc.nc_attn_fwd(qd, k2, v2, window=W)
    assert torch.equal(out[:, i], base[:, i])


# ------------------------------------------------------------------------------------------------ decode

def decode_case(nc, B, Hq, Hkv, Tcap, lens, W, with_new, seed):
    d = decode_inputs(B, Hq, Hkv, 128, Tcap, 1, 2, seed=seed, with_new=with_new)
    lens = torch.tensor(lens, dtype=torch.int32)
    kc, vc = d["kcache"].clone(), d["vcache"].clone()
    q, kn, vn = d["q"], d["k_new"], d["v_new"]
    exp, kn_ref = ref.attn_decode(f64(q), f64(kc), f64(vc), lens.numpy(), W,
                                  f64(kn) if with_new else None, f64(vn) if with_new else None)
    kcd, vcd = cuda(kc, vc)
    out = nc.nc_attn_decode(*cuda(q), kcd, vcd, lens.cuda(), k_new=kn.cuda() if with_new else None,
                            v_new=vn.cuda() if with_new else None, window=W)
    torch.cuda.synchronize()
    return out, exp, kcd, vcd, kn_ref, d, lens


@pytest.mark.parametrize("W", [-1, 0, 5, 128, 2048])
@pytest.mark.parametrize("with_new", [False, True])
def test_decode_small(nc, W, with_new):
    lens = [0, 1, 127, 128, 129, 255, 256, 298]
    out, exp, kcd, vcd, kn_ref, d, lens_t = decode_case(nc, len(lens), 12, 4, 300, lens, W, with_new, seed=3)
    assert_close(out, exp, f"decode W={W} new={with_new}")
    if with_new:
        for b, p in enumerate(lens):
            g = f64(kcd[b, p])
            assert np.all(np.abs(g - kn_ref[b]) <= np.abs(kn_ref[b]) * 2.0 ** -8 + 1e-3)
            assert torch.equal(vcd[b, p].cpu(), d["v_new"][b])
    else:
        assert torch.count_nonzero(out[0]) == 0       # empty visible set


@pytest.mark.parametrize("G", [1, 2, 3, 8, 12, 16])
def test_decode_group_sizes(nc, G):
    lens = [3, 500, 1000]
    out, exp, *_ = decode_case(nc, 3, 2 * G, 2, 1024, lens, 300, True, seed=G)
    assert_close(out, exp, f"decode G={G}")


@pytest.mark.parametrize("W", [-1, 700])
@pytest.mark.parametrize("with_new", [False, True])
def test_decode_many_sequences_mixed_lengths(nc, W, with_new):
    """Hundreds of (sequence, kv head) segments of every length, so that CTA ranges start and end inside segments,
    some segments span several CTAs and some CTAs hold many short segments."""
    rng = np.random.default_rng(11)
    B, Tcap = 300, 2100
    lens = rng.integers(0, Tcap, size=B)
    lens[:8] = [0, 1, 127, 128, 129, 2099, 256, 0]
    out, exp, *_ = decode_case(nc, B, 8, 2, Tcap, lens.tolist(), W, with_new, seed=21)
    assert_close(out, exp, f"decode mixed lengths W={W} new={with_new}")


@pytest.mark.parametrize("L", [129, 5000, 19999])
def test_decode_one_long_sequence_split_over_ctas(nc, L):
    """One segment cut into many CTA ranges (up to one tile each): many partials merged by the last CTA."""
    out, exp, *_ = decode_case(nc, 1, 4, 1, 20000, [L], -1, True, seed=L)
    assert_close(out, exp, f"decode one sequence L={L}")


def test_decode_ignores_garbage_past_the_cache_length(nc):
    """Cache rows at and after cache_lens[b] may hold anything (here NaN): they must not reach the output."""
    B, Hq, Hkv, Tcap = 4, 6, 2, 400
    lens = [1, 100, 130, 300]
    d = decode_inputs(B, Hq, Hkv, 128, Tcap, 1, 2, seed=8)
    kc, vc = d["kcache"].clone(), d["vcache"].clone()
    for b, p in enumerate(lens):
        kc[b, p:] = float("nan")
        vc[b, p:] = float("nan")
    lt = torch.tensor(lens, dtype=torch.int32)
    exp, _ = ref.attn_decode(f64(d["q"]), f64(d["kcache"]), f64(d["vcache"]), lt.numpy(), -1)
    out = nc.nc_attn_decode(*cuda(d["q"], kc, vc), lt.cuda(), window=-1)
    assert_close(out, exp, "decode with NaN past the cache length")


def test_decode_full_config(nc):
    w = DECODE
    for with_new in (False, True):
        d = decode_inputs(w.B, w.Hq, w.Hkv, w.D, w.Tcap, w.len_lo, w.len_hi, seed=0, with_new=with_new)
        lens = d["cache_lens"]
        exp, _ = ref.attn_decode(f64(d["q"]), d["kcache"].float().numpy(), d["vcache"].float().numpy(),
                                 lens.numpy(), w.window, f64(d["k_new"]) if with_new else None,
                                 f64(d["v_new"]) if with_new else None)
        kc, vc = cuda(d["kcache"], d["vcache"])
        out = nc.nc_attn_decode(d["q"].cuda(), kc, vc, lens.cuda(),
                                k_new=d["k_new"].cuda() if with_new else None,
                                v_new=d["v_new"].cuda() if with_new else None, window=w.window)
        assert_close(out, exp, f"decode full config new={with_new}")
        # a second call on the same workspace gives the same result (the counters were left at zero)
        out2 = nc.nc_attn_decode(d["q"].cuda(), kc, vc, lens.cuda(),
                                 k_new=d["k_new"].cuda() if with_new else None,
                                 v_new=d["v_new"].cuda() if with_new else None, window=w.window)
        assert torch.equal(out, out2)


@pytest.mark.parametrize("W", [-1, 33])
def test_decode_equals_prefill_row_on_gpu(nc, W):
    """Cache-vs-full self-consistency between the two GPU kernels: decode of token p against a cache holding the
    prologue's kn[0:p] and v[0:p] (plus k[p], v[p] as the new key/value) equals prefill row p."""
    B, T, Hq, Hkv = 2, 300, 6, 2
    q, k, v = cuda(*fwd_inputs(B, T, Hq, Hkv, 128, seed=9))
    full = nc.nc_attn_fwd(q, k, v, window=W)
    _, kn = nc.nc_attn_qk_prologue(q, k)
    for p in (0, 1, 150, 299):
        kc = torch.zeros(B, T, Hkv, 128, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        kc[:, :p] = kn[:, :p]
        vc[:, :p] = v[:, :p]
        lens = torch.full((B,), p, dtype=torch.int32, device="cuda")
        out = nc.nc_attn_decode(q[:, p].contiguous(), kc, vc, lens, k_new=k[:, p].contiguous(),
                                v_new=v[:, p].contiguous(), window=W)
        assert_close(out, f64(full[:, p]), f"decode vs prefill row p={p} W={W}")
        assert torch.equal(kc[:, p], kn[:, p])    # the new key is written exactly as the prologue computes it


def test_decode_workspace_reused_across_shapes(nc):
    """One workspace, calls with different (B, Hkv): a small call leaves split partials where a larger call's
    arrival counters go.  The caller-side contract (zero the workspace when B*Hkv changes) and the binding's cached
    workspace both keep the results exact."""
    shapes = [(3, 4, 2, 300, [5, 200, 299]), (9, 12, 4, 300, [1, 50, 130, 260, 299, 7, 140, 256, 280]),
              (2, 8, 1, 300, [299, 180])]
    for B, Hq, Hkv, Tcap, lens in shapes * 2:
        out, exp, *_ = decode_case(nc, B, Hq, Hkv, Tcap, lens, -1, False, seed=B)
        assert_close(out, exp, f"decode B={B} Hkv={Hkv} after other shapes")
    nbytes = max(nc.nc_attn_decode_workspace_bytes(B, Hq, Hkv, 128, Tcap, -1) for B, Hq, Hkv, Tcap, _ in shapes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    prev = None
    for B, Hq, Hkv, Tcap, lens in shapes * 2:
        if prev is not None and prev != B * Hkv:
            ws.zero_()
        prev = B * Hkv
        d = decode_inputs(B, Hq, Hkv, 128, Tcap, 1, 2, seed=B)
        lt = torch.tensor(lens, dtype=torch.int32)
        exp, _ = ref.attn_decode(f64(d["q"]), f64(d["kcache"]), f64(d["vcache"]), lt.numpy(), -1)
        out = nc.nc_attn_decode(*cuda(d["q"], d["kcache"], d["vcache"]), lt.cuda(), window=-1, workspace=ws)
        assert_close(out, exp, f"decode caller workspace B={B} Hkv={Hkv}")
        # the entry point without a workspace argument (library-held buffer), through the raw C ABI
        import ctypes
        qd, kd, vd, ld = cuda(d["q"], d["kcache"], d["vcache"], lt)
        out2 = torch.empty_like(qd)
        p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        st = nc.lib.nc_attn_decode(p(qd), p(kd), p(vd), p(ld), p(out2), None, None, B, Hq, Hkv, 128, Tcap, -1,
                                   1e5, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == nc.NC_OK
        assert_close(out2, exp, f"decode library workspace B={B} Hkv={Hkv}")


def test_decode_bad_cache_length_sets_status_and_zero_row(nc):
    d = decode_inputs(3, 4, 2, 128, 64, 1, 60, seed=4, with_new=True)
    lens = torch.tensor([10, 64, -1], dtype=torch.int32)   # 64 = Tcap: no room for the new key
    kc, vc = cuda(d["kcache"], d["vcache"])
    out = nc.nc_attn_decode(d["q"].cuda(), kc, vc, lens.cuda(), k_new=d["k_new"].cuda(), v_new=d["v_new"].cuda(),
                            window=-1)
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_ERR_DEVICE_BAD_INPUT
    assert torch.count_nonzero(out[1:]) == 0
    exp, _ = ref.attn_decode(f64(d["q"][:1]), f64(d["kcache"][:1]), f64(d["vcache"][:1]), lens[:1].numpy(), -1,
                             f64(d["k_new"][:1]), f64(d["v_new"][:1]))
    assert_close(out[:1], exp, "valid row next to invalid ones")
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_OK


# ------------------------------------------------------------------------------------------------ bounded waits

def test_bounded_wait_times_out_and_context_survives(nc):
    nc.nc_attn_selftest_wait_timeout(2000)       # 2 ms limit on a barrier nothing completes
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_ERR_DEVICE_TIMEOUT
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_OK
    q, k, v = fwd_inputs(1, 64, 2, 1, 128, seed=1)
    out = nc.nc_attn_fwd(*cuda(q, k, v))
    assert_close(out, ref.attn_fwd(f64(q), f64(k), f64(v), -1), "after the timeout self-test")
