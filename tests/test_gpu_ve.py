"""GPU parity of the gated value embedding (v' = v + sigmoid(g) ve, formed in fp32 and rounded to bf16 once) on the
prefill, the chunked prefill and the decode step against the fp64 oracle, same tolerance as the other parity tests."""

import pytest
import torch

from oracle import ref
from seeded_inputs import fwd_inputs
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


@pytest.mark.parametrize("B,T,Hq,Hkv,W,gain", [(2, 300, 6, 2, 127, 1.0), (1, 520, 8, 8, -1, 1.2), (1, 77, 12, 4, 0, 1.0)])
def test_fwd_value_embedding(nc, B, T, Hq, Hkv, W, gain):
    q, k, v = fwd_inputs(B, T, Hq, Hkv, 128, seed=B + T)
    g = torch.Generator("cpu").manual_seed(T)
    ve = torch.randn(v.shape, generator=g).to(torch.bfloat16)
    gate = (2 * torch.randn(v.shape[:3], generator=g)).to(torch.bfloat16)
    out = nc.nc_attn_fwd(q.cuda(), k.cuda(), v.cuda(), window=W, qk_gain=gain, ve=ve.cuda(), ve_gate=gate.cuda())
    torch.cuda.synchronize()
    exp = ref.attn_fwd(f64(q), f64(k), f64(v), W, qk_gain=gain, ve=f64(ve), ve_gate=f64(gate))
    assert_close(out, exp, f"value embedding B{B} T{T} Hq{Hq} Hkv{Hkv} W{W}")


@pytest.mark.parametrize("B,Tq,Hq,Hkv,Tcap,lens,W", [(2, 130, 6, 2, 700, [0, 300], -1), (3, 1, 8, 8, 300, [5, 128, 255], 64),
                                                     (2, 200, 16, 1, 520, [320, 77], 63)])
def test_chunk_value_embedding(nc, B, Tq, Hq, Hkv, Tcap, lens, W):
    """The chunk's values carry their gated embedding into the cache and into the attention (the zero-padded copy of
    the last V tile included)."""
    from seeded_inputs import chunk_inputs
    d = chunk_inputs(B, Tq, Hq, Hkv, 128, Tcap, seed=B * Tq)
    g = torch.Generator("cpu").manual_seed(Tq)
    ve = torch.randn(d["v_new"].shape, generator=g).to(torch.bfloat16)
    gate = (2 * torch.randn(d["v_new"].shape[:3], generator=g)).to(torch.bfloat16)
    kc, vc = d["kcache"].cuda(), d["vcache"].cuda()
    out = nc.nc_attn_prefill_chunk(d["q"].cuda(), d["k_new"].cuda(), d["v_new"].cuda(), kc, vc,
                                   torch.tensor(lens, dtype=torch.int32, device="cuda"), window=W, ve_new=ve.cuda(),
                                   ve_gate=gate.cuda())
    torch.cuda.synchronize()
    exp, _ = ref.attn_prefill_chunk(*(f64(d[x]) for x in ("q", "k_new", "v_new", "kcache", "vcache")), lens, W,
                                    ve_new=f64(ve), ve_gate_new=f64(gate))
    assert_close(out, exp, f"chunk value embedding {B} {Tq} {Hq} {Hkv} {lens} W{W}")
    vmix = ref.value_mix(f64(d["v_new"]), f64(ve), f64(gate))
    vcc = f64(vc)
    for b, p in enumerate(lens):
        # the cache holds v' rounded to bf16 once: within half a bf16 ulp of the fp64 mix
        err = abs(vcc[b, p:p + Tq] - vmix[b])
        assert (err <= abs(vmix[b]) * 2.0 ** -8 + 1e-6).all()


@pytest.mark.parametrize("W", [-1, 700])
def test_decode_value_embedding(nc, W):
    """The new value of a decode step carries its gated embedding into the cache row and the attention."""
    from seeded_inputs import decode_inputs
    B, Hq, Hkv, Tcap = 9, 12, 4, 1200
    lens = [0, 1, 127, 128, 129, 700, 1000, 1198, 5]
    d = decode_inputs(B, Hq, Hkv, 128, Tcap, 1, 2, seed=31, with_new=True)
    g = torch.Generator("cpu").manual_seed(W + 2)
    ve = torch.randn(d["v_new"].shape, generator=g).to(torch.bfloat16)
    gate = (2 * torch.randn(d["v_new"].shape[:2], generator=g)).to(torch.bfloat16)
    lt = torch.tensor(lens, dtype=torch.int32)
    kc, vc = d["kcache"].cuda(), d["vcache"].cuda()
    out = nc.nc_attn_decode(d["q"].cuda(), kc, vc, lt.cuda(), k_new=d["k_new"].cuda(), v_new=d["v_new"].cuda(),
                            window=W, ve_new=ve.cuda(), ve_gate=gate.cuda())
    torch.cuda.synchronize()
    exp, _ = ref.attn_decode(f64(d["q"]), f64(d["kcache"]), f64(d["vcache"]), lt.numpy(), W, f64(d["k_new"]),
                             f64(d["v_new"]), ve_new=f64(ve), ve_gate_new=f64(gate))
    assert_close(out, exp, f"decode value embedding W={W}")
    vmix = ref.value_mix(f64(d["v_new"]), f64(ve), f64(gate))
    for b, p in enumerate(lens):
        err = abs(f64(vc[b, p]) - vmix[b])
        assert (err <= abs(vmix[b]) * 2.0 ** -8 + 1e-6).all()
