"""GPU parity of the gated value embedding (v' = v + sigmoid(g) ve, formed in the prologue kernel) against the fp64
oracle, same tolerance as the other prefill parity tests (v' is rounded to bf16 once, like v itself)."""

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
