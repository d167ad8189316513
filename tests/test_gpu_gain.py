"""GPU parity of the QK-norm gain (the factor on every logit; 1.2 in nanochat) on the three paths, against the fp64
oracle with the same gain.  The largest accepted gain (4) on long causal rows exercises the bound that lets the
prefill softmax run without a running maximum (base-2 logits up to 66 in magnitude).

Tolerance: the kernels hold qn and kn in bf16, so every logit carries their rounding (relative 2^-9 per element)
multiplied by the gain, and the output error grows in proportion; the parity bar (max-abs 2e-2, mean-abs 2e-3 at
gain <= 1.2) is scaled by max(1, gain / 1.2).  The oracle works from the same bf16 inputs in fp64 without that
rounding."""

import pytest
import torch

from oracle import ref
from seeded_inputs import chunk_inputs, decode_inputs, fwd_inputs
from tests.parity import MAX_ABS, MEAN_ABS, assert_close, f64

pytestmark = pytest.mark.gpu


def close(got, exp, what, gain):
    s = max(1.0, gain / 1.2)
    return assert_close(got, exp, what, max_abs=MAX_ABS * s, mean_abs=MEAN_ABS * s)


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_attention_06_b300 import nc_attn
    nc_attn.nc_attn_get_device_status(clear=True)
    yield nc_attn
    assert nc_attn.nc_attn_get_device_status(clear=True) == nc_attn.NC_OK


@pytest.mark.parametrize("gain,B,T,Hq,Hkv,W", [(1.2, 2, 300, 6, 2, 127), (1.2, 1, 700, 4, 4, -1),
                                               (4.0, 1, 700, 4, 4, -1), (0.25, 1, 200, 8, 2, 50)])
def test_fwd_gain(nc, gain, B, T, Hq, Hkv, W):
    q, k, v = fwd_inputs(B, T, Hq, Hkv, 128, seed=31)
    out = nc.nc_attn_fwd(q.cuda(), k.cuda(), v.cuda(), window=W, qk_gain=gain)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    close(out, ref.attn_fwd(f64(q), f64(k), f64(v), W, qk_gain=gain), f"fwd gain={gain}", gain)


@pytest.mark.parametrize("gain", [1.2, 4.0])
def test_decode_gain(nc, gain):
    d = decode_inputs(5, 12, 4, 128, 600, 1, 598, seed=12, with_new=True)
    kc, vc = d["kcache"].cuda(), d["vcache"].cuda()
    out = nc.nc_attn_decode(d["q"].cuda(), kc, vc, d["cache_lens"].cuda(), k_new=d["k_new"].cuda(),
                            v_new=d["v_new"].cuda(), window=300, qk_gain=gain)
    torch.cuda.synchronize()
    exp, _ = ref.attn_decode(f64(d["q"]), f64(d["kcache"]), f64(d["vcache"]), d["cache_lens"].numpy(), 300,
                             f64(d["k_new"]), f64(d["v_new"]), qk_gain=gain)
    close(out, exp, f"decode gain={gain}", gain)


def test_chunk_gain(nc):
    d = chunk_inputs(2, 150, 6, 2, 128, 600, seed=13)
    lens = [0, 321]
    kc, vc = d["kcache"].cuda(), d["vcache"].cuda()
    out = nc.nc_attn_prefill_chunk(d["q"].cuda(), d["k_new"].cuda(), d["v_new"].cuda(), kc, vc,
                                   torch.tensor(lens, dtype=torch.int32, device="cuda"), window=200, qk_gain=1.2)
    torch.cuda.synchronize()
    exp, _ = ref.attn_prefill_chunk(*(f64(d[x]) for x in ("q", "k_new", "v_new", "kcache", "vcache")), lens, 200,
                                    qk_gain=1.2)
    close(out, exp, "chunk gain=1.2", 1.2)
