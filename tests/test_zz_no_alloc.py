"""The decode entry point that allocates nothing, against the decode entry point with a caller workspace.

``nc_attn_decode_noalloc`` exists for callers that may not allocate device memory at all: code running inside a host
framework's plugin hook, where that framework owns the memory budget, or serving loops that forbid cudaMalloc /
cudaFree after start-up because those calls can synchronize the device.  It keeps its split partials in a fixed array
inside the library, shared by every call, so the GPU test makes several calls in a row with different B * Hkv (a call
may find the previous call's partials where its own counters go) and checks that each result is bit-identical to
``nc_attn_decode_ws`` on the same inputs (both run the same kernel).

This file is named so that pytest collects it last.
"""

import pytest
import torch

from seeded_inputs import decode_inputs


def _nc():
    from transformer_attention_06_b300 import build
    build.build()
    from transformer_attention_06_b300 import nc_attn
    return nc_attn


def test_noalloc_rejects_requests_beyond_its_scratch():
    # Checked on the host before any CUDA call: a non-null, aligned dummy address is never dereferenced.
    nc = _nc()
    P = 0x10000
    B, Hq, Hkv, Tcap = 65535, 64, 64, 4096    # 4 Mi sequence x kv-head arrival counters alone exceed the array
    need = nc.nc_attn_decode_workspace_bytes(B, Hq, Hkv, 128, Tcap, -1)
    assert need > nc.NC_ATTN_DECODE_NOALLOC_MAX_BYTES
    st = nc.lib.nc_attn_decode_noalloc(P, P, P, P, P, None, None, B, Hq, Hkv, 128, Tcap, -1, 1e5, None)
    assert st == nc.NC_ERR_SCRATCH_LIMIT
    assert "NOALLOC_MAX_BYTES" in nc.status_string(st)
    # Argument errors keep their own codes.
    st = nc.lib.nc_attn_decode_noalloc(None, P, P, P, P, None, None, 4, 12, 4, 128, 300, 128, 1e5, None)
    assert st == nc.NC_ERR_INVALID_ARG


# (B, Hq, Hkv, Tcap, len_lo, len_hi, window, with_new, seed): the 64-sequence decode workload, then a request with
# another B * Hkv and a new key, then the first shape again.
CALLS = [
    (64, 12, 4, 4097, 1, 4096, 2048, False, 0),
    (7, 8, 2, 700, 0, 699, -1, True, 5),
    (64, 12, 4, 4097, 1, 4096, 2048, True, 9),
]


@pytest.mark.gpu
def test_noalloc_matches_decode_ws_on_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nc = _nc()
    dev = torch.device("cuda:0")
    nc.nc_attn_get_device_status(clear=True)
    for (B, Hq, Hkv, Tcap, lo, hi, W, with_new, seed) in CALLS:
        assert nc.nc_attn_decode_workspace_bytes(B, Hq, Hkv, 128, Tcap, W) <= nc.NC_ATTN_DECODE_NOALLOC_MAX_BYTES
        d = decode_inputs(B, Hq, Hkv, 128, Tcap, lo, hi, seed=seed, with_new=with_new)
        q, lens = d["q"].to(dev), d["cache_lens"].to(dev)
        kn = d["k_new"].to(dev) if with_new else None
        vn = d["v_new"].to(dev) if with_new else None
        # Each entry point gets its own cache copies, since a new key is written into the cache.
        kc_a, vc_a = d["kcache"].to(dev), d["vcache"].to(dev)
        kc_b, vc_b = kc_a.clone(), vc_a.clone()

        ws = torch.zeros(nc.nc_attn_decode_workspace_bytes(B, Hq, Hkv, 128, Tcap, W), dtype=torch.uint8, device=dev)
        want = nc.nc_attn_decode(q, kc_a, vc_a, lens, k_new=kn, v_new=vn, window=W, workspace=ws)
        got = torch.full_like(q, float("nan"))
        nc.nc_attn_decode_noalloc(q, kc_b, vc_b, lens, got, k_new=kn, v_new=vn, window=W)
        torch.cuda.synchronize()
        # the same kernel on the same inputs: bit-identical, so a stale partial left in the shared array would show
        assert torch.equal(got, want), f"noalloc vs ws, B={B} Hq={Hq} Hkv={Hkv} W={W}"
        assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b)
    assert nc.nc_attn_get_device_status(clear=True) == nc.NC_OK
