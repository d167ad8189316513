"""Host-side tests of the C ABI (no GPU needed, no kernel launched).

* the shared library loads and exports every function ``include/nc_attn.h`` declares;
* invalid arguments are rejected on the host with the documented status code before anything is launched;
* workspace sizes and status strings.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nc_attn.h")


@pytest.fixture(scope="module")
def nc():
    from transformer_attention_06_b300 import build
    build.build()
    from transformer_attention_06_b300 import nc_attn
    return nc_attn


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nc_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("nc_attn_fwd", "nc_attn_fwd_ws", "nc_attn_decode", "nc_attn_decode_ws", "nc_attn_status_string",
              "nc_attn_get_device_status", "nc_attn_qk_prologue", "nc_attn_prefill_chunk", "nc_attn_prefill_chunk_ws",
              "nc_attn_fwd_ex", "nc_attn_prefill_chunk_ex", "nc_attn_decode_ex", "nc_attn_bwd_ws", "nc_attn_fwd_ve"):
        assert n in names


def test_library_exports_every_declared_symbol(nc):
    raw = ctypes.CDLL(nc.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


P = ctypes.c_void_p(0x10000)          # a non-null, 16-byte-aligned dummy address (never dereferenced)
PM = ctypes.c_void_p(0x10008)         # misaligned


def fwd(nc, q=P, k=P, v=P, out=P, B=1, T=256, Hq=4, Hkv=2, D=128, W=-1, base=1e5, ws=None, wsb=0):
    return nc.lib.nc_attn_fwd_ws(q, k, v, out, B, T, Hq, Hkv, D, W, base, ws, wsb, None)


def test_fwd_rejects_bad_arguments(nc):
    E, U, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_UNSUPPORTED, nc.NC_ERR_WORKSPACE
    assert fwd(nc, q=None) == E
    assert fwd(nc, out=None) == E
    assert fwd(nc, v=PM) == E
    assert fwd(nc, B=0) == E
    assert fwd(nc, T=0) == E
    assert fwd(nc, Hq=3, Hkv=2) == E           # Hq % Hkv != 0
    assert fwd(nc, W=-2) == E
    assert fwd(nc, base=0.0) == E
    assert fwd(nc, base=float("nan")) == E
    assert fwd(nc, D=64) == U
    assert fwd(nc, T=1 << 24) == U
    assert fwd(nc, B=1 << 20, T=1 << 12) == U      # B * T tokens beyond 32-bit indexing
    # the prologue rounds B * T up to its 32-token blocks in 32-bit arithmetic: 2^31 - 1 - 32 tokens is the largest
    # accepted count (the call then fails only for want of a workspace), one more is refused
    assert fwd(nc, B=155, T=13854733) == WS         # 2147483615 tokens
    assert fwd(nc, B=87392, T=24573) == U           # 2147483616 tokens
    assert fwd(nc, Hq=256, Hkv=1) == U          # group larger than one 128-row tile
    assert fwd(nc) == WS                        # no workspace
    need = nc.nc_attn_fwd_workspace_bytes(1, 256, 4, 2)
    assert fwd(nc, ws=P, wsb=need - 1) == WS
    assert fwd(nc, ws=PM, wsb=need) == WS


def test_prologue_rejects_bad_arguments(nc):
    f = nc.lib.nc_attn_qk_prologue
    assert f(None, P, P, P, 1, 8, 2, 2, 128, 1e5, None) == nc.NC_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 8, 2, 2, 96, 1e5, None) == nc.NC_ERR_UNSUPPORTED
    assert f(P, P, P, P, 1, 8, 2, 2, 128, -1.0, None) == nc.NC_ERR_INVALID_ARG


def dec(nc, q=P, kc=P, vc=P, lens=P, out=P, kn=None, vn=None, B=4, Hq=12, Hkv=4, D=128, Tcap=64, W=-1, base=1e5,
        ws=None, wsb=0):
    return nc.lib.nc_attn_decode_ws(q, kc, vc, lens, out, kn, vn, B, Hq, Hkv, D, Tcap, W, base, ws, wsb, None)


def test_decode_rejects_bad_arguments(nc):
    E, U, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_UNSUPPORTED, nc.NC_ERR_WORKSPACE
    assert dec(nc, lens=None) == E
    assert dec(nc, kc=None) == E
    assert dec(nc, kn=P) == E                   # k_new without v_new
    assert dec(nc, kn=P, vn=PM) == E
    assert dec(nc, lens=ctypes.c_void_p(0x10002)) == E
    assert dec(nc, Tcap=0) == E
    assert dec(nc, Hq=10, Hkv=4) == E
    assert dec(nc, W=-5) == E
    assert dec(nc, base=float("inf")) == E
    assert dec(nc, D=256) == U
    assert dec(nc, Hq=68, Hkv=4) == U           # group of 17 > 16
    assert dec(nc) == WS
    need = nc.nc_attn_decode_workspace_bytes(4, 12, 4, 128, 64, -1)
    assert dec(nc, ws=P, wsb=need - 1) == WS


def chunk(nc, q=P, kn=P, vn=P, kc=P, vc=P, lens=P, out=P, B=2, Tq=100, Hq=6, Hkv=2, D=128, Tcap=300, W=-1,
          base=1e5, ws=None, wsb=0):
    return nc.lib.nc_attn_prefill_chunk_ws(q, kn, vn, kc, vc, lens, out, B, Tq, Hq, Hkv, D, Tcap, W, base, ws, wsb,
                                           None)


def test_prefill_chunk_rejects_bad_arguments(nc):
    E, U, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_UNSUPPORTED, nc.NC_ERR_WORKSPACE
    assert chunk(nc, q=None) == E
    assert chunk(nc, vn=None) == E
    assert chunk(nc, lens=None) == E
    assert chunk(nc, kc=PM) == E
    assert chunk(nc, lens=ctypes.c_void_p(0x10002)) == E
    assert chunk(nc, Tq=0) == E
    assert chunk(nc, Tcap=99) == E               # the chunk does not fit the cache
    assert chunk(nc, Hq=5, Hkv=2) == E
    assert chunk(nc, W=-2) == E
    assert chunk(nc, base=0.0) == E
    assert chunk(nc, D=64) == U
    assert chunk(nc, Tcap=1 << 24) == U          # cache positions must be exact in fp32
    assert chunk(nc, Hq=256, Hkv=1) == U
    assert chunk(nc) == WS
    need = nc.nc_attn_prefill_chunk_workspace_bytes(2, 100, 6, 2)
    assert chunk(nc, ws=P, wsb=need - 1) == WS
    assert chunk(nc, ws=PM, wsb=need) == WS


def test_qk_gain_range_is_checked(nc):
    # (0, 4]: outside it the prefill softmax's bound on the logits would not hold; checked before anything else
    E = nc.NC_ERR_INVALID_ARG
    for g in (0.0, -1.0, 4.01, float("nan"), float("inf")):
        assert nc.lib.nc_attn_fwd_ex(P, P, P, P, 1, 256, 4, 2, 128, -1, 1e5, g, None, 0, None) == E
        assert nc.lib.nc_attn_prefill_chunk_ex(P, P, P, P, P, P, P, 2, 100, 6, 2, 128, 300, -1, 1e5, g, None, 0,
                                               None) == E
        assert nc.lib.nc_attn_decode_ex(P, P, P, P, P, None, None, 4, 12, 4, 128, 64, -1, 1e5, g, None, 0, None) == E
    # a valid gain reaches the next check (the missing workspace)
    assert nc.lib.nc_attn_fwd_ex(P, P, P, P, 1, 256, 4, 2, 128, -1, 1e5, 4.0, None, 0, None) == nc.NC_ERR_WORKSPACE
    assert nc.lib.nc_attn_decode_ex(P, P, P, P, P, None, None, 4, 12, 4, 128, 64, -1, 1e5, 1.2, None, 0,
                                    None) == nc.NC_ERR_WORKSPACE


def test_bwd_rejects_bad_arguments(nc):
    E, U, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_UNSUPPORTED, nc.NC_ERR_WORKSPACE
    f = nc.lib.nc_attn_bwd_ws

    def call(q=P, dq=P, B=1, T=64, Hq=4, Hkv=2, D=128, W=-1, gain=1.0, ws=None, wsb=0):
        return f(q, P, P, P, dq, P, P, B, T, Hq, Hkv, D, W, 1e5, gain, ws, wsb, None)
    assert call(q=None) == E
    assert call(dq=None) == E
    assert call(dq=PM) == E
    assert call(Hq=3, Hkv=2) == E
    assert call(W=-2) == E
    assert call(gain=0.0) == E
    assert call(D=64) == U
    assert call() == WS
    need = nc.lib.nc_attn_bwd_workspace_bytes(1, 64, 4, 2, 128)
    # qn, kn in bf16, then the row statistics: two fp32 values per row of each padded 128-row Q tile (G = 2: P = 64
    # positions per tile, one tile per kv head)
    assert need >= 2 * 64 * 6 * 128 + 2 * 2 * 128 * 4
    assert call(ws=P, wsb=need - 1) == WS
    assert call(Hq=256, Hkv=1) == U             # group larger than one 128-row tile


def test_saved_statistics_entry_points_reject_bad_arguments(nc):
    E, U, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_UNSUPPORTED, nc.NC_ERR_WORKSPACE
    # statistics of B=4, T=2048, Hq=Hkv=6 (G = 1: P = 128 positions per tile, 16 tiles): one float per packed row
    assert nc.lib.nc_attn_lse_bytes(4, 2048, 6, 6) == 4 * 6 * 16 * 128 * 4
    # G = 3: P = 42 positions per tile, ceil(300 / 42) = 8 tiles per kv head, 128 rows each (126 hold queries)
    assert nc.lib.nc_attn_lse_bytes(1, 300, 3, 1) == 8 * 128 * 4
    assert nc.lib.nc_attn_lse_bytes(1, 300, 4, 3) == 0
    fwd = nc.lib.nc_attn_fwd_lse_ws

    def f(q=P, lse=P, B=1, T=64, Hq=4, Hkv=2, D=128, gain=1.0, ws=None, wsb=0):
        return fwd(q, P, P, P, lse, B, T, Hq, Hkv, D, -1, 1e5, gain, ws, wsb, None)
    assert f(lse=None) == E
    assert f(lse=PM) == E                      # misaligned statistics buffer
    assert f(q=None) == E
    assert f(gain=5.0) == E
    assert f(D=64) == U
    assert f() == WS
    bwd = nc.lib.nc_attn_bwd_saved_ws

    def g(out=P, lse=P, B=1, T=64, Hq=4, Hkv=2, D=128, ws=None, wsb=0):
        return bwd(P, P, P, out, P, lse, P, P, P, B, T, Hq, Hkv, D, -1, 1e5, 1.0, ws, wsb, None)
    assert g(out=None) == E
    assert g(lse=None) == E
    assert g(out=PM) == E
    assert g(Hq=3, Hkv=2) == E
    assert g(D=64) == U
    assert g() == WS


def test_fwd_ve_rejects_bad_arguments(nc):
    E, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_WORKSPACE
    f = nc.lib.nc_attn_fwd_ve
    assert f(P, P, P, None, P, P, 1, 64, 4, 2, 128, -1, 1e5, 1.0, None, 0, None) == E        # no ve
    assert f(P, P, P, P, None, P, 1, 64, 4, 2, 128, -1, 1e5, 1.0, None, 0, None) == E        # no gate
    assert f(P, P, P, PM, P, P, 1, 64, 4, 2, 128, -1, 1e5, 1.0, None, 0, None) == E          # misaligned ve
    assert f(P, P, P, P, P, P, 1, 64, 4, 2, 128, -1, 1e5, 1.0, None, 0, None) == WS
    need = nc.lib.nc_attn_fwd_ve_workspace_bytes(1, 64, 4, 2, 128)
    assert need == nc.nc_attn_fwd_workspace_bytes(1, 64, 4, 2) + 2 * 64 * 2 * 128
    fwd_need = nc.nc_attn_fwd_workspace_bytes(1, 64, 4, 2)
    assert f(P, P, P, P, P, P, 1, 64, 4, 2, 128, -1, 1e5, 1.0, P, fwd_need, None) == WS      # room for v' missing


def test_workspace_sizes(nc):
    # chunked prefill: qn of the chunk and one 128-row V tail copy per sequence, in bf16, plus a counter
    assert nc.nc_attn_prefill_chunk_workspace_bytes(4, 512, 6, 6) >= 2 * 4 * 512 * 6 * 128 + 2 * 4 * 128 * 6 * 128
    assert nc.nc_attn_prefill_chunk_workspace_bytes(4, 512, 6, 4) == 0
    # qn + kn in bf16 plus a small pad
    assert nc.nc_attn_fwd_workspace_bytes(4, 2048, 6, 6) >= 2 * 4 * 2048 * 12 * 128
    assert nc.nc_attn_fwd_workspace_bytes(0, 2048, 6, 6) == 0
    # decode: B*Hkv counters + (m, l) and 128 floats for 2 partials per CTA (at most 256 CTAs) and group head;
    # independent of the cache length and window
    n = nc.nc_attn_decode_workspace_bytes(64, 12, 4, 128, 4097, 2048)
    assert n >= 64 * 4 * 4 + 256 * 2 * 3 * 130 * 4
    assert n == nc.nc_attn_decode_workspace_bytes(64, 12, 4, 128, 100, 100)
    assert nc.nc_attn_decode_workspace_bytes(128, 12, 4, 128, 4097, 2048) > n
    assert nc.nc_attn_decode_workspace_bytes(64, 12, 2, 128, 4097, 2048) > n   # larger group
    assert nc.nc_attn_decode_workspace_bytes(64, 12, 4, 64, 4097, 2048) == 0


def test_status_strings(nc):
    for s in range(7):
        assert nc.status_string(s).startswith("NC_")
    assert "unknown" in nc.status_string(99)


def test_binding_rejects_host_tensors(nc):
    import torch
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        nc.nc_attn_fwd(q, q, q)
    with pytest.raises(ValueError):
        nc.nc_attn_decode(q[:, 0], q, q, torch.zeros(1, dtype=torch.int32))


def test_a_c_program_links_and_calls_the_library(tmp_path):
    """The boundary is plain C: a C99 translation unit includes the header, links libnc_attn.so and calls host-only
    entry points (no GPU needed)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from transformer_attention_06_b300 import nc_attn
    src = tmp_path / "caller.c"
    src.write_text(
        '#include <stdio.h>\n#include "nc_attn.h"\n'
        "int main(void) {\n"
        "  size_t n = nc_attn_fwd_workspace_bytes(4, 2048, 6, 6, 128);\n"
        "  nc_status s = nc_attn_fwd_ws(0, 0, 0, 0, 1, 8, 2, 2, 128, -1, 1e5f, 0, 0, 0);\n"
        '  printf("%zu %d %s\\n", n, (int)s, nc_attn_status_string(s));\n'
        "  return 0;\n}\n")
    libdir = os.path.dirname(nc_attn.LIB_PATH)
    exe = tmp_path / "caller"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-o", str(exe), str(src), "-I", os.path.dirname(HEADER), "-I", cuda_inc,
                    "-L", libdir, "-lnc_attn", f"-Wl,-rpath,{libdir}"], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == nc_attn.nc_attn_fwd_workspace_bytes(4, 2048, 6, 6)
    assert int(out[1]) == nc_attn.NC_ERR_INVALID_ARG


def test_fwd_fp8_rejects_bad_arguments(nc):
    E, U, WS = nc.NC_ERR_INVALID_ARG, nc.NC_ERR_UNSUPPORTED, nc.NC_ERR_WORKSPACE
    f = nc.lib.nc_attn_fwd_fp8

    def call(q=P, k=P, v=P, out=P, B=1, T=256, Hq=4, Hkv=2, D=128, W=-1, base=1e5, gain=1.0, ws=None, wsb=0):
        return f(q, k, v, out, B, T, Hq, Hkv, D, W, base, gain, ws, wsb, None)

    assert call(q=None) == E
    assert call(v=PM) == E
    assert call(Hq=3, Hkv=2) == E
    assert call(W=-2) == E
    assert call(gain=0.0) == E and call(gain=4.5) == E
    assert call(D=64) == U
    assert call() == WS
    need = nc.lib.nc_attn_fwd_fp8_workspace_bytes(1, 256, 4, 2, 128)
    assert need == 256 * (4 + 2) * 128 + 256          # one byte per element of qn and kn, then the counter
    assert call(ws=P, wsb=need - 1) == WS
    g = nc.lib.nc_attn_qk_prologue_fp8
    assert g(None, P, P, P, 1, 8, 2, 2, 128, 1e5, 1.0, None) == E
    assert g(P, P, P, P, 1, 8, 2, 2, 128, 1e5, 5.0, None) == E
    assert g(P, P, P, P, 1, 8, 2, 2, 96, 1e5, 1.0, None) == U
