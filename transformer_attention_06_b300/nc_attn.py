"""Python binding of the C-ABI library ``libnc_attn.so`` (argument marshalling only).

Every function here checks the torch tensors it is given (device, dtype, contiguity, shapes), passes their device
pointers and the current CUDA stream to the library entry point of the same name, and raises ``NcAttnError`` on a
non-zero status.  All arithmetic runs in the library's CUDA kernels; there is no other implementation and no CPU
fallback: if the shared library is missing, importing this module fails.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnc_attn.so")

ROPE_BASE = 100000.0

NC_OK = 0
NC_ERR_INVALID_ARG = 1
NC_ERR_UNSUPPORTED = 2
NC_ERR_CUDA = 3
NC_ERR_DEVICE_TIMEOUT = 4
NC_ERR_DEVICE_BAD_INPUT = 5
NC_ERR_WORKSPACE = 6
NC_ERR_SCRATCH_LIMIT = 7


class NcAttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m transformer_attention_06_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sigs = {
        "nc_attn_fwd_workspace_bytes": (sz, [i, i, i, i, i]),
        "nc_attn_fwd_ws": (i, [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp]),
        "nc_attn_fwd": (i, [vp, vp, vp, vp, i, i, i, i, i, i, f, vp]),
        "nc_attn_fwd_ws_events": (i, [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp, vp, vp, vp]),
        "nc_attn_qk_prologue": (i, [vp, vp, vp, vp, i, i, i, i, i, f, vp]),
        "nc_attn_decode_workspace_bytes": (sz, [i, i, i, i, i, i]),
        "nc_attn_fwd_ex": (i, [vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_bwd_workspace_bytes": (sz, [i, i, i, i, i]),
        "nc_attn_fwd_ve_workspace_bytes": (sz, [i, i, i, i, i]),
        "nc_attn_fwd_ve": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_bwd_ws": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_lse_bytes": (sz, [i, i, i, i]),
        "nc_attn_fwd_lse_ws": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_bwd_saved_ws": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_prefill_chunk_ex": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_decode_ex": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_prefill_chunk_workspace_bytes": (sz, [i, i, i, i, i]),
        "nc_attn_prefill_chunk_ws": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz, vp]),
        "nc_attn_prefill_chunk": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]),
        "nc_attn_decode_ws": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp]),
        "nc_attn_decode": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]),
        "nc_attn_decode_noalloc": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]),
        "nc_attn_fwd_fp8_workspace_bytes": (sz, [i, i, i, i, i]),
        "nc_attn_fwd_fp8": (i, [vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_fwd_fp8_events": (i, [vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp, vp, vp, vp]),
        "nc_attn_qk_prologue_fp8": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, vp]),
        "nc_attn_prefill_chunk_ve": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_decode_ve": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, vp, sz, vp]),
        "nc_attn_status_string": (ctypes.c_char_p, [i]),
        "nc_attn_get_device_status": (i, [vp, i]),
        "nc_attn_selftest_wait_timeout": (i, [i, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status):
    return lib.nc_attn_status_string(int(status)).decode()


def _check(status, where):
    if status != NC_OK:
        raise NcAttnError(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _event_handle(e, stream):
    """Raw cudaEvent_t of a torch.cuda.Event.  torch creates the CUDA event on its first record, so an event that was
    never recorded is recorded once here (the library records it again at the right place)."""
    if e is None:
        return None
    if e.cuda_event == 0:
        e.record(stream if stream is not None else torch.cuda.current_stream())
    return ctypes.c_void_p(e.cuda_event)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, ndim, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# Workspaces cached per (device, kind); the decode one starts zero-filled and every call leaves its counters zero.
# A decode call with another B * Hkv than the previous one may find the previous call's partials where its counters
# go, so the cached decode workspace is cleared when B * Hkv changes.
_ws_cache = {}
_ws_decode_tag = {}


def _workspace(kind, nbytes, device, zero):
    key = (kind, device.index if device.index is not None else torch.cuda.current_device())
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = (torch.zeros if zero else torch.empty)(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D=128):
    return int(lib.nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D))


def nc_attn_prefill_chunk_workspace_bytes(B, Tq, Hq, Hkv, D=128):
    return int(lib.nc_attn_prefill_chunk_workspace_bytes(B, Tq, Hq, Hkv, D))


def nc_attn_decode_workspace_bytes(B, Hq, Hkv, D, Tcap, window):
    return int(lib.nc_attn_decode_workspace_bytes(B, Hq, Hkv, D, Tcap, window))


def nc_attn_fwd(q, k, v, out=None, window=-1, rope_base=ROPE_BASE, workspace=None, stream=None, events=None,
                qk_gain=1.0, ve=None, ve_gate=None):
    """Prefill / training forward.  q [B,T,Hq,D], k and v [B,T,Hkv,D] (bf16, CUDA, contiguous) -> out [B,T,Hq,D].

    ``events``: optional (k1_begin, k2_begin, k2_end) torch.cuda.Event objects (any may be None), recorded on the
    stream around the prologue kernel and the attention kernel.  ``qk_gain``: factor on every logit (the QK-norm
    gain, 1.2 in nanochat; ``nc_attn_fwd_ex``); not combined with ``events``.  ``ve`` [B,T,Hkv,D] and ``ve_gate``
    [B,T,Hkv] (bf16): gated value embedding, the attention runs on v + sigmoid(ve_gate) * ve (``nc_attn_fwd_ve``).
    """
    _need(q, "q", 4)
    _need(k, "k", 4)
    _need(v, "v", 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, T, Hkv, D) or tuple(v.shape) != (B, T, Hkv, D):
        raise ValueError(f"k/v shapes {tuple(k.shape)}/{tuple(v.shape)} do not match q {tuple(q.shape)}")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 4)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have the shape of q")
    if ve is not None or ve_gate is not None:
        nbytes = int(lib.nc_attn_fwd_ve_workspace_bytes(B, T, Hq, Hkv, D))
    else:
        nbytes = nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D)
    if workspace is None:
        workspace = _workspace("fwd", nbytes, q.device, zero=False)
    if ve is not None or ve_gate is not None:
        if ve is None or ve_gate is None or events is not None:
            raise ValueError("ve and ve_gate go together, and without events")
        _need(ve, "ve", 4)
        _need(ve_gate, "ve_gate", 3)
        if tuple(ve.shape) != tuple(v.shape) or tuple(ve_gate.shape) != tuple(v.shape[:3]):
            raise ValueError("ve must have v's shape and ve_gate [B, T, Hkv]")
        st = lib.nc_attn_fwd_ve(_ptr(q), _ptr(k), _ptr(v), _ptr(ve), _ptr(ve_gate), _ptr(out), B, T, Hq, Hkv, D,
                                int(window), float(rope_base), float(qk_gain), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
        _check(st, "nc_attn_fwd")
        return out
    wsb = workspace.numel() * workspace.element_size()
    if qk_gain != 1.0:
        if events is not None:
            raise ValueError("events are recorded only with qk_gain = 1")
        st = lib.nc_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, Hq, Hkv, D, int(window), float(rope_base),
                                float(qk_gain), _ptr(workspace), wsb, _stream(stream))
        _check(st, "nc_attn_fwd")
        return out
    ev = [_event_handle(e, stream) for e in (events or (None, None, None))]
    st = lib.nc_attn_fwd_ws_events(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, Hq, Hkv, D, int(window),
                                   float(rope_base), _ptr(workspace), wsb, ev[0], ev[1], ev[2], _stream(stream))
    _check(st, "nc_attn_fwd")
    return out


def nc_attn_fwd_fp8_workspace_bytes(B, T, Hq, Hkv, D=128):
    return int(lib.nc_attn_fwd_fp8_workspace_bytes(B, T, Hq, Hkv, D))


def nc_attn_fwd_fp8(q, k, v, out=None, window=-1, rope_base=ROPE_BASE, qk_gain=1.0, workspace=None, stream=None,
                    events=None):
    """Prefill forward with the score contraction on e4m3 operands (``nc_attn_fwd_fp8``): q [B,T,Hq,D], k and v
    [B,T,Hkv,D] (bf16, CUDA, contiguous) -> out [B,T,Hq,D] bf16.  ``events``: optional (k1_begin, k2_begin, k2_end)
    torch.cuda.Event objects recorded around the prologue and the attention kernel."""
    _need(q, "q", 4)
    _need(k, "k", 4)
    _need(v, "v", 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, T, Hkv, D) or tuple(v.shape) != (B, T, Hkv, D):
        raise ValueError(f"k/v shapes {tuple(k.shape)}/{tuple(v.shape)} do not match q {tuple(q.shape)}")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 4)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have the shape of q")
    if workspace is None:
        workspace = _workspace("fwd", nc_attn_fwd_fp8_workspace_bytes(B, T, Hq, Hkv, D), q.device, zero=False)
    wsb = workspace.numel() * workspace.element_size()
    ev = [_event_handle(e, stream) for e in (events or (None, None, None))]
    st = lib.nc_attn_fwd_fp8_events(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, Hq, Hkv, D, int(window),
                                    float(rope_base), float(qk_gain), _ptr(workspace), wsb, ev[0], ev[1], ev[2],
                                    _stream(stream))
    _check(st, "nc_attn_fwd_fp8")
    return out


def nc_attn_qk_prologue_fp8(q, k, qk_gain=1.0, rope_base=ROPE_BASE, stream=None):
    """The e4m3 prologue alone: returns (qn8, kn8), uint8 tensors of q's and k's shapes holding the e4m3 codes of
    norm(rope(q)) * s_q and norm(rope(k)) * s_k (``nc_attn_qk_prologue_fp8``)."""
    _need(q, "q", 4)
    _need(k, "k", 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    qn8 = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    kn8 = torch.empty(k.shape, dtype=torch.uint8, device=k.device)
    st = lib.nc_attn_qk_prologue_fp8(_ptr(q), _ptr(k), _ptr(qn8), _ptr(kn8), B, T, Hq, Hkv, D, float(rope_base),
                                     float(qk_gain), _stream(stream))
    _check(st, "nc_attn_qk_prologue_fp8")
    return qn8, kn8


def nc_attn_bwd(q, k, v, dout, window=-1, rope_base=ROPE_BASE, qk_gain=1.0, workspace=None, stream=None):
    """Gradients of sum(dout * nc_attn_fwd(q, k, v, window, qk_gain=...)) with respect to q, k, v.

    q, dout [B,T,Hq,D] and k, v [B,T,Hkv,D] (bf16, CUDA, contiguous) -> (dq, dk, dv) fp32 tensors of the same shapes.
    """
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, name, 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, T, Hkv, D) or tuple(v.shape) != (B, T, Hkv, D) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("k / v / dout shapes do not match q")
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    nbytes = int(lib.nc_attn_bwd_workspace_bytes(B, T, Hq, Hkv, D))
    if workspace is None:
        workspace = _workspace("bwd", nbytes, q.device, zero=False)
    st = lib.nc_attn_bwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, T, Hq, Hkv, D,
                            int(window), float(rope_base), float(qk_gain), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nc_attn_bwd")
    return dq, dk, dv


def nc_attn_fwd_lse(q, k, v, out=None, lse=None, window=-1, rope_base=ROPE_BASE, qk_gain=1.0, workspace=None,
                    stream=None):
    """Training forward: (out, lse) where lse holds every query row's base-2 log-sum-exp (float32, the packed layout
    of nc_attn_lse_bytes / nc_attn_fwd_lse_ws: [B][Hkv][ceil(T / P)][128], P = 128 // (Hq // Hkv)) for
    nc_attn_bwd_saved."""
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, name, 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, T, Hkv, D) or tuple(v.shape) != (B, T, Hkv, D):
        raise ValueError("k / v shapes do not match q")
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", 4)
    nl = int(lib.nc_attn_lse_bytes(B, T, Hq, Hkv))
    if lse is None:
        lse = torch.empty(max(nl, 4) // 4, dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or not lse.is_cuda or lse.numel() * 4 < nl:
        raise ValueError(f"lse must be a CUDA float32 tensor of at least {nl} bytes")
    nbytes = int(lib.nc_attn_fwd_workspace_bytes(B, T, Hq, Hkv, D))
    if workspace is None:
        workspace = _workspace("fwd", nbytes, q.device, zero=False)
    st = lib.nc_attn_fwd_lse_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, T, Hq, Hkv, D, int(window),
                                float(rope_base), float(qk_gain), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nc_attn_fwd_lse")
    return out, lse


def nc_attn_bwd_saved(q, k, v, out, dout, lse, window=-1, rope_base=ROPE_BASE, qk_gain=1.0, workspace=None,
                      stream=None):
    """Gradients (dq, dk, dv) like nc_attn_bwd, reusing the output and lse of nc_attn_fwd_lse instead of running the
    forward again."""
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, name, 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if (tuple(k.shape) != (B, T, Hkv, D) or tuple(v.shape) != (B, T, Hkv, D) or tuple(dout.shape) != tuple(q.shape)
            or tuple(out.shape) != tuple(q.shape)):
        raise ValueError("k / v / out / dout shapes do not match q")
    if lse.dtype != torch.float32 or not lse.is_cuda or lse.numel() * 4 < int(lib.nc_attn_lse_bytes(B, T, Hq, Hkv)):
        raise ValueError("lse must be the float32 statistics of nc_attn_fwd_lse for these shapes")
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    nbytes = int(lib.nc_attn_bwd_workspace_bytes(B, T, Hq, Hkv, D))
    if workspace is None:
        workspace = _workspace("bwd", nbytes, q.device, zero=False)
    st = lib.nc_attn_bwd_saved_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, T, Hq, Hkv, D, int(window), float(rope_base), float(qk_gain),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nc_attn_bwd_saved")
    return dq, dk, dv


def nc_attn_qk_prologue(q, k, qn=None, kn=None, rope_base=ROPE_BASE, stream=None):
    """RoPE + weightless RMSNorm of q [B,T,Hq,D] and k [B,T,Hkv,D] at positions 0..T-1 -> (qn, kn), bf16."""
    _need(q, "q", 4)
    _need(k, "k", 4)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, T, Hkv, D):
        raise ValueError("k shape does not match q")
    qn = torch.empty_like(q) if qn is None else qn
    kn = torch.empty_like(k) if kn is None else kn
    _need(qn, "qn", 4)
    _need(kn, "kn", 4)
    st = lib.nc_attn_qk_prologue(_ptr(q), _ptr(k), _ptr(qn), _ptr(kn), B, T, Hq, Hkv, D, float(rope_base),
                                 _stream(stream))
    _check(st, "nc_attn_qk_prologue")
    return qn, kn


def nc_attn_prefill_chunk(q, k_new, v_new, kcache, vcache, cache_lens, out=None, window=-1, rope_base=ROPE_BASE,
                          workspace=None, stream=None, qk_gain=1.0, ve_new=None, ve_gate=None):
    """Chunked prefill against a KV cache.  q [B,Tq,Hq,D], k_new / v_new [B,Tq,Hkv,D] (raw), caches
    [B,Tcap,Hkv,D], cache_lens int32 [B] (device) -> out [B,Tq,Hq,D].

    The chunk's keys (roped at cache_lens[b] + t and normed) and values are written into the caches at rows
    cache_lens[b] .. cache_lens[b] + Tq - 1; query t attends to the cache rows up to its own position.  cache_lens is
    not modified.  ``ve_new`` [B,Tq,Hkv,D] and ``ve_gate`` [B,Tq,Hkv]: gated value embedding of the chunk's values
    (``nc_attn_prefill_chunk_ve``).
    """
    _need(q, "q", 4)
    _need(k_new, "k_new", 4)
    _need(v_new, "v_new", 4)
    _need(kcache, "kcache", 4)
    _need(vcache, "vcache", 4)
    _need(cache_lens, "cache_lens", 1, dtype=torch.int32)
    B, Tq, Hq, D = q.shape
    Hkv = k_new.shape[2]
    Tcap = kcache.shape[1]
    if tuple(k_new.shape) != (B, Tq, Hkv, D) or tuple(v_new.shape) != (B, Tq, Hkv, D):
        raise ValueError("k_new / v_new must be [B, Tq, Hkv, D]")
    if tuple(kcache.shape) != (B, Tcap, Hkv, D) or tuple(vcache.shape) != (B, Tcap, Hkv, D):
        raise ValueError("cache shapes do not match q")
    if cache_lens.shape[0] != B:
        raise ValueError("cache_lens must have B entries")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 4)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have the shape of q")
    nbytes = nc_attn_prefill_chunk_workspace_bytes(B, Tq, Hq, Hkv, D)
    if workspace is None:
        workspace = _workspace("chunk", nbytes, q.device, zero=False)
    wsb = workspace.numel() * workspace.element_size()
    if ve_new is not None or ve_gate is not None:
        if ve_new is None or ve_gate is None:
            raise ValueError("ve_new and ve_gate go together")
        _need(ve_new, "ve_new", 4)
        _need(ve_gate, "ve_gate", 3)
        if tuple(ve_new.shape) != tuple(v_new.shape) or tuple(ve_gate.shape) != tuple(v_new.shape[:3]):
            raise ValueError("ve_new must have v_new's shape and ve_gate [B, Tq, Hkv]")
        st = lib.nc_attn_prefill_chunk_ve(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(ve_new), _ptr(ve_gate), _ptr(kcache),
                                          _ptr(vcache), _ptr(cache_lens), _ptr(out), B, Tq, Hq, Hkv, D, Tcap,
                                          int(window), float(rope_base), float(qk_gain), _ptr(workspace), wsb,
                                          _stream(stream))
    else:
        st = lib.nc_attn_prefill_chunk_ex(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache),
                                          _ptr(cache_lens), _ptr(out), B, Tq, Hq, Hkv, D, Tcap, int(window),
                                          float(rope_base), float(qk_gain), _ptr(workspace), wsb, _stream(stream))
    _check(st, "nc_attn_prefill_chunk")
    return out


def nc_attn_decode(q, kcache, vcache, cache_lens, out=None, k_new=None, v_new=None, window=-1,
                   rope_base=ROPE_BASE, workspace=None, stream=None, qk_gain=1.0, ve_new=None, ve_gate=None):
    """Single-token decode.  q [B,Hq,D]; caches [B,Tcap,Hkv,D]; cache_lens int32 [B] (device) -> out [B,Hq,D].

    With k_new / v_new [B,Hkv,D], the new key (roped + normed at cache_lens[b]) and value are written into the caches
    at row cache_lens[b] and attended to.  cache_lens is not modified.  ``ve_new`` [B,Hkv,D] and ``ve_gate`` [B,Hkv]
    (with k_new / v_new): gated value embedding of the new value (``nc_attn_decode_ve``).
    """
    _need(q, "q", 3)
    _need(kcache, "kcache", 4)
    _need(vcache, "vcache", 4)
    _need(cache_lens, "cache_lens", 1, dtype=torch.int32)
    B, Hq, D = q.shape
    _, Tcap, Hkv, _ = kcache.shape
    if tuple(kcache.shape) != (B, Tcap, Hkv, D) or tuple(vcache.shape) != (B, Tcap, Hkv, D):
        raise ValueError("cache shapes do not match q")
    if cache_lens.shape[0] != B:
        raise ValueError("cache_lens must have B entries")
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _need(k_new, "k_new", 3)
        _need(v_new, "v_new", 3)
        if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
            raise ValueError("k_new / v_new must be [B, Hkv, D]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 3)
    nbytes = nc_attn_decode_workspace_bytes(B, Hq, Hkv, D, Tcap, int(window))
    if workspace is None:
        workspace = _workspace("decode", nbytes, q.device, zero=True)
        key = workspace.data_ptr()
        if _ws_decode_tag.get(key, B * Hkv) != B * Hkv:
            workspace.zero_()
        _ws_decode_tag[key] = B * Hkv
    wsb = workspace.numel() * workspace.element_size()
    if ve_new is not None or ve_gate is not None:
        if ve_new is None or ve_gate is None or k_new is None:
            raise ValueError("ve_new and ve_gate go together, with k_new / v_new")
        _need(ve_new, "ve_new", 3)
        _need(ve_gate, "ve_gate", 2)
        if tuple(ve_new.shape) != (B, Hkv, D) or tuple(ve_gate.shape) != (B, Hkv):
            raise ValueError("ve_new must be [B, Hkv, D] and ve_gate [B, Hkv]")
        st = lib.nc_attn_decode_ve(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_lens), _ptr(out), _ptr(k_new),
                                   _ptr(v_new), _ptr(ve_new), _ptr(ve_gate), B, Hq, Hkv, D, Tcap, int(window),
                                   float(rope_base), float(qk_gain), _ptr(workspace), wsb, _stream(stream))
    else:
        st = lib.nc_attn_decode_ex(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_lens), _ptr(out), _ptr(k_new),
                                   _ptr(v_new), B, Hq, Hkv, D, Tcap, int(window), float(rope_base), float(qk_gain),
                                   _ptr(workspace), wsb, _stream(stream))
    _check(st, "nc_attn_decode")
    return out


# Largest decode workspace that nc_attn_decode_noalloc can serve from its fixed device array (bytes).
NC_ATTN_DECODE_NOALLOC_MAX_BYTES = 8 * 1024 * 1024


def nc_attn_decode_noalloc(q, kcache, vcache, cache_lens, out, k_new=None, v_new=None, window=-1,
                           rope_base=ROPE_BASE, stream=None):
    """Single-token decode that allocates nothing, for callers that may not allocate device memory.

    Same arguments and results as ``nc_attn_decode``, except that ``out`` must be given: the split partials live in
    a fixed device array of NC_ATTN_DECODE_NOALLOC_MAX_BYTES bytes inside the library, shared by every call on the
    device, so calls that overlap on the GPU race.  Requests needing a larger workspace raise NcAttnError with
    NC_ERR_SCRATCH_LIMIT.  Make the first call on a device before any stream capture (it looks up the array's
    address).
    """
    _need(q, "q", 3)
    _need(kcache, "kcache", 4)
    _need(vcache, "vcache", 4)
    _need(cache_lens, "cache_lens", 1, dtype=torch.int32)
    _need(out, "out", 3)
    B, Hq, D = q.shape
    _, Tcap, Hkv, _ = kcache.shape
    if tuple(kcache.shape) != (B, Tcap, Hkv, D) or tuple(vcache.shape) != (B, Tcap, Hkv, D):
        raise ValueError("cache shapes do not match q")
    if cache_lens.shape[0] != B or tuple(out.shape) != tuple(q.shape):
        raise ValueError("cache_lens must have B entries and out the shape of q")
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _need(k_new, "k_new", 3)
        _need(v_new, "v_new", 3)
        if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
            raise ValueError("k_new / v_new must be [B, Hkv, D]")
    st = lib.nc_attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_lens), _ptr(out), _ptr(k_new),
                                    _ptr(v_new), B, Hq, Hkv, D, Tcap, int(window), float(rope_base),
                                    _stream(stream))
    _check(st, "nc_attn_decode_noalloc")
    return out


def nc_attn_get_device_status(clear=True, stream=None):
    """Synchronizes the stream and returns the sticky device status code (NC_OK when clean)."""
    return int(lib.nc_attn_get_device_status(_stream(stream), 1 if clear else 0))


def nc_attn_selftest_wait_timeout(limit_us, stream=None):
    _check(lib.nc_attn_selftest_wait_timeout(int(limit_us), _stream(stream)), "nc_attn_selftest_wait_timeout")
