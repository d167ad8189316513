"""nanochat attention block (RoPE -> QK-RMSNorm -> causal GQA with sliding window) on B300 (sm_103a).

The compute lives in ``libnc_attn.so`` (C ABI declared in ``include/nc_attn.h``); ``nc_attn`` is its Python
binding.  Build the library with ``python -m transformer_attention_06_b300.build``.  The binding is loaded on first
use of one of its names, so that the build module can run before the library exists.
"""

_EXPORTS = (
    "NcAttnError",
    "nc_attn_decode",
    "nc_attn_decode_workspace_bytes",
    "nc_attn_bwd",
    "nc_attn_bwd_saved",
    "nc_attn_fwd",
    "nc_attn_fwd_fp8",
    "nc_attn_fwd_lse",
    "nc_attn_fwd_workspace_bytes",
    "nc_attn_get_device_status",
    "nc_attn_qk_prologue",
    "nc_attn_selftest_wait_timeout",
    "status_string",
)


def __getattr__(name):
    if name in _EXPORTS:
        from . import nc_attn
        return getattr(nc_attn, name)
    raise AttributeError(name)
