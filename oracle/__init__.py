"""fp64 CPU oracle for the nanochat attention block.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The product path (the CUDA library
under ``transformer_attention_06_b300/`` and its Python binding) never imports it, and this package
imports nothing from the product path.

Modules:

* ``ref``   -- numpy fp64, blocked over query chunks so that only the causal / sliding-window band is
               computed.  The reference for every parity test.
* ``brute`` -- scalar Python loops with an explicit full score matrix and mask.  Tiny inputs only; it pins
               ``ref`` (brute force on tiny inputs).
* ``fp8``   -- the prefill forward with its score contraction on e4m3 operands (per-tensor scales fixed by the
               QK-norm); pinned by the e4m3 code table, exhaustive nearest search, torch's float8 cast and
               brute force (``tests/test_oracle_fp8.py``).
* ``backward`` -- the chain rule of the block in fp64; pinned by central finite differences.

Parity status: every function here is pinned by ``tests/test_oracle.py`` (closed forms, brute force,
invariants), except two documented readings that no page decides: the sign of the RoPE rotation and the
RMSNorm epsilon (1e-6).  For those two, "parity unpinned" applies: the oracle and the CUDA path make the
same documented choice, and a discriminator test shows that the other choice would fail parity.
"""

from .ref import (  # noqa: F401
    RMS_EPS,
    ROPE_BASE,
    attn_decode,
    attn_fwd,
    attn_fwd_rows,
    inv_freq,
    qk_prologue,
    rms_norm,
    rope,
    visible,
)
