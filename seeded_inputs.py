"""Seeded synthetic inputs and workload shapes shared by the oracle side and the CUDA side.

This module holds no arithmetic of the attention block: it only draws random tensors and names the
workloads.  Recipe (the same bf16 tensors go to both sides):

* ``torch.Generator('cpu').manual_seed(seed)``;
* ``torch.randn(shape, dtype=float32, generator=g)`` in the order q, k, v (prefill) or
  k-cache, v-cache, cache lengths, q, [k_new, v_new] (decode);
* each draw is rounded to bfloat16 (round-to-nearest-even) with ``.to(torch.bfloat16)``;
* decode cache lengths: ``torch.randint(lo, hi + 1, (B,), generator=g)`` (uniform on [lo, hi]);
* chunked prefill: k-cache, v-cache, q, k_new, v_new in that order; the cache lengths are given, not drawn;
* backward: q, k, v, then the upstream gradient dout.

Values are N(0, 1), the distribution the nanochat workloads below are quoted with.  Shapes follow nanochat
configurations (depth 12 gives model dim 768 = 6 heads of 128; GQA and long-context variants).
"""

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class FwdWorkload:
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    windows: tuple   # one attention call per entry (a layer pattern); -1 = unbounded causal


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Tcap: int
    window: int
    len_lo: int
    len_hi: int


# Prefill / training-forward workloads.  "depth12_sssl" is one pass over the SSSL layer pattern (three
# short-window layers, one full-context layer).
TINY = FwdWorkload("tiny_b1_t256_hq4_hkv2", 1, 256, 4, 2, 128, (128, 256))
DEPTH12 = FwdWorkload("depth12_sssl_b4_t2048_h6", 4, 2048, 6, 6, 128, (1024, 1024, 1024, 2048))
GQA = FwdWorkload("gqa_b8_t2048_hq16_hkv4", 8, 2048, 16, 4, 128, (1024, 2048))
LONG = FwdWorkload("long_b2_t8192_hq12_hkv4", 2, 8192, 12, 4, 128, (1024, 8192))
FWD_WORKLOADS = (TINY, DEPTH12, GQA, LONG)

# Decode workload: 64 sequences, cache lengths uniform on [1, 4096], window 2048.  Tcap = 4097 leaves room to
# append one new key at the longest length.
DECODE = DecodeWorkload("decode_b64_hq12_hkv4_w2048", 64, 12, 4, 128, 4097, 2048, 1, 4096)


@dataclass(frozen=True)
class ChunkWorkload:
    name: str
    B: int
    Tq: int
    Hq: int
    Hkv: int
    D: int
    Tcap: int
    p0: int          # cache length of every sequence when the chunk arrives
    windows: tuple


# Chunked prefill: the last 512 tokens of a 2048-token depth-12 context appended to a cache holding the first
# 1536, once with a short-window layer's window and once with the full-context layer's.
CHUNK = ChunkWorkload("chunk_depth12_b4_tq512_p1536", 4, 512, 6, 6, 128, 2048, 1536, (1024, 2048))


def _randn(shape, g):
    return torch.randn(shape, dtype=torch.float32, generator=g).to(torch.bfloat16)


def fwd_inputs(B, T, Hq, Hkv, D, seed=0):
    """q [B,T,Hq,D], k [B,T,Hkv,D], v [B,T,Hkv,D]: bf16 CPU tensors, N(0,1)."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = _randn((B, T, Hq, D), g)
    k = _randn((B, T, Hkv, D), g)
    v = _randn((B, T, Hkv, D), g)
    return q, k, v


def decode_inputs(B, Hq, Hkv, D, Tcap, len_lo, len_hi, seed=0, with_new=False):
    """Decode inputs as bf16 CPU tensors (cache lengths int32).

    Returns dict with kcache, vcache [B,Tcap,Hkv,D], cache_lens [B], q [B,Hq,D], and k_new, v_new [B,Hkv,D]
    when ``with_new`` (else None).
    """
    gen = torch.Generator("cpu").manual_seed(seed)
    kcache = _randn((B, Tcap, Hkv, D), gen)
    vcache = _randn((B, Tcap, Hkv, D), gen)
    cache_lens = torch.randint(len_lo, len_hi + 1, (B,), generator=gen, dtype=torch.int64).to(torch.int32)
    q = _randn((B, Hq, D), gen)
    k_new = v_new = None
    if with_new:
        k_new = _randn((B, Hkv, D), gen)
        v_new = _randn((B, Hkv, D), gen)
    return dict(kcache=kcache, vcache=vcache, cache_lens=cache_lens, q=q, k_new=k_new, v_new=v_new)


def chunk_inputs(B, Tq, Hq, Hkv, D, Tcap, seed=0):
    """Chunked-prefill inputs as bf16 CPU tensors: kcache, vcache [B,Tcap,Hkv,D] (taken as already roped and
    normed, like the decode cache), q [B,Tq,Hq,D], k_new, v_new [B,Tq,Hkv,D]."""
    gen = torch.Generator("cpu").manual_seed(seed)
    kcache = _randn((B, Tcap, Hkv, D), gen)
    vcache = _randn((B, Tcap, Hkv, D), gen)
    q = _randn((B, Tq, Hq, D), gen)
    k_new = _randn((B, Tq, Hkv, D), gen)
    v_new = _randn((B, Tq, Hkv, D), gen)
    return dict(kcache=kcache, vcache=vcache, q=q, k_new=k_new, v_new=v_new)


def bwd_inputs(B, T, Hq, Hkv, D, seed=0):
    """Backward inputs as bf16 CPU tensors: q [B,T,Hq,D], k, v [B,T,Hkv,D] and the upstream gradient dout [B,T,Hq,D]."""
    gen = torch.Generator("cpu").manual_seed(seed)
    q = _randn((B, T, Hq, D), gen)
    k = _randn((B, T, Hkv, D), gen)
    v = _randn((B, T, Hkv, D), gen)
    dout = _randn((B, T, Hq, D), gen)
    return q, k, v, dout
