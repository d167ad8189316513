"""Host logic of the measurement: the in-band FLOP and byte counts bench.py divides by, against direct counting."""

import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_counts", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def visible_pairs(T, W, p0=0, Tq=None):
    """(query, key) pairs visible under the causal / window rule, by enumeration."""
    Tq = T if Tq is None else Tq
    n = 0
    for t in range(Tq):
        a = p0 + t
        for j in range(a + 1):
            n += W < 0 or a - j <= W
    return n


@pytest.mark.parametrize("T,W", [(1, -1), (7, -1), (7, 0), (7, 3), (7, 6), (7, 100), (130, 64), (257, 128)])
def test_n_vis_and_forward_flops(T, W):
    assert bench.n_vis(T, W) == visible_pairs(T, W)
    assert bench.fwd_flops(2, T, 3, 128, W) == 4 * 128 * visible_pairs(T, W) * 2 * 3


@pytest.mark.parametrize("Tq,p0,W", [(5, 0, -1), (5, 9, -1), (5, 9, 2), (40, 100, 30), (1, 3, 0)])
def test_chunk_flops(Tq, p0, W):
    assert bench.chunk_flops(3, Tq, p0, 2, 128, W) == 4 * 128 * visible_pairs(None, W, p0, Tq) * 3 * 2


def test_decode_bytes():
    # two sequences: 10 cached rows (window 4: rows 6..9 visible) and 3 rows (all visible), Hq=4, Hkv=2, D=128
    lens, W, B, Hq, Hkv, D = [10, 3], 4, 2, 4, 2, 128
    rows = 4 + 3
    base = rows * Hkv * D * 2 * 2 + 2 * B * Hq * D * 2 + 4 * B
    assert bench.decode_bytes(lens, W, B, Hq, Hkv, D, False) == base
    # with a new key at position p the window is p - W .. p: the same cache rows are read (6..9 and 0..2), and the new
    # key and value are read from k_new / v_new and written into the cache
    assert bench.decode_bytes(lens, W, B, Hq, Hkv, D, True) == (
        rows * Hkv * D * 2 * 2 + 2 * B * Hq * D * 2 + 4 * B + 2 * (B * Hkv * D * 2) * 2)
    assert bench.decode_bytes([0], -1, 1, 1, 1, 128, False) == 2 * 1 * 1 * 128 * 2 + 4
