"""The layer-pattern helper (host logic, CPU only)."""

import pytest

from transformer_attention_06_b300.windows import window_sizes


def test_sssl_is_tiled_and_the_last_layer_is_full():
    w = window_sizes("SSSL", 12, 1024)
    assert w == [1024, 1024, 1024, -1] * 3
    # a pattern that would end on S still ends on L
    assert window_sizes("SSSL", 7, 512) == [512, 512, 512, -1, 512, 512, -1]
    assert window_sizes("S", 3, 100) == [100, 100, -1]


def test_all_full_and_case():
    assert window_sizes("L", 5, 1024) == [-1] * 5
    assert window_sizes("ssl", 3, 64) == [64, 64, -1]
    assert window_sizes("SL", 1, 64) == [-1]


def test_the_depth12_step_matches_its_windows():
    # the depth-12 bench step (T = 2048): SSSL with half-context short windows; -1 and 2048 are the same window there
    w = window_sizes("SSSL", 4, 1024)
    assert [2048 if x < 0 else x for x in w] == [1024, 1024, 1024, 2048]


@pytest.mark.parametrize("args", [("", 4, 10), ("SXL", 4, 10), ("SL", 0, 10), ("SL", 4, -1), (None, 4, 10)])
def test_bad_arguments(args):
    with pytest.raises(ValueError):
        window_sizes(*args)
