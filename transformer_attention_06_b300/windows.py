"""Per-layer attention windows from a layer pattern (host-side configuration for ``nc_attn_fwd``'s ``window``).

"nanochat Admin & Developer Guide", section 3, "Sliding-window attention": the pattern string (L = full context,
S = short window; nanochat's default is SSSL) is tiled across the layers, and the final layer is always L whatever
the pattern says.  The same section describes the short window as a quarter of the context rounded up to a multiple
of 128, but its example (2048 -> 768) does not follow that rule, so the short window is an argument here; the
nanochat workloads in this package use half the context (1024 for 2048).
"""


def window_sizes(pattern, n_layer, short_window):
    """Window argument of each of ``n_layer`` layers: -1 (unbounded causal) for L, ``short_window`` for S.

    ``pattern``: non-empty string of 'S' and 'L' (either case), repeated as often as needed; the last layer is L.
    """
    if not isinstance(pattern, str) or not pattern:
        raise ValueError("pattern must be a non-empty string of 'S' and 'L'")
    p = pattern.upper()
    if set(p) - {"S", "L"}:
        raise ValueError(f"pattern {pattern!r} may only hold 'S' and 'L'")
    if n_layer < 1:
        raise ValueError("n_layer must be at least 1")
    if short_window < 0:
        raise ValueError("short_window must be >= 0")
    out = [short_window if p[i % len(p)] == "S" else -1 for i in range(n_layer)]
    out[-1] = -1
    return out
