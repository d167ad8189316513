"""Plain fp64 definition of the nanochat attention block (test infrastructure only; see ``oracle/__init__``).

What is computed, and where the pages say so:

* RoPE, half-split, base 100000 -- "nanochat Admin & Developer Guide", section 3 "The GPT Model
  (Internals)" (rotary embeddings, base theta 100000); "nanochat (Fucina port)", section "Architecture"
  (the half-split RoPE kernel with an inverse-built frequency table).
* QK-norm: RMSNorm with no learnable weight on every q and k head vector -- Guide section 3 (QK-norm bullet
  and "no learnable params in RMSNorm"); Fucina port, "Architecture" (RMSNorm, no-weight).
* Causal grouped-query attention, n_kv_head <= n_head, scale 1/sqrt(D) -- Guide section 3 (GQA bullet) and
  section 6 "Attention: FA3 with SDPA Fallback" (SDPA with enable_gqa); Fucina port (grouped causal
  attention).
* Per-layer sliding window, passed to Flash Attention as a (left, right) tuple -- Guide section 3,
  "Sliding-window attention".  Reading: key j is visible to query i iff 0 <= i - j <= window; window = -1
  means no left bound (plain causal).
* KV-cache single-token decode -- Guide section 7 "The Inference Engine & Tool Use", "KV cache" (FA3 layout
  (B, T, H, D), per-row int32 cache_seqlens, in-place append) and section 6 (SDPA decode case slices the KV
  window).

Readings where the pages are silent:

* RoPE pairs element i with element i + D/2 (half-split), frequency theta_i = base^(-2i/D), angle t*theta_i,
  and the rotation  y[i] = x[i] cos a + x[i+D/2] sin a,  y[i+D/2] = -x[i] sin a + x[i+D/2] cos a.
  The sign of the rotation is not fixed by any page: parity unpinned for the sign.
* RoPE is applied first and the norm second.  A rotation keeps the sum of squares, so in exact arithmetic
  the order does not matter (pinned by an invariant test).
* RMSNorm epsilon = 1e-6 (not stated on the pages: parity unpinned for its value).
* Grouping: query head h reads kv head h // (Hq / Hkv).
* Decode: the query is at position p = cache_lens[b]; cached keys 0..p-1 are used as given; an optional new
  key/value is roped + normed at position p, written at cache index p, and attended to.  An empty visible set
  gives a zero output row.
"""

import numpy as np

ROPE_BASE = 100000.0
RMS_EPS = 1e-6
# QK_GAIN_NOTE: Guide section 3 (QK-norm bullet): after the norm, q and k carry a combined factor of 1.2, shared
# between them, so every logit is multiplied by 1.2.  ``qk_gain`` is that factor on the logits (1.0: the plain 1/sqrt(D)
# scale of the workloads; 1.2: the sharpened QK-norm).


def inv_freq(D, base=ROPE_BASE):
    """theta_i = base^(-2i/D) for i in [0, D/2): the "inverse-built" RoPE frequency table (fp64)."""
    if D % 2:
        raise ValueError("head dim must be even for half-split RoPE")
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / D)


def rope(x, pos, base=ROPE_BASE):
    """Half-split rotary embedding.

    x:   fp64 array [..., H, D]  (the last two axes are head and head dim)
    pos: positions with shape x.shape[:-2] (one position per token)
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None, None] * inv_freq(D, base)  # [..., 1, D/2]
    c = np.cos(ang)
    s = np.sin(ang)
    x1 = x[..., :h]
    x2 = x[..., h:]
    return np.concatenate([x1 * c + x2 * s, -x1 * s + x2 * c], axis=-1)


def rms_norm(x, eps=RMS_EPS):
    """Weightless RMSNorm over the last axis: y / sqrt(mean(y^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def qk_prologue(x, pos, base=ROPE_BASE, eps=RMS_EPS):
    """RoPE at the given positions, then weightless RMSNorm (the QK-norm)."""
    return rms_norm(rope(x, pos, base), eps)


def visible(i, j, window):
    """Key position j is visible to query position i: causal, and within the window when window >= 0."""
    i = np.asarray(i)
    j = np.asarray(j)
    ok = j <= i
    if window >= 0:
        ok = ok & (i - j <= window)
    return ok


def _softmax_rows(s):
    """Row softmax of a score matrix whose masked entries are -inf (each row has one finite entry at least)."""
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def attn_fwd(q, k, v, window, rope_base=ROPE_BASE, eps=RMS_EPS, chunk=128, qk_gain=1.0, ve=None, ve_gate=None):
    """Prefill / training forward of the attention block.

    q: [B, T, Hq, D], k and v: [B, T, Hkv, D] (any real dtype; computed in fp64).  Positions are 0..T-1.
    Returns out [B, T, Hq, D] fp64.  Query rows are processed in chunks of ``chunk``; for each chunk only the
    keys that can be visible to some row of it are scored (the band), then the exact mask is applied.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = value_mix(v, ve, ve_gate)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    pos = np.broadcast_to(np.arange(T), (B, T))
    qn = qk_prologue(q, pos, rope_base, eps)
    kn = qk_prologue(k, pos, rope_base, eps)
    scale = qk_gain / np.sqrt(D)   # see QK_GAIN_NOTE
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i0 in range(0, T, chunk):
                i1 = min(T, i0 + chunk)
                j0 = 0 if window < 0 else max(0, i0 - window)
                j1 = i1
                s = (qn[b, i0:i1, h] @ kn[b, j0:j1, g].T) * scale
                mask = visible(np.arange(i0, i1)[:, None], np.arange(j0, j1)[None, :], window)
                s = np.where(mask, s, -np.inf)
                out[b, i0:i1, h] = _softmax_rows(s) @ v[b, j0:j1, g]
    return out


def value_mix(v, ve=None, ve_gate=None):
    """Values with the gated value embedding mixed in -- the catalog pages ("nanochat (Python)", "nanochat (.NET)")
    list value embeddings with a sigmoid gate, in the ResFormer manner.  They give no formula; the reading taken is:
    v' = v + sigmoid(g) * ve, with one gate logit g per (token, kv head) and ve of v's shape.  Without ve, v."""
    v = np.asarray(v, dtype=np.float64)
    if ve is None:
        return v
    g = np.asarray(ve_gate, dtype=np.float64)
    return v + (1.0 / (1.0 + np.exp(-g)))[..., None] * np.asarray(ve, dtype=np.float64)


def attn_fwd_rows(q, k, v, window, rows, rope_base=ROPE_BASE, eps=RMS_EPS, qk_gain=1.0):
    """Selected output rows of ``attn_fwd``, one by one (for full-size inputs).

    rows: iterable of (b, i, h).  Returns an fp64 array [len(rows), D].  Each row is computed from scratch:
    the query at position i, the keys of its band for kv head h // G, the exact mask and softmax.
    """
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    scale = qk_gain / np.sqrt(D)   # see QK_GAIN_NOTE
    res = []
    for (b, i, h) in rows:
        g = h // G
        j0 = 0 if window < 0 else max(0, i - window)
        qi = np.asarray(q[b, i, h], dtype=np.float64)[None, None, :]     # [1, 1(head), D]
        qn = qk_prologue(qi, np.array([i]), rope_base, eps)[0, 0]
        kj = np.asarray(k[b, j0:i + 1, g], dtype=np.float64)[:, None, :]  # [n, 1, D]
        kn = qk_prologue(kj, np.arange(j0, i + 1), rope_base, eps)[:, 0]
        s = (kn @ qn) * scale
        p = _softmax_rows(s[None, :])[0]
        res.append(p @ np.asarray(v[b, j0:i + 1, g], dtype=np.float64))
    return np.stack(res) if res else np.zeros((0, D))


def attn_decode(q, kcache, vcache, cache_lens, window, k_new=None, v_new=None,
                rope_base=ROPE_BASE, eps=RMS_EPS, qk_gain=1.0, ve_new=None, ve_gate_new=None):
    """KV-cache single-token decode.

    q: [B, Hq, D] raw query of the new token; kcache, vcache: [B, Tcap, Hkv, D] (rows already roped+normed);
    cache_lens: [B] integers p_b; k_new, v_new: [B, Hkv, D] or None.

    Returns (out [B, Hq, D] fp64, kn_new [B, Hkv, D] fp64 or None).  The query is roped at position p_b and
    normed.  Keys: cache rows 0..p_b-1 as given, plus, when k_new is given, norm(rope(k_new, p_b)) with v_new
    at position p_b.  Visible keys j satisfy p_b - j <= window (window >= 0).  An empty visible set (p_b = 0
    and no new key) gives a zero row.  With ve_new [B, Hkv, D] and ve_gate_new [B, Hkv], the new value is
    ``value_mix(v_new, ve_new, ve_gate_new)`` (the gated value embedding of the new token).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = kcache.shape[2]
    G = Hq // Hkv
    scale = qk_gain / np.sqrt(D)   # see QK_GAIN_NOTE
    out = np.zeros((B, Hq, D), dtype=np.float64)
    kn_new = None
    if ve_new is not None:
        v_new = value_mix(v_new, ve_new, ve_gate_new)
    if k_new is not None:
        kn_new = qk_prologue(np.asarray(k_new, dtype=np.float64)[:, None], np.asarray(cache_lens)[:, None],
                             rope_base, eps)[:, 0]
    for b in range(B):
        p = int(cache_lens[b])
        qn = qk_prologue(q[b][None, None], np.array([[p]]), rope_base, eps)[0, 0]   # [Hq, D]
        keys = np.asarray(kcache[b, :p], dtype=np.float64)
        vals = np.asarray(vcache[b, :p], dtype=np.float64)
        if k_new is not None:
            keys = np.concatenate([keys, kn_new[b][None]], axis=0)
            vals = np.concatenate([vals, np.asarray(v_new[b], dtype=np.float64)[None]], axis=0)
        L = keys.shape[0]
        lo = 0 if window < 0 else max(0, p - window)
        if L - lo <= 0:
            continue
        for h in range(Hq):
            g = h // G
            s = (keys[lo:L, g] @ qn[h]) * scale
            pr = _softmax_rows(s[None, :])[0]
            out[b, h] = pr @ vals[lo:L, g]
    return out, kn_new


def attn_prefill_chunk(q, k_new, v_new, kcache, vcache, cache_lens, window, rope_base=ROPE_BASE, eps=RMS_EPS,
                       qk_gain=1.0, ve_new=None, ve_gate_new=None):
    """Chunked prefill against a KV cache -- Guide section 6 (the SDPA fallback's chunked / sliding-window
    inference case: the chunk's queries attend to the cache plus the chunk) and section 7 "KV cache" (in-place
    append at cache_seqlens).

    q: [B, Tq, Hq, D] raw queries; k_new, v_new: [B, Tq, Hkv, D] raw keys and values of the chunk;
    kcache, vcache: [B, Tcap, Hkv, D] with rows 0..p_b-1 already roped + normed; cache_lens: [B] integers p_b.

    Returns (out [B, Tq, Hq, D] fp64, kn_new [B, Tq, Hkv, D] fp64).  Query t and key t of the chunk sit at
    position p_b + t.  The keys of sequence b are its cache rows 0..p_b-1 as given followed by
    norm(rope(k_new[b, t], p_b + t)), with the values vcache[b, :p_b] followed by v_new[b]; key position j is
    visible to query position i under ``visible``.  A p_b outside [0, Tcap - Tq] gives zero rows (and a zero
    kn_new) for that sequence.  With ve_new [B, Tq, Hkv, D] and ve_gate_new [B, Tq, Hkv], the chunk's values are
    ``value_mix(v_new, ve_new, ve_gate_new)`` (the gated value embedding of its tokens).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Tq, Hq, D = q.shape
    Hkv = k_new.shape[2]
    Tcap = kcache.shape[1]
    v_new = value_mix(v_new, ve_new, ve_gate_new)
    G = Hq // Hkv
    scale = qk_gain / np.sqrt(D)   # see QK_GAIN_NOTE
    out = np.zeros((B, Tq, Hq, D), dtype=np.float64)
    kn_new = np.zeros((B, Tq, Hkv, D), dtype=np.float64)
    for b in range(B):
        p = int(cache_lens[b])
        if p < 0 or p + Tq > Tcap:
            continue
        pos = p + np.arange(Tq)
        qn = qk_prologue(q[b][None], pos[None], rope_base, eps)[0]                                   # [Tq, Hq, D]
        kn_new[b] = qk_prologue(np.asarray(k_new[b], dtype=np.float64)[None], pos[None], rope_base, eps)[0]
        keys = np.concatenate([np.asarray(kcache[b, :p], dtype=np.float64), kn_new[b]], axis=0)      # [p+Tq, Hkv, D]
        vals = np.concatenate([np.asarray(vcache[b, :p], dtype=np.float64),
                               np.asarray(v_new[b], dtype=np.float64)], axis=0)
        mask = visible(pos[:, None], np.arange(p + Tq)[None, :], window)
        for h in range(Hq):
            g = h // G
            s = np.where(mask, (qn[:, h] @ keys[:, g].T) * scale, -np.inf)
            out[b, :, h] = _softmax_rows(s) @ vals[:, g]
    return out, kn_new
