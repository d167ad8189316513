"""Scalar-loop oracle for tiny inputs (test infrastructure only; see ``oracle/__init__``).

Same definition as ``oracle.ref`` (nanochat Admin & Developer Guide, sections 3 and 6; nanochat (Fucina
port), "Architecture"), written out element by element with the ``math`` module: every rotation pair, every
square in the norm, the full T x T score matrix, an explicit boolean mask and an explicit softmax.  It is the
brute-force pin for ``oracle.ref``.
"""

import math


def _rope_norm_vec(x, pos, base, eps):
    D = len(x)
    h = D // 2
    y = [0.0] * D
    for i in range(h):
        theta = base ** (-2.0 * i / D)
        a = pos * theta
        c = math.cos(a)
        s = math.sin(a)
        x1 = float(x[i])
        x2 = float(x[i + h])
        y[i] = x1 * c + x2 * s
        y[i + h] = -x1 * s + x2 * c
    ms = 0.0
    for e in y:
        ms += e * e
    ms /= D
    r = math.sqrt(ms + eps)
    return [e / r for e in y]


def attn_fwd_brute(q, k, v, window, rope_base=100000.0, eps=1e-6):
    """q [B][T][Hq][D], k/v [B][T][Hkv][D] nested sequences (or arrays).  Returns nested lists [B][T][Hq][D]."""
    B = len(q)
    T = len(q[0])
    Hq = len(q[0][0])
    D = len(q[0][0][0])
    Hkv = len(k[0][0])
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    out = [[[[0.0] * D for _ in range(Hq)] for _ in range(T)] for _ in range(B)]
    for b in range(B):
        qn = [[_rope_norm_vec(q[b][t][h], t, rope_base, eps) for h in range(Hq)] for t in range(T)]
        kn = [[_rope_norm_vec(k[b][t][g], t, rope_base, eps) for g in range(Hkv)] for t in range(T)]
        for h in range(Hq):
            g = h // G
            # full score matrix and explicit mask
            S = [[sum(qn[i][h][d] * kn[j][g][d] for d in range(D)) * scale for j in range(T)] for i in range(T)]
            M = [[(j <= i) and (window < 0 or i - j <= window) for j in range(T)] for i in range(T)]
            for i in range(T):
                mx = max(S[i][j] for j in range(T) if M[i][j])
                e = [math.exp(S[i][j] - mx) if M[i][j] else 0.0 for j in range(T)]
                z = sum(e)
                for d in range(D):
                    out[b][i][h][d] = sum(e[j] / z * float(v[b][j][g][d]) for j in range(T))
    return out


def attn_decode_brute(q, kcache, vcache, cache_lens, window, k_new=None, v_new=None,
                      rope_base=100000.0, eps=1e-6):
    """Scalar decode: q [B][Hq][D], caches [B][Tcap][Hkv][D], cache_lens [B].  Returns nested [B][Hq][D]."""
    B = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(kcache[0][0])
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        p = int(cache_lens[b])
        keys = [[list(map(float, kcache[b][j][g])) for g in range(Hkv)] for j in range(p)]
        vals = [[list(map(float, vcache[b][j][g])) for g in range(Hkv)] for j in range(p)]
        if k_new is not None:
            keys.append([_rope_norm_vec(k_new[b][g], p, rope_base, eps) for g in range(Hkv)])
            vals.append([list(map(float, v_new[b][g])) for g in range(Hkv)])
        for h in range(Hq):
            g = h // G
            qn = _rope_norm_vec(q[b][h], p, rope_base, eps)
            vis = [j for j in range(len(keys)) if (window < 0 or p - j <= window)]
            if not vis:
                continue
            s = {j: sum(qn[d] * keys[j][g][d] for d in range(D)) * scale for j in vis}
            mx = max(s.values())
            e = {j: math.exp(s[j] - mx) for j in vis}
            z = sum(e.values())
            for d in range(D):
                out[b][h][d] = sum(e[j] / z * vals[j][g][d] for j in vis)
    return out
