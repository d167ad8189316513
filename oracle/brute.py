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


def _e4m3_values():
    """Every finite float8_e4m3fn value with its code, from the bit layout: sign, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent field 0 holds the subnormals m * 2^-9; S.1111.111 is NaN."""
    vals = []
    for code in range(256):
        e, m = (code >> 3) & 0xF, code & 7
        if e == 0xF and m == 7:
            continue
        mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append((-mag if code & 0x80 else mag, code))
    return vals


_E4M3 = _e4m3_values()


def e4m3_nearest(x):
    """Nearest finite e4m3 value to x by exhaustive search; on a tie the value whose mantissa (lowest code bit) is
    even."""
    best = None
    for val, code in _E4M3:
        d = abs(val - x)
        if best is None or d < best[0] or (d == best[0] and (code & 1) == 0 and (best[2] & 1) == 1):
            best = (d, val, code)
    return best[1]


def attn_fwd_fp8_brute(q, k, v, window, s_q, s_k, rope_base=100000.0, eps=1e-6):
    """Scalar version of the fp8 prefill: qn * s_q and kn * s_k rounded to e4m3 element by element (exhaustive
    nearest search), the full score matrix of the quantised vectors divided by s_q s_k and scaled by 1 / sqrt(D), an
    explicit mask and softmax, values as given."""
    B, T, Hq, D, Hkv = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0]), len(k[0][0])
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    out = [[[[0.0] * D for _ in range(Hq)] for _ in range(T)] for _ in range(B)]
    for b in range(B):
        qn = [[[e4m3_nearest(x * s_q) for x in _rope_norm_vec(q[b][t][h], t, rope_base, eps)] for h in range(Hq)]
              for t in range(T)]
        kn = [[[e4m3_nearest(x * s_k) for x in _rope_norm_vec(k[b][t][g], t, rope_base, eps)] for g in range(Hkv)]
              for t in range(T)]
        for h in range(Hq):
            g = h // G
            for i in range(T):
                vis = [j for j in range(T) if j <= i and (window < 0 or i - j <= window)]
                s = {j: sum(qn[i][h][d] * kn[j][g][d] for d in range(D)) / (s_q * s_k) * scale for j in vis}
                mx = max(s.values())
                e = {j: math.exp(s[j] - mx) for j in vis}
                z = sum(e.values())
                for d in range(D):
                    out[b][i][h][d] = sum(e[j] / z * float(v[b][j][g][d]) for j in vis)
    return out
