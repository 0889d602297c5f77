"""NumPy brute force for tiny inputs (test infrastructure only).

Independent of oracle.c: the mask is built by *constructing the layout* --
walking the blocks, the prefix and the copies and marking what each one may
see -- rather than by evaluating a per-element predicate, and the attention is
done with whole-matrix NumPy operations.  Used to pin the C oracle on tiny
inputs (L <= 64 or so).

Block-causal: ORL announcement thread (24vids.com mirror), highlight 3.
Staircase: same thread, Insight 3; ORL paper card (thelatestinai.com),
Figure 3 caption.
"""
import numpy as np


def blocks(n, B):
    """[start, end) of consecutive blocks of B tokens covering [0, n)."""
    return [(s, min(s + B, n)) for s in range(0, n, B)]


def mask_block_causal(Lq, Lk, B):
    """Queries are the last Lq key positions; a query in block b sees blocks 0..b."""
    M = np.zeros((Lq, Lk), dtype=bool)
    kb = blocks(Lk, B)
    off = Lk - Lq
    for b, (s, e) in enumerate(kb):
        visible = np.zeros(Lk, dtype=bool)
        for (s2, e2) in kb[: b + 1]:
            visible[s2:e2] = True
        for p in range(s, e):
            if p - off >= 0:
                M[p - off] = visible
    return M


def mask_staircase(L, B, P):
    """Prefix of P tokens, block-causal inside itself; then (L-P)/B copies of
    B tokens; each copy sees the whole prefix and itself."""
    assert (L - P) % B == 0
    M = np.zeros((L, L), dtype=bool)
    pb = blocks(P, B)
    for b, (s, e) in enumerate(pb):
        for (s2, e2) in pb[: b + 1]:
            M[s:e, s2:e2] = True
    for c in range((L - P) // B):
        s, e = P + c * B, P + (c + 1) * B
        M[s:e, :P] = True
        M[s:e, s:e] = True
    return M


def mask_staircase_multi(L, B, P, copies, visible):
    """Prefix of P tokens, block-causal inside itself; then, group after
    group, copies[g] copies of B tokens, each seeing the clean keys
    [0, visible[g]) and itself."""
    M = np.zeros((L, L), dtype=bool)
    pb = blocks(P, B)
    for b, (s, e) in enumerate(pb):
        for (s2, e2) in pb[: b + 1]:
            M[s:e, s2:e2] = True
    s = P
    for n, vis in zip(copies, visible):
        for _ in range(n):
            M[s:s + B, :vis] = True
            M[s:s + B, s:s + B] = True
            s += B
    assert s == L
    return M


def attention(Q, K, V, M, scale, hkv):
    """Q [Lq][Hq][d], K/V [Lk][Hkv][d], M [Lq][Lk] bool.  fp64 dense.
    Returns O [Lq][Hq][d], LSE [Hq][Lq], P [Hq][Lq][Lk]."""
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    Lq, Hq, d = Q.shape
    G = Hq // hkv
    O = np.zeros_like(Q)
    LSE = np.zeros((Hq, Lq))
    Pall = np.zeros((Hq, Lq, K.shape[0]))
    for h in range(Hq):
        g = h // G
        S = scale * Q[:, h, :] @ K[:, g, :].T
        S = np.where(M, S, -np.inf)
        mx = S.max(axis=1, keepdims=True)
        E = np.exp(S - mx)
        Z = E.sum(axis=1, keepdims=True)
        Pm = E / Z
        O[:, h, :] = Pm @ V[:, g, :]
        LSE[h] = (mx + np.log(Z))[:, 0]
        Pall[h] = Pm
    return O, LSE, Pall


def attention_bwd(Q, K, V, dO, M, scale, hkv):
    """Matrix-form gradients of sum(O * dO).  Returns dQ, dK, dV (fp64)."""
    Q, K, V, dO = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, dO))
    O, _, Pall = attention(Q, K, V, M, scale, hkv)
    Lq, Hq, d = Q.shape
    G = Hq // hkv
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for h in range(Hq):
        g = h // G
        Pm = Pall[h]
        dV[:, g, :] += Pm.T @ dO[:, h, :]
        dP = dO[:, h, :] @ V[:, g, :].T
        D = (dO[:, h, :] * O[:, h, :]).sum(axis=1, keepdims=True)
        dS = Pm * (dP - D)
        dQ[:, h, :] = scale * dS @ K[:, g, :]
        dK[:, g, :] += scale * dS.T @ Q[:, h, :]
    return dQ, dK, dV
