"""Pins for the oracle's forward and backward (CPU only, tiny sizes).

Each check is independent of oracle.c's arithmetic:
- torch scaled_dot_product_attention in fp64 with an explicit boolean mask
  (built by oracle/brute.py's layout construction), GQA by repeating KV heads;
- special cases that are textbook routines: block_size=1 is causal attention,
  block_size=L is full bidirectional attention;
- each staircase copy equals standalone full attention over [prefix; copy],
  the prefix rows equal block-causal attention over the prefix alone
  (ORL announcement thread, Insight 3; ORL paper card, Figure 3 caption);
- invariants: Q=0 gives the mean of the allowed V rows and LSE = ln(#allowed);
  constant V gives constant O; permuting keys inside a block changes nothing;
- backward: central finite differences of <O, dO> in fp64, torch autograd of
  SDPA, and the NumPy brute force.
"""
import math
import random

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import brute

BC, SC = oracle.BLOCK_CAUSAL, oracle.STAIRCASE


def rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


def sdpa_ref(Q, K, V, M, scale, hkv):
    """torch SDPA, fp64 CPU.  Q [Lq][Hq][d], K/V [Lk][Hkv][d], M [Lq][Lk] bool."""
    Hq = Q.shape[1]
    G = Hq // hkv
    q = Q.permute(1, 0, 2)
    k = K.permute(1, 0, 2).repeat_interleave(G, dim=0)
    v = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
    mask = None if M is None else torch.as_tensor(M)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = (q @ k.transpose(1, 2)) * scale
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(1, 0, 2), lse


def brute_mask(kind, B, P, Lq, Lk):
    if kind == BC:
        return brute.mask_block_causal(Lq, Lk, B)
    return brute.mask_staircase(Lk, B, P)


CASES = [
    # kind, B, P, Lq, Lk, Hq, Hkv, d
    (BC, 4, 0, 16, 16, 2, 1, 8),
    (BC, 3, 0, 17, 17, 4, 2, 8),      # ragged last block, GQA 2
    (BC, 5, 0, 7, 19, 4, 1, 16),      # decode-style Lq < Lk, GQA 4
    (BC, 8, 0, 24, 24, 3, 3, 4),      # MHA
    (SC, 4, 8, 20, 20, 4, 2, 8),      # prefix 8 + 3 copies
    (SC, 3, 7, 16, 16, 2, 1, 8),      # prefix not a multiple of B
    (SC, 2, 0, 8, 8, 2, 2, 4),        # copies only
]


@pytest.mark.parametrize("case", CASES)
def test_fwd_matches_sdpa(case):
    kind, B, P, Lq, Lk, Hq, Hkv, d = case
    Q, K, V = rand((Lq, Hq, d), 1), rand((Lk, Hkv, d), 2), rand((Lk, Hkv, d), 3)
    scale = 0.3
    O, LSE = oracle.fwd_seq(kind, B, P, Q, K, V, Hq, Hkv, scale)
    M = brute_mask(kind, B, P, Lq, Lk)
    Or, Lr = sdpa_ref(Q, K, V, M, scale, Hkv)
    np.testing.assert_allclose(O, Or.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, Lr.numpy(), rtol=0, atol=1e-12)
    Ob, Lb, _ = brute.attention(Q, K, V, M, scale, Hkv)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, Lb, rtol=0, atol=1e-12)


def test_block_size_one_is_causal():
    L, Hq, Hkv, d = 13, 4, 2, 8
    Q, K, V = rand((L, Hq, d), 4), rand((L, Hkv, d), 5), rand((L, Hkv, d), 6)
    O, _ = oracle.fwd_seq(BC, 1, 0, Q, K, V, Hq, Hkv, 0.5)
    G = Hq // Hkv
    o = F.scaled_dot_product_attention(Q.permute(1, 0, 2),
                                       K.permute(1, 0, 2).repeat_interleave(G, 0),
                                       V.permute(1, 0, 2).repeat_interleave(G, 0),
                                       is_causal=True, scale=0.5).permute(1, 0, 2)
    np.testing.assert_allclose(O, o.numpy(), atol=1e-12, rtol=0)


def test_block_size_L_is_full():
    L, Hq, Hkv, d = 11, 2, 1, 8
    Q, K, V = rand((L, Hq, d), 7), rand((L, Hkv, d), 8), rand((L, Hkv, d), 9)
    for B in (L, L + 5):
        O, _ = oracle.fwd_seq(BC, B, 0, Q, K, V, Hq, Hkv, 0.25)
        Or, _ = sdpa_ref(Q, K, V, None, 0.25, Hkv)
        np.testing.assert_allclose(O, Or.numpy(), atol=1e-12, rtol=0)


def test_staircase_copy_is_standalone_attention():
    P, B, Kc, Hq, Hkv, d = 12, 4, 3, 2, 1, 8
    L = P + Kc * B
    Q, K, V = rand((L, Hq, d), 10), rand((L, Hkv, d), 11), rand((L, Hkv, d), 12)
    O, LSE = oracle.fwd_seq(SC, B, P, Q, K, V, Hq, Hkv, 0.4)
    for c in range(Kc):
        s, e = P + c * B, P + (c + 1) * B
        idx = list(range(P)) + list(range(s, e))
        Or, Lr = sdpa_ref(Q[s:e], K[idx], V[idx], None, 0.4, Hkv)
        np.testing.assert_allclose(O[s:e], Or.numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[:, s:e], Lr.numpy(), atol=1e-12, rtol=0)
    # prefix rows = block-causal attention over the prefix alone
    Op, Lp = oracle.fwd_seq(BC, B, 0, Q[:P], K[:P], V[:P], Hq, Hkv, 0.4)
    np.testing.assert_allclose(O[:P], Op, atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE[:, :P], Lp, atol=1e-12, rtol=0)


def test_decode_equals_staircase_single_copy():
    # 32 queries of the active block over a 2048-key committed prefix + the
    # block itself (decode step) == the copy rows of a staircase with P=2048,
    # one copy.  Small heads / head_dim keep it fast.
    P, B, Hq, Hkv, d = 2048, 32, 2, 1, 8
    L = P + B
    Q, K, V = rand((L, Hq, d), 13), rand((L, Hkv, d), 14), rand((L, Hkv, d), 15)
    Od, Ld = oracle.fwd_seq(BC, B, 0, Q[P:], K, V, Hq, Hkv, 0.3)
    Os, Ls = oracle.fwd_seq(SC, B, P, Q, K, V, Hq, Hkv, 0.3, rows=list(range(P, L)))
    np.testing.assert_allclose(Od, Os, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Ld, Ls, atol=1e-12, rtol=0)


@pytest.mark.parametrize("case", CASES)
def test_zero_queries_give_mean_of_allowed_values(case):
    kind, B, P, Lq, Lk, Hq, Hkv, d = case
    Q = torch.zeros((Lq, Hq, d), dtype=torch.float64)
    K, V = rand((Lk, Hkv, d), 16), rand((Lk, Hkv, d), 17)
    O, LSE = oracle.fwd_seq(kind, B, P, Q, K, V, Hq, Hkv, 0.7)
    M = brute_mask(kind, B, P, Lq, Lk)
    G = Hq // Hkv
    for h in range(Hq):
        for i in range(Lq):
            js = np.nonzero(M[i])[0]
            np.testing.assert_allclose(O[i, h], V[js, h // G].numpy().mean(axis=0), atol=1e-12)
            assert abs(LSE[h, i] - math.log(len(js))) < 1e-12


def test_constant_values_give_constant_output():
    kind, B, P, Lq, Lk, Hq, Hkv, d = SC, 4, 8, 20, 20, 4, 2, 8
    Q, K = rand((Lq, Hq, d), 18), rand((Lk, Hkv, d), 19)
    V = torch.ones((Lk, Hkv, d), dtype=torch.float64) * 1.75
    O, _ = oracle.fwd_seq(kind, B, P, Q, K, V, Hq, Hkv, 0.5)
    np.testing.assert_allclose(O, 1.75, atol=1e-13)


def test_key_permutation_inside_block_is_invisible():
    B, L, Hq, Hkv, d = 4, 16, 2, 1, 8
    Q, K, V = rand((L, Hq, d), 20), rand((L, Hkv, d), 21), rand((L, Hkv, d), 22)
    perm = list(range(L))
    rng = random.Random(3)
    for b in range(L // B):
        blk = perm[b * B:(b + 1) * B]
        rng.shuffle(blk)
        perm[b * B:(b + 1) * B] = blk
    O1, L1 = oracle.fwd_seq(BC, B, 0, Q, K, V, Hq, Hkv, 0.5)
    O2, L2 = oracle.fwd_seq(BC, B, 0, Q, K[perm], V[perm], Hq, Hkv, 0.5)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def test_rows_and_heads_subsets_match_full():
    kind, B, P, Lq, Lk, Hq, Hkv, d = SC, 4, 8, 20, 20, 4, 2, 8
    Q, K, V = rand((Lq, Hq, d), 23), rand((Lk, Hkv, d), 24), rand((Lk, Hkv, d), 25)
    O, LSE = oracle.fwd_seq(kind, B, P, Q, K, V, Hq, Hkv, 0.5)
    rows = [19, 0, 7, 8]
    Os, Ls = oracle.fwd_seq(kind, B, P, Q, K, V, Hq, Hkv, 0.5, heads=(2, 4), rows=rows)
    np.testing.assert_allclose(Os[:, 2:], O[rows, 2:], atol=1e-13)
    np.testing.assert_allclose(Ls[2:], LSE[2:, rows], atol=1e-13)
    assert np.isnan(Os[:, :2]).all()


def test_packed_varlen_is_per_sequence():
    lens = [5, 12, 9]
    cu = [0, 5, 17, 26]
    Hq, Hkv, d, B = 2, 1, 8, 4
    T = cu[-1]
    Q, K, V = rand((T, Hq, d), 26), rand((T, Hkv, d), 27), rand((T, Hkv, d), 28)
    O, LSE = oracle.fwd(BC, B, cu, cu, None, Q, K, V, Hq, Hkv, 0.5)
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        M = brute.mask_block_causal(L, L, B)
        Or, Lr = sdpa_ref(Q[a:b], K[a:b], V[a:b], M, 0.5, Hkv)
        np.testing.assert_allclose(O[a:b], Or.numpy(), atol=1e-12)
        np.testing.assert_allclose(LSE[:, a:b], Lr.numpy(), atol=1e-12)


# ---------------------------------------------------------------- backward


def fd_grad(kind, B, P, Q, K, V, dO, Hq, Hkv, scale, which, idx, h=1e-6):
    """Central difference of f = <O, dO> w.r.t. one element of Q, K or V."""
    arrs = {"q": Q.clone(), "k": K.clone(), "v": V.clone()}

    def f(delta):
        a = {n: t.clone() for n, t in arrs.items()}
        a[which][idx] += delta
        O, _ = oracle.fwd_seq(kind, B, P, a["q"], a["k"], a["v"], Hq, Hkv, scale)
        return float((torch.from_numpy(O) * dO).sum())

    return (f(h) - f(-h)) / (2 * h)


@pytest.mark.parametrize("case", [CASES[1], CASES[2], CASES[4], CASES[5]])
def test_bwd_finite_differences(case):
    kind, B, P, Lq, Lk, Hq, Hkv, d = case
    Q, K, V = rand((Lq, Hq, d), 30), rand((Lk, Hkv, d), 31), rand((Lk, Hkv, d), 32)
    dO = rand((Lq, Hq, d), 33)
    scale = 0.45
    dQ, dK, dV = oracle.bwd_seq(kind, B, P, Q, K, V, dO, Hq, Hkv, scale)
    rng = random.Random(4)
    for which, shape, g in (("q", Q.shape, dQ), ("k", K.shape, dK), ("v", V.shape, dV)):
        for _ in range(6):
            idx = tuple(rng.randrange(n) for n in shape)
            num = fd_grad(kind, B, P, Q, K, V, dO, Hq, Hkv, scale, which, idx)
            assert abs(num - g[idx]) <= 1e-6 * max(1.0, abs(num)), (which, idx, num, g[idx])


@pytest.mark.parametrize("case", CASES)
def test_bwd_matches_autograd_and_brute(case):
    kind, B, P, Lq, Lk, Hq, Hkv, d = case
    Q, K, V = rand((Lq, Hq, d), 40), rand((Lk, Hkv, d), 41), rand((Lk, Hkv, d), 42)
    dO = rand((Lq, Hq, d), 43)
    scale = 0.35
    dQ, dK, dV = oracle.bwd_seq(kind, B, P, Q, K, V, dO, Hq, Hkv, scale)
    M = brute_mask(kind, B, P, Lq, Lk)
    q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
    O, _ = sdpa_ref(q, k, v, M, scale, Hkv)
    (O * dO).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-11)
    bq, bk, bv = brute.attention_bwd(Q, K, V, dO, M, scale, Hkv)
    np.testing.assert_allclose(dQ, bq, atol=1e-11)
    np.testing.assert_allclose(dK, bk, atol=1e-11)
    np.testing.assert_allclose(dV, bv, atol=1e-11)


def test_bwd_subsets_and_sum_rules():
    kind, B, P, Lq, Lk, Hq, Hkv, d = SC, 4, 8, 20, 20, 4, 2, 8
    Q, K, V = rand((Lq, Hq, d), 50), rand((Lk, Hkv, d), 51), rand((Lk, Hkv, d), 52)
    dO = rand((Lq, Hq, d), 53)
    dQ, dK, dV = oracle.bwd_seq(kind, B, P, Q, K, V, dO, Hq, Hkv, 0.5)
    q2, k2, v2 = oracle.bwd_seq(kind, B, P, Q, K, V, dO, Hq, Hkv, 0.5, kv_heads=(1, 2),
                                qrows=[3, 19], krows=[0, 17])
    np.testing.assert_allclose(q2[:, 2:], dQ[[3, 19], 2:], atol=1e-13)
    np.testing.assert_allclose(k2[:, 1:], dK[[0, 17], 1:], atol=1e-13)
    np.testing.assert_allclose(v2[:, 1:], dV[[0, 17], 1:], atol=1e-13)
    # sum rules that hold at any size: every row of dS sums to zero, so the
    # keys' dK sum to zero; the rows of P sum to one, so the keys' dV sum to
    # the sum of dO over the group's heads.
    G = Hq // Hkv
    for g in range(Hkv):
        np.testing.assert_allclose(dK[:, g].sum(axis=0), 0.0, atol=1e-12)
        want = dO[:, g * G:(g + 1) * G].sum(dim=(0, 1)).numpy()
        np.testing.assert_allclose(dV[:, g].sum(axis=0), want, atol=1e-12)


def test_rows_are_convex_combinations_and_lse_normalises():
    """Each O row lies inside the box spanned by the V rows it may see, and
    sum_j over the allowed keys of exp(scale q.k - LSE) is 1 (the softmax
    normaliser), for all three mask kinds."""
    Hq, Hkv, d, scale = 4, 2, 8, 0.6
    layouts = [("bc", 4, 0, None, 18), ("sc", 3, 6, None, 15), ("multi", 2, 6, ([2, 1], [2, 6]), 12)]
    for name, B, P, groups, L in layouts:
        Q, K, V = rand((L, Hq, d), 90), rand((L, Hkv, d), 91), rand((L, Hkv, d), 92)
        if name == "bc":
            O, LSE = oracle.fwd_seq(BC, B, 0, Q, K, V, Hq, Hkv, scale)
            M = brute.mask_block_causal(L, L, B)
        elif name == "sc":
            O, LSE = oracle.fwd_seq(SC, B, P, Q, K, V, Hq, Hkv, scale)
            M = brute.mask_staircase(L, B, P)
        else:
            O, LSE = oracle.fwd_seq_multi(B, P, groups[0], groups[1], Q, K, V, Hq, Hkv, scale)
            M = brute.mask_staircase_multi(L, B, P, groups[0], groups[1])
        Qn, Kn, Vn = Q.numpy(), K.numpy(), V.numpy()
        G = Hq // Hkv
        for h in range(Hq):
            for i in range(L):
                vis = np.nonzero(M[i])[0]
                Vv = Vn[vis, h // G, :]
                assert (O[i, h] >= Vv.min(axis=0) - 1e-12).all()
                assert (O[i, h] <= Vv.max(axis=0) + 1e-12).all()
                s = scale * Kn[vis, h // G, :] @ Qn[i, h, :]
                assert abs(np.exp(s - LSE[h, i]).sum() - 1.0) < 1e-12
