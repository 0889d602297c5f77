"""Pins for the oracle's multi-block staircase (CPU only, tiny sizes).

Several active blocks per trajectory (ORL announcement thread, 24vids.com
mirror, Insight 3: "irregular trajectories" replayed by the staircase kernel;
ORL paper card, Figure 3 caption): after the block-causal clean prefix come
groups of copies, one group per active block; a group's copies see the clean
keys before their block and themselves only.  Checks independent of oracle.c:
- hand-drawn masks (tests/golden/masks_multi.txt);
- oracle/brute.py's layout construction, exhaustively on random layouts;
- one group that sees the whole prefix is the single-block staircase;
- the closed-form pair count;
- every copy equals standalone attention (torch SDPA, fp64) over its visible
  clean keys and itself; the prefix rows equal block-causal attention over
  the prefix alone;
- backward against torch autograd of SDPA with the constructed mask, the NumPy
  brute force, and central finite differences.
"""
import os
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

from test_oracle_attn import rand, sdpa_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "masks_multi.txt")


def load_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.rstrip("\n")
        if not line or line.startswith("#"):
            continue
        if line.startswith("case "):
            parts = line.split()
            meta = dict(p.split("=") for p in parts[2:])
            cur = dict(name=parts[1], B=int(meta["B"]), P=int(meta["P"]), L=int(meta["L"]),
                       copies=[int(x) for x in meta["copies"].split(",")],
                       visible=[int(x) for x in meta["visible"].split(",")], rows=[])
            cases.append(cur)
        else:
            cur["rows"].append([c == "x" for c in line])
    for c in cases:
        assert len(c["rows"]) == c["L"] and all(len(r) == c["L"] for r in c["rows"]), c["name"]
    return cases


GOLD = load_golden()


@pytest.mark.parametrize("case", GOLD, ids=[c["name"] for c in GOLD])
def test_multi_mask_matches_hand_drawn(case):
    args = (case["B"], case["P"], case["copies"], case["visible"], case["L"])
    assert (oracle.mask_multi(*args) == np.array(case["rows"])).all()
    m = brute.mask_staircase_multi(case["L"], case["B"], case["P"], case["copies"],
                                   case["visible"])
    assert (m == np.array(case["rows"])).all()


def random_layout(rng):
    B = rng.randint(1, 5)
    P = rng.randint(0, 13)
    copies = [rng.randint(0, 3) for _ in range(rng.randint(0, 4))]
    visible = [rng.randint(0, P) for _ in copies]
    L = P + B * sum(copies)
    return B, P, copies, visible, L


def closed_form_pairs(B, P, copies, visible):
    prefix = sum(min(P, (p // B + 1) * B) for p in range(P))
    return prefix + sum(n * B * (v + B) for n, v in zip(copies, visible))


def test_multi_mask_exhaustive_vs_construction():
    rng = random.Random(21)
    for _ in range(400):
        B, P, copies, visible, L = random_layout(rng)
        if L == 0:
            continue
        m = oracle.mask_multi(B, P, copies, visible, L)
        assert (m == brute.mask_staircase_multi(L, B, P, copies, visible)).all()
        assert oracle.count_pairs_multi(B, P, copies, visible, L) == \
            closed_form_pairs(B, P, copies, visible) == m.sum()


def test_single_group_seeing_the_prefix_is_the_staircase():
    rng = random.Random(22)
    for _ in range(100):
        B, P, K = rng.randint(1, 5), rng.randint(0, 13), rng.randint(0, 4)
        L = P + B * K
        if L == 0:
            continue
        m = oracle.mask_multi(B, P, [K], [P], L)
        assert (m == oracle.mask(oracle.STAIRCASE, B, P, L, L)).all()
    B, P, K, Hq, Hkv, d = 3, 7, 3, 4, 2, 8
    L = P + K * B
    Q, K_, V = rand((L, Hq, d), 60), rand((L, Hkv, d), 61), rand((L, Hkv, d), 62)
    O1, L1 = oracle.fwd_seq_multi(B, P, [K], [P], Q, K_, V, Hq, Hkv, 0.3)
    O2, L2 = oracle.fwd_seq(oracle.STAIRCASE, B, P, Q, K_, V, Hq, Hkv, 0.3)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_copies_are_standalone_attention():
    B, P, Hq, Hkv, d = 4, 12, 4, 2, 8
    copies, visible = [2, 0, 3], [4, 8, 12]
    L = P + B * sum(copies)
    Q, K, V = rand((L, Hq, d), 63), rand((L, Hkv, d), 64), rand((L, Hkv, d), 65)
    O, LSE = oracle.fwd_seq_multi(B, P, copies, visible, Q, K, V, Hq, Hkv, 0.4)
    s = P
    for n, vis in zip(copies, visible):
        for _ in range(n):
            idx = list(range(vis)) + list(range(s, s + B))
            Or, Lr = sdpa_ref(Q[s:s + B], K[idx], V[idx], None, 0.4, Hkv)
            np.testing.assert_allclose(O[s:s + B], Or.numpy(), atol=1e-12, rtol=0)
            np.testing.assert_allclose(LSE[:, s:s + B], Lr.numpy(), atol=1e-12, rtol=0)
            s += B
    assert s == L
    Op, Lp = oracle.fwd_seq(oracle.BLOCK_CAUSAL, B, 0, Q[:P], K[:P], V[:P], Hq, Hkv, 0.4)
    np.testing.assert_allclose(O[:P], Op, atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE[:, :P], Lp, atol=1e-12, rtol=0)


MULTI = [
    # B, P, copies, visible, Hq, Hkv, d
    (4, 12, [2, 1], [4, 12], 4, 2, 8),
    (3, 7, [1, 0, 2], [0, 3, 7], 2, 1, 8),  # a group that sees no clean key
    (2, 0, [3], [0], 2, 2, 4),             # copies only
]


@pytest.mark.parametrize("case", MULTI)
def test_multi_fwd_bwd_match_sdpa_autograd_and_brute(case):
    B, P, copies, visible, Hq, Hkv, d = case
    L = P + B * sum(copies)
    Q, K, V = rand((L, Hq, d), 70), rand((L, Hkv, d), 71), rand((L, Hkv, d), 72)
    dO = rand((L, Hq, d), 73)
    scale = 0.35
    M = brute.mask_staircase_multi(L, B, P, copies, visible)
    O, LSE = oracle.fwd_seq_multi(B, P, copies, visible, Q, K, V, Hq, Hkv, scale)
    Or, Lr = sdpa_ref(Q, K, V, M, scale, Hkv)
    np.testing.assert_allclose(O, Or.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, Lr.numpy(), atol=1e-12, rtol=0)
    dQ, dK, dV = oracle.bwd_seq_multi(B, P, copies, visible, Q, K, V, dO, Hq, Hkv, scale)
    q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
    Oa, _ = sdpa_ref(q, k, v, M, scale, Hkv)
    (Oa * dO).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-11)
    bq, bk, bv = brute.attention_bwd(Q, K, V, dO, M, scale, Hkv)
    np.testing.assert_allclose(dQ, bq, atol=1e-11)
    np.testing.assert_allclose(dK, bk, atol=1e-11)
    np.testing.assert_allclose(dV, bv, atol=1e-11)


def test_multi_bwd_finite_differences():
    B, P, copies, visible, Hq, Hkv, d = 3, 6, [2, 1], [3, 6], 2, 1, 4
    L = P + B * sum(copies)
    Q, K, V = rand((L, Hq, d), 80), rand((L, Hkv, d), 81), rand((L, Hkv, d), 82)
    dO = rand((L, Hq, d), 83)
    scale = 0.5
    dQ, dK, dV = oracle.bwd_seq_multi(B, P, copies, visible, Q, K, V, dO, Hq, Hkv, scale)
    arrs = {"q": Q, "k": K, "v": V}

    def f(which, idx, delta):
        a = {n: t.clone() for n, t in arrs.items()}
        a[which][idx] += delta
        O, _ = oracle.fwd_seq_multi(B, P, copies, visible, a["q"], a["k"], a["v"], Hq, Hkv, scale)
        return float((torch.from_numpy(O) * dO).sum())

    rng = random.Random(5)
    h = 1e-6
    for which, g in (("q", dQ), ("k", dK), ("v", dV)):
        for _ in range(6):
            idx = tuple(rng.randrange(n) for n in arrs[which].shape)
            num = (f(which, idx, h) - f(which, idx, -h)) / (2 * h)
            assert abs(num - g[idx]) <= 1e-6 * max(1.0, abs(num)), (which, idx, num, g[idx])


def test_multi_rejects_layouts_that_do_not_tile():
    with pytest.raises(ValueError):
        oracle.mask_multi(2, 4, [1], [4], 8)  # copies cover [4, 6), not [4, 8)
    with pytest.raises(ValueError):
        oracle.mask_multi(2, 4, [2], [5], 8)  # a group seeing past the prefix
