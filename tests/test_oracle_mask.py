"""Pins for the oracle's mask predicate and pair count (CPU only).

- hand-drawn masks (tests/golden/masks.txt) drawn from the sources' wording:
  ORL announcement thread (24vids.com mirror), highlight 3 (block-causal) and
  Insight 3 (staircase); ORL paper card (thelatestinai.com), Figure 3 caption;
- an independent construction of the same masks (oracle/brute.py walks the
  blocks / prefix / copies instead of evaluating a predicate);
- closed-form pair counts.
"""
import os
import random

import numpy as np
import pytest

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "masks.txt")


def load_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.rstrip("\n")
        if not line or line.startswith("#"):
            continue
        if line.startswith("case "):
            parts = line.split()
            meta = dict(p.split("=") for p in parts[2:])
            cur = dict(name=parts[1], kind=meta["kind"], B=int(meta["B"]), P=int(meta["P"]),
                       Lq=int(meta["Lq"]), Lk=int(meta["Lk"]), rows=[])
            cases.append(cur)
        else:
            cur["rows"].append([c == "x" for c in line])
    for c in cases:
        assert len(c["rows"]) == c["Lq"] and all(len(r) == c["Lk"] for r in c["rows"]), c["name"]
    return cases


GOLD = load_golden()


@pytest.mark.parametrize("case", GOLD, ids=[c["name"] for c in GOLD])
def test_oracle_mask_matches_hand_drawn(case):
    kind = oracle.BLOCK_CAUSAL if case["kind"] == "bc" else oracle.STAIRCASE
    m = oracle.mask(kind, case["B"], case["P"], case["Lq"], case["Lk"])
    assert (m == np.array(case["rows"])).all()


@pytest.mark.parametrize("case", GOLD, ids=[c["name"] for c in GOLD])
def test_brute_construction_matches_hand_drawn(case):
    if case["kind"] == "bc":
        m = brute.mask_block_causal(case["Lq"], case["Lk"], case["B"])
    else:
        m = brute.mask_staircase(case["Lk"], case["B"], case["P"])
    assert (m == np.array(case["rows"])).all()


def test_mask_exhaustive_vs_construction():
    rng = random.Random(1)
    for _ in range(300):
        B = rng.choice([1, 2, 3, 4, 5, 8])
        Lk = rng.randint(1, 40)
        Lq = rng.randint(1, Lk)
        m = oracle.mask(oracle.BLOCK_CAUSAL, B, 0, Lq, Lk)
        assert (m == brute.mask_block_causal(Lq, Lk, B)).all(), (B, Lq, Lk)
    for _ in range(300):
        B = rng.choice([1, 2, 3, 4, 8])
        P = rng.randint(0, 30)
        K = rng.randint(0, 5)
        L = P + K * B
        if L == 0:
            continue
        m = oracle.mask(oracle.STAIRCASE, B, P, L, L)
        assert (m == brute.mask_staircase(L, B, P)).all(), (B, P, K)


def test_staircase_without_copies_is_block_causal():
    for B in (1, 2, 3, 32):
        for L in (1, 7, 64, 65):
            a = oracle.mask(oracle.STAIRCASE, B, L, L, L)
            b = oracle.mask(oracle.BLOCK_CAUSAL, B, 0, L, L)
            assert (a == b).all()


def test_special_cases_causal_and_full():
    for L in (1, 5, 33):
        causal = np.tril(np.ones((L, L), dtype=bool))
        assert (oracle.mask(oracle.BLOCK_CAUSAL, 1, 0, L, L) == causal).all()
        assert oracle.mask(oracle.BLOCK_CAUSAL, L, 0, L, L).all()


def test_every_row_sees_something():
    rng = random.Random(2)
    for _ in range(100):
        B = rng.choice([1, 2, 3, 8])
        P = rng.randint(0, 20)
        L = P + rng.randint(0, 4) * B
        if L == 0:
            continue
        assert oracle.mask(oracle.STAIRCASE, B, P, L, L).any(axis=1).all()


def closed_form_bc(L, B):
    # full blocks: n blocks of B -> B^2 * n(n+1)/2; a ragged last block of r
    # queries sees all L keys.
    n, r = divmod(L, B)
    return B * B * n * (n + 1) // 2 + r * L


def test_pair_counts_closed_form():
    for L, B in [(256, 32), (100, 7), (64, 64), (65, 64), (1, 1), (33, 1)]:
        assert oracle.count_pairs(oracle.BLOCK_CAUSAL, B, 0, L, L) == closed_form_bc(L, B)
    # staircase: block-causal prefix + each copy sees P prefix keys and its B keys
    for P, B, K in [(1024, 32, 16), (0, 4, 3), (10, 4, 2), (7, 3, 5)]:
        L = P + K * B
        want = closed_form_bc(P, B) + K * (B * P + B * B)
        assert oracle.count_pairs(oracle.STAIRCASE, B, P, L, L) == want
    # decode: every query of the active block sees all keys
    assert oracle.count_pairs(oracle.BLOCK_CAUSAL, 32, 0, 32, 2080) == 32 * 2080


def test_pair_counts_of_named_workloads():
    from diffusion_lm_block_bda_b300 import workloads as W
    w1 = W.named("c1")
    assert oracle.count_pairs_packed(w1.kind, w1.block_size, w1.cu_seqlens_q, w1.cu_seqlens_k,
                                     w1.prefix) == 36864
    w2 = W.named("c2")
    assert oracle.count_pairs_packed(w2.kind, w2.block_size, w2.cu_seqlens_q, w2.cu_seqlens_k,
                                     w2.prefix) == 66560
    w4 = W.named("c4")
    assert oracle.count_pairs_packed(w4.kind, w4.block_size, w4.cu_seqlens_q, w4.cu_seqlens_k,
                                     w4.prefix) == 8650752
    # c5 by closed form only (the explicit count walks 2^30 pairs)
    assert closed_form_bc(32768, 64) == 537919488
