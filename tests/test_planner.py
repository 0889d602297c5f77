"""Tile planner checks (host only): the plan written by bda_attn_plan_host is
decoded and compared exhaustively with the oracle's explicit mask.

Forward: every allowed (query, key) pair of every query tile falls in exactly
one listed key tile; tiles marked FULL hold only allowed pairs; no listed tile
is empty.  Backward: the query-token tiles of each key tile (one or two
ranges) hold every query that sees one of its keys, and no query twice.
Multi-block staircase layouts are checked against the oracle's mask too.  Order: forward longest unit first, backward
sequence-major (longest sequences first, longest key tiles first inside each)
up to its last wave, which runs longest-first;
a list schedule over 148 SMs ends within one unit of max(total / 148, longest
unit)."""
import random

import numpy as np
import pytest
import torch

import oracle
import diffusion_lm_block_bda_b300 as bda
from diffusion_lm_block_bda_b300 import Problem, workloads as W

HDR = 256
ITEM_INTS = 16
FWD_FIELDS = ["q_row", "q_len", "pos0", "k_row", "lk", "prefix", "n_full", "r1_end", "r2_begin",
              "r2_end", "work", "seq", "grp_off", "n_grp", "n_split", "part0"]
BWD_FIELDS = ["k_row", "k_len", "kpos0", "q_row", "lq", "lk", "prefix", "q_begin", "q_end",
              "q2_begin", "q2_end", "n_tiles1", "work", "seq", "grp_off", "n_grp"]


def decode(pb):
    buf = torch.zeros(bda.bda_attn_plan_size(pb), dtype=torch.uint8)
    bda.bda_attn_plan_host(pb, buf)
    a = buf.numpy().view(np.int32)
    hdr = a[:HDR // 4]
    magic, n_fwd, n_bwd, hg, tok = int(hdr[1]) & 0xffffffff, int(hdr[2]), int(hdr[3]), int(hdr[4]), int(hdr[5])
    assert magic == 0x42444131
    n_items = n_fwd + n_bwd
    items = a[HDR // 4:HDR // 4 + n_items * ITEM_INTS].reshape(-1, ITEM_INTS)
    fw = [dict(zip(FWD_FIELDS, map(int, r))) for r in items[:n_fwd]]
    bw = [dict(zip(BWD_FIELDS, map(int, r))) for r in items[n_fwd:n_fwd + n_bwd]]
    n_cg, n_dec, n_parts, split_c = int(hdr[8]), int(hdr[9]), int(hdr[10]), int(hdr[11])
    table = a[HDR // 4 + n_items * ITEM_INTS:][:2 * n_cg].reshape(-1, 2)
    table_words = -(-8 * n_cg // 16) * 4
    assert a.size * 4 == HDR + 64 * n_items + 4 * table_words + 16 * n_dec
    dec = a[HDR // 4 + n_items * ITEM_INTS + table_words:].reshape(-1, 4)
    assert dec.shape[0] == n_dec
    for it in fw + bw:
        it["groups"] = [tuple(map(int, r)) for r in table[it["grp_off"]:it["grp_off"] + it["n_grp"]]]
    check_split(fw, dec, n_parts, split_c)
    return fw, bw, hg, tok


def check_split(fw, dec, n_parts, split_c):
    """Split-forward units: each item's chunks cover its key tiles [0, work)
    in order, each chunk non-empty and at most split_c + 1 tiles; partial
    slots are numbered consecutively over the split items."""
    by_item = {}
    for item, lo, hi, part in dec.tolist():
        by_item.setdefault(item, []).append((lo, hi, part))
    assert sorted(by_item) == list(range(len(fw)))
    next_part = 0
    for i, it in enumerate(fw):
        chunks = by_item[i]
        assert len(chunks) == it["n_split"]
        assert chunks[0][0] == 0 and chunks[-1][1] == it["work"]
        assert all(a[1] == b[0] for a, b in zip(chunks, chunks[1:]))
        assert all(hi > lo for lo, hi, _ in chunks)
        if it["n_split"] > 1:
            assert split_c > 0 and all(hi - lo <= split_c + 1 for lo, hi, _ in chunks)
            assert it["part0"] == next_part
            assert [p for _, _, p in chunks] == list(range(next_part, next_part + it["n_split"]))
            next_part += it["n_split"]
        else:
            assert chunks[0][2] == -1 and it["part0"] == -1
    assert next_part == n_parts


def key_tiles(it):
    return list(range(it["r1_end"])) + list(range(it["r2_begin"], it["r2_end"]))


def check_plan(w):
    pb = Problem.from_workload(w)
    fw, bw, hg, tok = decode(pb)
    G = w.hq // w.hkv
    assert G % hg == 0 and hg * tok == 128
    cq, ck = w.cu_seqlens_q, w.cu_seqlens_k
    masks = []
    for s in range(w.nseq):
        lq, lk = cq[s + 1] - cq[s], ck[s + 1] - ck[s]
        if w.kind == W.STAIRCASE_MULTI:
            g = w.groups[s]
            masks.append(oracle.mask_multi(w.block_size, w.prefix[s], [c for c, _ in g],
                                           [v for _, v in g], lq) if lq else None)
            continue
        P = w.prefix[s] if w.kind == W.STAIRCASE else lk
        masks.append(oracle.mask(w.kind, w.block_size, P, lq, lk) if lq and lk else None)
    # forward coverage
    seen_tiles = {}
    for it in fw:
        s = it["seq"]
        M = masks[s]
        t0 = it["q_row"] - cq[s]
        rows = M[t0:t0 + it["q_len"]]
        assert it["q_len"] == min(tok, (cq[s + 1] - cq[s]) - t0)
        tiles = key_tiles(it)
        assert len(tiles) == len(set(tiles)) == it["work"]
        covered = np.zeros_like(rows)
        for n, kt in enumerate(tiles):
            blk = rows[:, kt * 128:(kt + 1) * 128]
            assert blk.any(), ("empty tile scheduled", s, t0, kt)
            if n < it["n_full"]:
                assert blk.all() and blk.shape[1] == 128, ("FULL tile not full", s, t0, kt)
            covered[:, kt * 128:(kt + 1) * 128] = True
        assert not (rows & ~covered).any(), ("allowed pair not covered", s, t0)
        seen_tiles[(s, t0)] = True
    for s in range(w.nseq):
        lq = cq[s + 1] - cq[s]
        assert all((s, t0) in seen_tiles for t0 in range(0, lq, tok))
    # backward coverage
    for it in bw:
        s = it["seq"]
        kp = it["kpos0"]
        assert it["k_row"] == ck[s] + kp and it["k_len"] == min(128, ck[s + 1] - ck[s] - kp)
        M = masks[s]
        if M is None:
            assert it["q_end"] == it["q_begin"] and it["q2_end"] == it["q2_begin"]
            continue
        lq = cq[s + 1] - cq[s]
        n1 = -(-(it["q_end"] - it["q_begin"]) // tok)
        n2 = -(-(it["q2_end"] - it["q2_begin"]) // tok)
        assert it["n_tiles1"] == n1
        # the tiles the kernel walks: no query token twice, every seeing row inside
        tokens = [t for i in range(n1) for t in range(it["q_begin"] + i * tok,
                                                        it["q_begin"] + (i + 1) * tok)]
        tokens += [t for i in range(n2) for t in range(it["q2_begin"] + i * tok,
                                                         it["q2_begin"] + (i + 1) * tok)]
        assert len(tokens) == len(set(tokens)), ("query token visited twice", s, kp)
        sees = M[:, kp:kp + it["k_len"]].any(axis=1)
        idx = set(np.nonzero(sees)[0].tolist())
        assert idx <= set(t for t in tokens if t < lq), ("seeing row not visited", s, kp)
        assert it["work"] == (n1 + n2) * (G // hg)
    assert sorted(it["kpos0"] + ck[it["seq"]] for it in bw) == sorted(
        ck[s] + kp for s in range(w.nseq) for kp in range(0, ck[s + 1] - ck[s], 128))
    # Order: forward longest-first; backward sequence-major (sequences by total
    # work, longest first; inside a sequence its key tiles longest-first),
    # except its last wave (148 CTAs of hkv per item), which is the same
    # items re-sorted longest-first across sequences.
    works = [it["work"] for it in fw]
    assert works == sorted(works, reverse=True)
    n_tail = min(len(bw), -(-148 // w.hkv))
    seq_work = {}
    for it in bw:
        seq_work[it["seq"]] = seq_work.get(it["seq"], 0) + it["work"]
    def seq_major(items):
        return sorted(items, key=lambda it: (-seq_work[it["seq"]], it["seq"], -it["work"]))
    key = lambda it: (it["seq"], it["kpos0"])
    # stable sorts: equal keys keep their packing order, so compare positions
    expect = seq_major(sorted(bw, key=key))
    head, tail = expect[:len(expect) - n_tail], expect[len(expect) - n_tail:]
    tail = sorted(tail, key=lambda it: -it["work"])
    assert [key(it) for it in bw] == [key(it) for it in head + tail]
    # any list schedule ends within one unit of the mean load
    for items in (fw, bw):
        works = [it["work"] for it in items]
        if works:
            m = 148
            loads = [0] * m
            for x in works:
                i = loads.index(min(loads))
                loads[i] += x
            assert max(loads) <= sum(works) / m + max(works)
    return fw, bw


def random_multi_workload(rng):
    """Multi-block staircase layouts with groups in block order (visible
    non-decreasing), some groups empty."""
    B = rng.choice([1, 5, 16, 32, 64, 128])
    hq, hkv = rng.choice([(4, 4), (8, 2), (32, 8), (16, 1)])
    prefix, groups = [], []
    for _ in range(rng.randint(1, 3)):
        P = rng.randint(0, 400)
        vis = sorted(rng.randint(0, P) for _ in range(rng.randint(0, 4)))
        g = [(rng.choice([0, 1, 2, 3, 6]), v) for v in vis]
        if P == 0 and sum(c for c, _ in g) == 0:
            g = [(1, 0)]
        prefix.append(P)
        groups.append(g)
    return W.multi_staircase(prefix, groups, block_size=B, hq=hq, hkv=hkv)


def random_workload(rng):
    if rng.random() < 0.3:
        return random_multi_workload(rng)
    kind = rng.choice([W.BLOCK_CAUSAL, W.STAIRCASE])
    B = rng.choice([1, 5, 16, 32, 64, 128, 200])
    hq, hkv = rng.choice([(4, 4), (8, 2), (32, 8), (16, 1), (6, 2)])
    lens_q, lens_k, pref = [], [], []
    for _ in range(rng.randint(1, 4)):
        if kind == W.BLOCK_CAUSAL:
            lk = rng.randint(1, 700)
            lq = lk if rng.random() < 0.6 else rng.randint(0, lk)
            lens_q.append(lq)
            lens_k.append(lk)
        else:
            P = rng.randint(0, 500)
            L = P + B * rng.randint(0, 5)
            if L == 0:
                L = B
            lens_q.append(L)
            lens_k.append(L)
            pref.append(P)
    return W.custom(kind, B, hq, hkv, 128, lens_q, lens_k, pref or None)


def test_planner_random_exhaustive():
    rng = random.Random(11)
    for _ in range(90):
        check_plan(random_workload(rng))


def test_planner_multi_block_staircase_layouts():
    # the hand-drawn layouts' shapes, scaled up, and 4 groups x 8 copies after 1024
    ws = [W.multi_staircase([6 * 32], [[(2, 2 * 32), (1, 6 * 32)]], block_size=32, hq=8, hkv=2),
          W.multi_staircase([1024] * 2, [[(8, 256), (8, 512), (8, 768), (8, 1024)]] * 2),
          W.multi_staircase([1000, 130], [[(3, 0), (2, 640), (1, 1000)], [(0, 5), (4, 130)]],
                            block_size=16, hq=8, hkv=2)]
    for w in ws:
        fw, bw = check_plan(w)
        assert any(it["n_grp"] > 0 for it in fw)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4"])
def test_planner_named_workloads(name):
    fw, bw = check_plan(W.named(name))
    if name == "c4":
        # copy tiles: 8 FULL prefix tiles, then the copy's own key tile
        copy_items = [it for it in fw if it["pos0"] >= 1024]
        assert copy_items and all(it["n_full"] == 8 and it["work"] == 9 for it in copy_items)
    if name == "c2":
        assert len(fw) == 1 and fw[0]["work"] == 17 and fw[0]["n_full"] == 16


def test_split_forward_plans():
    """Problems with fewer than 74 query-tile units split their key tiles so
    the units number about 74; larger ones are not split."""
    def header(pb):
        buf = torch.zeros(bda.bda_attn_plan_size(pb), dtype=torch.uint8)
        bda.bda_attn_plan_host(pb, buf)
        h = buf[:64].numpy().view(np.int32)
        return int(h[9]), int(h[10]), int(h[11])  # n_dec, n_parts, split_c
    c2 = Problem.from_workload(W.named("c2"))
    assert header(c2) == (9, 9, 2)  # 17 key tiles x 8 head groups: 9 chunks of <= 2 tiles
    long_decode = Problem([0, 32], [0, 32 * 1024], 32, 8, 128, W.BLOCK_CAUSAL, 32)
    n_dec, n_parts, c = header(long_decode)  # 256 tiles x 8 groups: chunks of 28
    assert c == 28 and n_dec == n_parts == 10
    assert header(Problem.from_workload(W.named("c3")))[2] == 0
    check_plan(W.custom(W.BLOCK_CAUSAL, 32, 32, 8, 128, [32, 32, 5], [2080, 700, 133]))


def test_planner_long_sequence_counts():
    w = W.named("c5")
    fw, bw, hg, tok = decode(Problem.from_workload(w))
    assert hg == 4 and tok == 32
    assert len(fw) == 32768 // 32 and len(bw) == 32768 // 128
    works = sorted(it["work"] for it in fw)
    assert works[0] == 1 and works[-1] == 256
