"""C-ABI checks that need no GPU: libbda_attn.so loads, exports every function
include/bda_attn.h declares, validates arguments on the host (status codes,
nothing launched), and counts useful pairs like the oracle."""
import ctypes
import os
import random
import re

import pytest
import torch

import oracle
import diffusion_lm_block_bda_b300 as bda
from diffusion_lm_block_bda_b300 import Problem, workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bda_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bda_\w+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert "bda_attn_fwd" in names and "bda_attn_bwd" in names
    L = bda.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(bda.EXPORTED)


def test_status_strings():
    for s in range(6):
        assert bda.string(s)
    assert bda.string(0) == "ok"


def _pb(**kw):
    base = dict(cu_seqlens_q=[0, 100, 300], cu_seqlens_k=[0, 100, 300], hq=8, hkv=2,
                head_dim=128, kind=W.BLOCK_CAUSAL, block_size=32)
    base.update(kw)
    return Problem(**base)


FAKE = 1 << 20  # an aligned, never dereferenced "device" address


def _fwd_status(pb, ws_bytes=None, ptrs=None):
    L = bda.lib()
    n = bda.bda_attn_workspace_size(pb, False) if ws_bytes is None else ws_bytes
    p = ptrs or [FAKE] * 5
    return L.bda_attn_fwd(*pb.refs(), *p, FAKE, n, None)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), bda.BDA_ERR_UNSUPPORTED),
    (dict(head_dim=0), bda.BDA_ERR_INVALID_ARG),
    (dict(hq=6, hkv=4), bda.BDA_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=[0, 300, 100], cu_seqlens_k=[0, 300, 100]), bda.BDA_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=[1, 100, 300]), bda.BDA_ERR_INVALID_ARG),
    (dict(block_size=0), bda.BDA_ERR_INVALID_ARG),
    (dict(kind=7), bda.BDA_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=[0, 101, 300]), bda.BDA_ERR_INVALID_ARG),  # Lq > Lk (block-causal)
    (dict(kind=W.STAIRCASE, prefix_len=[4, 20]), bda.BDA_ERR_INVALID_ARG),  # (L-P) % B != 0
    (dict(kind=W.STAIRCASE, prefix_len=None), bda.BDA_ERR_INVALID_ARG),
    (dict(kind=W.STAIRCASE, prefix_len=[101, 12]), bda.BDA_ERR_INVALID_ARG),  # P > L
    (dict(kind=W.STAIRCASE, prefix_len=[4, 12], cu_seqlens_k=[0, 132, 332]),
     bda.BDA_ERR_INVALID_ARG),  # staircase needs Lq == Lk
])
def test_invalid_problems_rejected_on_host(kw, status):
    pb = _pb(**kw)
    L = bda.lib()
    assert L.bda_attn_plan_size(*pb.refs()) == 0
    assert L.bda_attn_workspace_size(*pb.refs(), 1) == 0
    assert L.bda_attn_count_pairs(*pb.refs()) == -1
    buf = torch.zeros(1 << 16, dtype=torch.uint8)
    assert L.bda_attn_plan_host(*pb.refs(), buf.data_ptr(), buf.numel()) == status
    assert _fwd_status(pb, ws_bytes=1 << 30) == status


def test_valid_staircase_accepted():
    pb = _pb(kind=W.STAIRCASE, prefix_len=[4, 8])
    buf = torch.zeros(bda.bda_attn_plan_size(pb), dtype=torch.uint8)
    bda.bda_attn_plan_host(pb, buf)


def test_pointer_and_workspace_errors():
    pb = _pb()
    L = bda.lib()
    need = bda.bda_attn_workspace_size(pb, False)
    assert _fwd_status(pb, ws_bytes=need - 1) == bda.BDA_ERR_WORKSPACE
    assert _fwd_status(pb, ptrs=[FAKE + 8] + [FAKE] * 4) == bda.BDA_ERR_INVALID_ARG
    assert _fwd_status(pb, ptrs=[None] + [FAKE] * 4) == bda.BDA_ERR_INVALID_ARG
    assert L.bda_attn_fwd(*pb.refs(), FAKE, FAKE, FAKE, FAKE, FAKE, None, need,
                          None) == bda.BDA_ERR_INVALID_ARG
    nb = bda.bda_attn_workspace_size(pb, True)
    assert nb > need
    # backward stages need the larger workspace
    for f, args in ((L.bda_attn_bwd_preprocess, [FAKE, FAKE]),
                    (L.bda_attn_bwd_dq_convert, [FAKE])):
        assert f(*pb.refs(), *args, FAKE, need, None) == bda.BDA_ERR_WORKSPACE
    assert L.bda_attn_bwd_dkdv(*pb.refs(), *[FAKE] * 7, FAKE, need, None) == bda.BDA_ERR_WORKSPACE
    assert L.bda_attn_bwd(*pb.refs(), *[FAKE] * 9, FAKE, need, None) == bda.BDA_ERR_WORKSPACE
    assert L.bda_attn_bwd(*pb.refs(), FAKE + 4, *[FAKE] * 8, FAKE, nb,
                          None) == bda.BDA_ERR_INVALID_ARG
    small = torch.zeros(8, dtype=torch.uint8)
    assert L.bda_attn_plan_host(*pb.refs(), small.data_ptr(), 8) == bda.BDA_ERR_WORKSPACE
    assert L.bda_attn_plan_host(*pb.refs(), None, 1 << 20) == bda.BDA_ERR_INVALID_ARG
    assert L.bda_attn_check_status(None, 0, None) == bda.BDA_ERR_INVALID_ARG


def test_empty_problem_is_a_no_op():
    pb = Problem([0], [0], 8, 2, 128, W.BLOCK_CAUSAL, 32)
    n = bda.bda_attn_workspace_size(pb, True)
    assert n > 0
    L = bda.lib()
    # nothing to launch: succeeds without touching the GPU
    assert L.bda_attn_fwd(*pb.refs(), None, None, None, None, None, FAKE, n, None) == bda.BDA_OK
    assert L.bda_attn_bwd(*pb.refs(), *[None] * 9, FAKE, n, None) == bda.BDA_OK


def test_count_pairs_matches_oracle():
    rng = random.Random(5)
    for _ in range(40):
        kind = rng.choice([W.BLOCK_CAUSAL, W.STAIRCASE])
        B = rng.choice([1, 3, 16, 32, 64])
        lens, lks, pref = [], [], []
        for _ in range(rng.randint(1, 4)):
            if kind == W.BLOCK_CAUSAL:
                lk = rng.randint(1, 400)
                lens.append(rng.randint(0, lk))
                lks.append(lk)
            else:
                P = rng.randint(0, 300)
                L = P + B * rng.randint(0, 6)
                if L == 0:
                    P, L = 0, B
                lens.append(L)
                lks.append(L)
                pref.append(P)
        w = W.custom(kind, B, 4, 2, 64, lens, lks, pref if kind == W.STAIRCASE else None)
        pb = Problem.from_workload(w)
        want = oracle.count_pairs_packed(kind, B, w.cu_seqlens_q, w.cu_seqlens_k, w.prefix)
        assert bda.bda_attn_count_pairs(pb) == want


def test_count_pairs_named_workloads():
    for name, want in (("c1", 36864), ("c2", 66560), ("c4", 8650752), ("c5", 537919488)):
        assert bda.bda_attn_count_pairs(Problem.from_workload(W.named(name))) == want


# Multi-block staircase: validated and counted on the host like the oracle;
# groups in block order (visible non-decreasing over a sequence's non-empty
# groups) are planned and computed, other layouts are counted only.
MULTI = dict(kind=bda.BDA_MASK_STAIRCASE_MULTI, cu_seqlens_q=[0, 224, 576],
             cu_seqlens_k=[0, 224, 576], prefix_len=[128, 64],
             groups=[[(2, 64), (1, 128)], [(4, 32), (0, 0), (5, 64)]])


def _multi_oracle_count(spec):
    want = 0
    for s, g in enumerate(spec["groups"]):
        n = spec["cu_seqlens_q"][s + 1] - spec["cu_seqlens_q"][s]
        want += oracle.count_pairs_multi(32, spec["prefix_len"][s], [c for c, _ in g],
                                         [v for _, v in g], n)
    return want


def test_multi_block_staircase_is_counted_like_the_oracle_and_planned():
    pb = _pb(**MULTI)
    L = bda.lib()
    assert L.bda_attn_count_pairs(*pb.refs()) == _multi_oracle_count(MULTI)
    n = L.bda_attn_plan_size(*pb.refs())
    assert n > 0 and L.bda_attn_workspace_size(*pb.refs(), 1) > n
    buf = torch.zeros(n, dtype=torch.uint8)
    assert L.bda_attn_plan_host(*pb.refs(), buf.data_ptr(), buf.numel()) == bda.BDA_OK


def test_multi_block_staircase_out_of_block_order_is_counted_not_computed():
    spec = {**MULTI, "groups": [[(2, 64), (1, 32)], [(4, 32), (0, 0), (5, 64)]]}
    pb = _pb(**spec)
    L = bda.lib()
    assert L.bda_attn_count_pairs(*pb.refs()) == _multi_oracle_count(spec)
    assert L.bda_attn_plan_size(*pb.refs()) == 0
    buf = torch.zeros(1 << 16, dtype=torch.uint8)
    assert L.bda_attn_plan_host(*pb.refs(), buf.data_ptr(), buf.numel()) == bda.BDA_ERR_UNSUPPORTED
    assert _fwd_status(pb, ws_bytes=1 << 30) == bda.BDA_ERR_UNSUPPORTED
    assert L.bda_attn_bwd(*pb.refs(), *[FAKE] * 9, FAKE, 1 << 30, None) == bda.BDA_ERR_UNSUPPORTED


def test_testing_hook_arguments():
    assert bda.bda_testing_arm_wait_timeout(3, 10**6) == bda.BDA_ERR_INVALID_ARG
    assert bda.bda_testing_arm_wait_timeout(1, 10) == bda.BDA_ERR_INVALID_ARG
    assert bda.bda_testing_arm_wait_timeout(1, 10**10) == bda.BDA_ERR_INVALID_ARG
    assert bda.bda_testing_arm_wait_timeout(0, 0) == bda.BDA_OK


@pytest.mark.parametrize("kw", [
    dict(groups=[[(2, 64), (2, 128)], [(4, 32), (0, 0), (5, 64)]]),   # copies overrun L
    dict(groups=[[(2, 64), (1, 129)], [(4, 32), (0, 0), (5, 64)]]),   # sees past the prefix
    dict(groups=[[(3, 64), (0, 128)], [(4, 32), (0, 0), (5, -1)]]),   # negative visible
    dict(groups=[[(2, 64), (1, 128)], [(-1, 32), (0, 0), (10, 64)]]),  # negative copies
    dict(groups=None),                                                 # no group arrays
    dict(cu_seqlens_k=[0, 224, 577]),                                  # Lq != Lk
    dict(prefix_len=None),
])
def test_malformed_multi_block_staircase_rejected(kw):
    pb = _pb(**{**MULTI, **kw})
    L = bda.lib()
    assert L.bda_attn_count_pairs(*pb.refs()) == -1
    assert _fwd_status(pb, ws_bytes=1 << 30) == bda.BDA_ERR_INVALID_ARG
