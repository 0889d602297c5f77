"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, at the tolerances in tests/_parity.py.

Small workloads and edge cases compare every output element.  The full-size
workloads run on the GPU exactly as the benchmark launches them and compare
sampled outputs the oracle computes one by one (query rows for O/LSE/dQ, key
rows from the end of the sequence for dK/dV, whose rows are few), plus sum
rules that hold at any size.
"""
import numpy as np
import pytest
import torch

from diffusion_lm_block_bda_b300 import workloads as W

from _parity import (check_sum_rules, compare_full, compare_sampled, gpu_run)

pytestmark = pytest.mark.gpu

BC, SC = W.BLOCK_CAUSAL, W.STAIRCASE


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


def test_tiny_block_causal_c1():
    w = W.named("c1")
    inp = W.make_inputs(w, seed=0)
    got = gpu_run(w, inp)
    compare_full(w, inp, got)


def test_decode_step_c2():
    w = W.named("c2")
    inp = W.make_inputs(w, seed=0)
    got = gpu_run(w, inp, with_bwd=False)
    compare_full(w, inp, got, with_bwd=False)


EDGE = [
    # kind, block, hq, hkv, d, seqlens_q, seqlens_k, prefix
    (BC, 16, 8, 2, 128, [1, 7, 130, 257, 33], None, None),          # ragged varlen, G=4
    (BC, 16, 8, 2, 64, [1, 7, 130, 257, 33], None, None),           # d = 64
    (BC, 32, 4, 4, 128, [200, 129], None, None),                    # MHA (G = 1)
    (BC, 8, 16, 2, 128, [64, 300], None, None),                     # G = 8
    (BC, 1, 4, 2, 128, [150], None, None),                          # B = 1: causal
    (BC, 512, 4, 2, 128, [300], None, None),                        # B >= L: full
    (BC, 32, 8, 2, 128, [5, 40, 0, 32], [300, 129, 17, 2080], None),  # decode, Lq < Lk, empty
    (BC, 24, 8, 2, 128, [97, 250], [97, 250], None),                # B not a power of two
    (SC, 16, 8, 2, 128, [260, 100], None, [100, 20]),               # prefix not % 128
    (SC, 32, 8, 2, 128, [1536], None, [1024]),                      # one staircase trajectory
    (SC, 16, 8, 2, 64, [96], None, [0]),                            # copies only, d = 64
    (SC, 128, 4, 1, 128, [640], None, [256]),                       # copies of 128 tokens
]


@pytest.mark.parametrize("case", EDGE, ids=[f"e{i}" for i in range(len(EDGE))])
def test_edge_cases_full_oracle(case):
    kind, B, hq, hkv, d, lq, lk, prefix = case
    w = W.custom(kind, B, hq, hkv, d, lq, lk, prefix, name=f"edge_{kind}_{B}_{hq}_{hkv}_{d}")
    inp = W.make_inputs(w, seed=3)
    got = gpu_run(w, inp)
    compare_full(w, inp, got)


def test_staircase_replay_c4():
    w = W.named("c4")
    inp = W.make_inputs(w, seed=0)
    got = gpu_run(w, inp)
    # exact on two trajectories and two KV heads (8 query heads), every row
    compare_sampled(w, inp, got, seqs=[0, 7], kv_heads=(3, 5),
                    qrows_fn=lambda L: list(range(L)), krows_fn=lambda L: list(range(L)))
    check_sum_rules(w, inp, got)


def _sample_rows(L, n=48):
    r = set(np.linspace(0, L - 1, n).astype(int).tolist())
    r.update([0, L - 1, min(L - 1, 31), min(L - 1, 32), min(L - 1, 127), min(L - 1, 128)])
    return sorted(r)


def _tail_keys(L, n=160):
    return list(range(max(0, L - n), L))


def test_packed_replay_c3():
    w = W.named("c3")
    inp = W.make_inputs(w, seed=0)
    got = gpu_run(w, inp)
    lens = w.seqlens_q
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 5})
    compare_sampled(w, inp, got, seqs=seqs, kv_heads=(0, 1), qrows_fn=_sample_rows,
                    krows_fn=_tail_keys)
    compare_sampled(w, inp, got, seqs=[int(np.argmin(lens))], kv_heads=(7, 8),
                    qrows_fn=_sample_rows, krows_fn=lambda L: list(range(L)))
    check_sum_rules(w, inp, got)


def test_long_block_causal_c5():
    w = W.named("c5")
    inp = W.make_inputs(w, seed=0)
    got = gpu_run(w, inp)
    compare_sampled(w, inp, got, seqs=[0], kv_heads=(0, 1),
                    qrows_fn=lambda L: _sample_rows(L, 24), krows_fn=lambda L: _tail_keys(L, 96))
    check_sum_rules(w, inp, got)
