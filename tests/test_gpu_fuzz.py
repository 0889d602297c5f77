"""GPU parity on 120 random small layouts: block-causal (with and without fewer
queries than keys), single-block staircase and multi-block staircase, drawn
from one seeded generator over block sizes 1..256, GQA ratios 1..8, head_dim
64 and 128, ragged and empty sequences.  Each case goes through both forward
kernels (persistent and split) and the backward, and every output element is
compared with the fp64 oracle at the tolerances of tests/_parity.py.

The layouts follow the readings the oracle implements: block-causal queries
aligned with the last keys when Lq < Lk; a staircase prefix followed by
whole copies of the block; multi-block groups in block order (the clean keys a
group sees do not decrease along the sequence)."""
import random

import pytest
import torch

from diffusion_lm_block_bda_b300 import workloads as W

from _parity import compare_full, gpu_run, oracle_full

pytestmark = pytest.mark.gpu

N_CASES = 120


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


def _case(i):
    rng = random.Random(1000 + i)
    kind = rng.choice([W.BLOCK_CAUSAL, W.BLOCK_CAUSAL, W.STAIRCASE, W.STAIRCASE_MULTI])
    d = rng.choice([64, 128])
    hq, hkv = rng.choice([(4, 1), (4, 2), (8, 2), (8, 8), (16, 2), (32, 8)])
    B = rng.choice([1, 2, 5, 16, 32, 48, 64, 128, 256])
    nseq = rng.randint(1, 3)
    name = f"fuzz{i}"
    if kind == W.BLOCK_CAUSAL:
        lq = [rng.choice([0, 1, rng.randint(2, 128), rng.randint(129, 400)]) for _ in range(nseq)]
        if rng.random() < 0.4:  # a decode-like step: the queries are the last keys
            lk = [q + rng.randint(0, 300) for q in lq]
            return W.custom(kind, B, hq, hkv, d, lq, lk, name=name)
        return W.custom(kind, B, hq, hkv, d, lq, name=name)
    if kind == W.STAIRCASE:
        B = min(B, 64)
        prefix, lens = [], []
        for _ in range(nseq):
            p = rng.randint(0, 300)
            c = rng.randint(0 if p else 1, 4)
            prefix.append(p)
            lens.append(p + c * B)
        return W.custom(kind, B, hq, hkv, d, lens, prefix=prefix, name=name)
    B = min(B, 64)
    prefix, groups = [], []
    for _ in range(nseq):
        p = rng.randint(0, 300)
        vis = sorted(rng.randint(0, p) for _ in range(rng.randint(1, 3)))
        g = [(rng.randint(0, 3), v) for v in vis]
        if sum(c for c, _ in g) == 0 and p == 0:
            g[0] = (1, g[0][1])
        prefix.append(p)
        groups.append(g)
    w = W.multi_staircase(prefix, groups, block_size=B, hq=hq, hkv=hkv, head_dim=d)
    w.name = name
    return w


@pytest.mark.parametrize("i", range(N_CASES), ids=[f"f{i}" for i in range(N_CASES)])
def test_random_layout_full_oracle(i):
    import diffusion_lm_block_bda_b300 as bda
    w = _case(i)
    inp = W.make_inputs(w, seed=50 + i)
    ref = oracle_full(w, inp)
    try:
        for which in (1, 2):
            assert bda.bda_testing_force_forward_kernel(which) == bda.BDA_OK
            got = gpu_run(w, inp)
            compare_full(w, inp, got, ref=ref)
    finally:
        bda.bda_testing_force_forward_kernel(0)
