"""Failure detection without a GPU fault: every mbarrier wait in the kernels
is bounded, and a wait that runs out records BDA_ERR_DEVICE_TIMEOUT in the
status word, after which the CTA lets its in-flight copies and MMAs land,
frees its TMEM and returns.  The library's testing hook arms one launch so
that CTA 0 leaves its first Q load un-issued (nothing is loaded from a bad
address, nothing traps, nothing waits without a limit) with a 1 ms limit.
Each test checks that the status is reported and cleared, and that a clean
call on the same workspace afterwards matches the fp64 oracle."""
import pytest
import torch

import diffusion_lm_block_bda_b300 as bda
from diffusion_lm_block_bda_b300 import Attention, Problem, workloads as W

from _parity import compare_full

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000  # 1 ms


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


@pytest.fixture(autouse=True)
def _disarm():
    yield
    bda.bda_testing_arm_wait_timeout(0, 0)


def _case():
    w = W.custom(W.STAIRCASE, 32, 8, 2, 128, [416, 160], prefix=[96, 64], name="fault")
    inp = W.make_inputs(w, seed=17)
    return w, inp, Problem.from_workload(w)


def _run(att, w, inp, pb):
    q, k, v, dout = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = att.forward(q, k, v)
    dq, dk, dv = att.backward(q, k, v, o, lse, dout)
    torch.cuda.synchronize()
    return {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}


@pytest.mark.parametrize("stage", [1, 2], ids=["forward", "backward_dkdv"])
def test_wait_timeout_is_reported_and_the_workspace_recovers(stage):
    w, inp, pb = _case()
    att = Attention(pb, device="cuda", with_bwd=True)
    assert bda.bda_testing_arm_wait_timeout(stage, LIMIT_NS) == bda.BDA_OK
    _run(att, w, inp, pb)  # the armed launch: outputs unspecified
    assert bda.bda_attn_check_status(att.ws) == bda.BDA_ERR_DEVICE_TIMEOUT
    assert bda.bda_attn_check_status(att.ws) == bda.BDA_OK  # the read cleared it
    # the fault was one-shot: the next forward + backward are clean and exact
    got = _run(att, w, inp, pb)
    assert bda.bda_attn_check_status(att.ws) == bda.BDA_OK
    compare_full(w, inp, got)
