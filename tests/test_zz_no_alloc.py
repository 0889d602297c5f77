"""bda_attn_fwd_noalloc: the forward for callers that cannot allocate device
memory where they run attention -- an engine plugin whose host process owns
every byte of device memory, or a decode loop that must not risk the
synchronisation an allocation can cause.  It takes no workspace: its tile
plan and status word live in a fixed 1 MiB array inside the library, shared
by every call.

Two no-alloc calls in a row with different problems (the second must fully
replace what the first left in the shared array) are checked against the
fp64 oracle and, bit for bit, against the workspace forward bda_attn_fwd
(same kernel, same plan).  Also: plans beyond the array are refused; a
stream under graph capture is refused; a bounded wait that runs out is
reported by the no-alloc status reader.  Collected last on purpose."""
import pytest
import torch

import diffusion_lm_block_bda_b300 as bda
from diffusion_lm_block_bda_b300 import Attention, Problem, workloads as W

from _parity import compare_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


def _inputs(w, seed):
    inp = W.make_inputs(w, seed=seed, with_dout=False)
    return inp, [inp[n].cuda() for n in ("q", "k", "v")]


def _outputs(w):
    pb = Problem.from_workload(w)
    o = torch.full((pb.total_q, w.hq, w.head_dim), float("nan"), dtype=torch.bfloat16,
                   device="cuda")
    lse = torch.full((w.hq, pb.total_q), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


CASES = [
    W.named("c2"),  # decode step: 32 queries over 2080 keys
    W.custom(W.STAIRCASE, 32, 8, 2, 128, [1536, 700], prefix=[1024, 316], name="sc"),
]


def test_noalloc_forward_matches_oracle_and_workspace_forward():
    data = [(w, *_inputs(w, seed=i + 7)) for i, w in enumerate(CASES)]
    got = []
    for w, _, (q, k, v) in data:  # two no-alloc calls in a row, back to back on the stream
        o, lse = _outputs(w)
        bda.bda_attn_fwd_noalloc(Problem.from_workload(w), q, k, v, o, lse)
        got.append((o, lse))
    torch.cuda.synchronize()
    assert bda.bda_attn_fwd_noalloc_check_status() == bda.BDA_OK
    for (w, inp, (q, k, v)), (o, lse) in zip(data, got):
        compare_full(w, inp, dict(o=o.float().cpu(), lse=lse.cpu()), with_bwd=False)
        # the no-alloc forward always runs the persistent kernel: the same
        # kernel on the same plan through the workspace path gives the same bits
        try:
            bda.bda_testing_force_forward_kernel(1)
            ref_o, ref_lse = Attention(Problem.from_workload(w), with_bwd=False).forward(q, k, v)
            torch.cuda.synchronize()
        finally:
            bda.bda_testing_force_forward_kernel(0)
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_plans_beyond_its_array():
    # 20000 one-token sequences need 20000 forward items: > 1 MiB of plan.
    n = 20000
    cu = list(range(n + 1))
    pb = Problem(cu, cu, 8, 2, 128, W.BLOCK_CAUSAL, 32)
    x = torch.zeros((n, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((n, 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((8, n), dtype=torch.float32, device="cuda")
    st = bda.lib().bda_attn_fwd_noalloc(*pb.refs(), x.data_ptr(), kv.data_ptr(), kv.data_ptr(),
                                        x.data_ptr(), lse.data_ptr(), None)
    assert st == bda.BDA_ERR_WORKSPACE


def test_noalloc_refuses_a_stream_under_capture():
    w = CASES[0]
    _, (q, k, v) = _inputs(w, seed=3)
    o, lse = _outputs(w)
    pb = Problem.from_workload(w)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        st = bda.lib().bda_attn_fwd_noalloc(*pb.refs(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse.data_ptr(), side.cuda_stream)
        o.add_(0)  # the capture holds one ordinary node
    assert st == bda.BDA_ERR_UNSUPPORTED
    torch.cuda.synchronize()


def test_noalloc_status_reader_reports_a_wait_timeout():
    w = CASES[1]
    inp, (q, k, v) = _inputs(w, seed=5)
    pb = Problem.from_workload(w)
    try:
        assert bda.bda_testing_arm_wait_timeout(1, 1_000_000) == bda.BDA_OK
        o, lse = _outputs(w)
        bda.bda_attn_fwd_noalloc(pb, q, k, v, o, lse)
        assert bda.bda_attn_fwd_noalloc_check_status() == bda.BDA_ERR_DEVICE_TIMEOUT
        assert bda.bda_attn_fwd_noalloc_check_status() == bda.BDA_OK
    finally:
        bda.bda_testing_arm_wait_timeout(0, 0)
    o, lse = _outputs(w)
    bda.bda_attn_fwd_noalloc(pb, q, k, v, o, lse)
    assert bda.bda_attn_fwd_noalloc_check_status() == bda.BDA_OK
    compare_full(w, inp, dict(o=o.float().cpu(), lse=lse.cpu()), with_bwd=False)
