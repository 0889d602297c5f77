"""bda_attn_fwd_noalloc: the forward for callers that cannot allocate device
memory where they run attention (an engine plugin whose host process owns
every byte of device memory, a decode loop that must not risk the
synchronisation an allocation can cause).  It takes no workspace: its tile
plan lives in a fixed 1 MiB array inside the library.

Checked through the C ABI against the workspace forward (bda_attn_fwd) on two
calls in a row with different problems, so the second call must fully replace
what the first left in the shared array.  Collected last on purpose."""
import pytest
import torch

import diffusion_lm_block_bda_b300 as bda
from diffusion_lm_block_bda_b300 import Attention, Problem, workloads as W

from _parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def _inputs(w, seed):
    inp = W.make_inputs(w, seed=seed, with_dout=False)
    return [inp[n].cuda() for n in ("q", "k", "v")]


def _outputs(w):
    pb = Problem.from_workload(w)
    o = torch.full((pb.total_q, w.hq, w.head_dim), float("nan"), dtype=torch.bfloat16,
                   device="cuda")
    lse = torch.full((w.hq, pb.total_q), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def test_noalloc_forward_matches_workspace_forward():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    cases = [
        W.named("c2"),  # decode step: 32 queries over 2080 keys
        W.custom(W.STAIRCASE, 32, 8, 2, 128, [1536, 700], prefix=[1024, 316], name="sc"),
    ]
    data = [(w, _inputs(w, seed=i + 7)) for i, w in enumerate(cases)]
    # two no-alloc calls in a row, back to back on the stream
    got = []
    for w, (q, k, v) in data:
        o, lse = _outputs(w)
        bda.bda_attn_fwd_noalloc(Problem.from_workload(w), q, k, v, o, lse)
        got.append((o, lse))
    torch.cuda.synchronize()
    for (w, (q, k, v)), (o, lse) in zip(data, got):
        ref_o, ref_lse = Attention(Problem.from_workload(w), with_bwd=False).forward(q, k, v)
        torch.cuda.synchronize()
        check_o(o.float().cpu().numpy(), ref_o.float().cpu().numpy(), "noalloc vs fwd")
        check_lse(lse.cpu().numpy(), ref_lse.cpu().numpy(), "noalloc vs fwd")


def test_noalloc_rejects_plans_beyond_its_array():
    # 20000 one-token sequences need 40000 work items: > 1 MiB of plan.
    n = 20000
    cu = list(range(n + 1))
    pb = Problem(cu, cu, 8, 2, 128, W.BLOCK_CAUSAL, 32)
    assert bda.bda_attn_plan_size(pb) > (1 << 20)
    x = torch.zeros((n, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((n, 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((8, n), dtype=torch.float32, device="cuda")
    st = bda.lib().bda_attn_fwd_noalloc(*pb.refs(), x.data_ptr(), kv.data_ptr(), kv.data_ptr(),
                                        x.data_ptr(), lse.data_ptr(), None)
    assert st == bda.BDA_ERR_WORKSPACE
