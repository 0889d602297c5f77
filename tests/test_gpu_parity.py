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

from _parity import (check_sum_rules, compare_full, compare_sampled, gpu_run, oracle_full)

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
    """The decode step takes the split forward (its 17 key tiles as 9 chunks
    x 8 head groups = 72 CTAs, merged by the combine kernel); the persistent
    forward must agree with the oracle too."""
    import diffusion_lm_block_bda_b300 as bda
    from diffusion_lm_block_bda_b300 import Problem
    w = W.named("c2")
    pb = Problem.from_workload(w)
    buf = torch.zeros(bda.bda_attn_plan_size(pb), dtype=torch.uint8)
    bda.bda_attn_plan_host(pb, buf)
    hdr = buf[:64].numpy().view(np.int32)
    assert hdr[11] == 2 and hdr[9] == 9 and hdr[10] == 9  # split_c, n_dec, n_parts
    inp = W.make_inputs(w, seed=0)
    ref = oracle_full(w, inp, with_bwd=False)
    compare_full(w, inp, gpu_run(w, inp, with_bwd=False), with_bwd=False, ref=ref)
    try:
        bda.bda_testing_force_forward_kernel(1)
        compare_full(w, inp, gpu_run(w, inp, with_bwd=False), with_bwd=False, ref=ref)
    finally:
        bda.bda_testing_force_forward_kernel(0)


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
    (BC, 32, 16, 1, 128, [300, 77], None, None),                    # G = 16: 8-token tiles
    (BC, 16, 32, 1, 64, [200, 9], None, None),                      # G = 32: two head groups per KV head
    (SC, 32, 12, 2, 128, [264], None, [72]),                        # G = 6 (head groups of 2)
    (BC, 16, 6, 2, 128, [130, 31], None, None),                     # G = 3 (head groups of 1)
]


@pytest.mark.parametrize("case", EDGE, ids=[f"e{i}" for i in range(len(EDGE))])
def test_edge_cases_full_oracle(case):
    """Every edge case through both forward kernels -- the persistent one and
    the split one (which small problems take by default) -- and the backward,
    each against the same oracle result."""
    import diffusion_lm_block_bda_b300 as bda
    kind, B, hq, hkv, d, lq, lk, prefix = case
    w = W.custom(kind, B, hq, hkv, d, lq, lk, prefix, name=f"edge_{kind}_{B}_{hq}_{hkv}_{d}")
    inp = W.make_inputs(w, seed=3)
    ref = oracle_full(w, inp)
    try:
        for which in (1, 2):
            assert bda.bda_testing_force_forward_kernel(which) == bda.BDA_OK
            got = gpu_run(w, inp)
            compare_full(w, inp, got, ref=ref)
    finally:
        bda.bda_testing_force_forward_kernel(0)


def _align256(n):
    return (n + 255) // 256 * 256


def _poison_dq_accumulator(ws, w, total_q):
    """Fill the workspace's fp32 dQ accumulator with NaN, so any row left
    unzeroed before a backward shows up.  A backward-sized workspace ends
    with the accumulator [total_q][hq][d]."""
    ws[ws.numel() - _align256(4 * total_q * w.hq * w.head_dim):].fill_(0xFF)


@pytest.mark.parametrize("case", [(BC, 16, 8, 2, 128, [1, 7, 130, 257, 33], None),
                                  (SC, 16, 8, 2, 64, [160, 96], [32, 0])],
                         ids=["bc_d128", "sc_d64"])
def test_dq_accumulator_reuse(case):
    """Each backward clears the workspace's dQ accumulator itself: garbage left
    there (NaN poison, or the sums of an earlier backward) never reaches dQ,
    whether or not a forward ran on the workspace first."""
    from diffusion_lm_block_bda_b300 import Attention, Problem
    kind, B, hq, hkv, d, lq, prefix = case
    w = W.custom(kind, B, hq, hkv, d, lq, None, prefix, name=f"dqacc_{kind}_{d}")
    inp = W.make_inputs(w, seed=5)
    pb = Problem.from_workload(w)
    q, k, v, dout = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    att = Attention(pb, device="cuda", with_bwd=True)
    _poison_dq_accumulator(att.ws, w, pb.total_q)
    o, lse = att.forward(q, k, v)
    runs = [att.backward(q, k, v, o, lse, dout)]
    runs.append(att.backward(q, k, v, o, lse, dout))  # no forward between
    fresh = Attention(pb, device="cuda", with_bwd=True)
    _poison_dq_accumulator(fresh.ws, w, pb.total_q)
    runs.append(fresh.backward(q, k, v, o, lse, dout))  # backward only
    torch.cuda.synchronize()
    att.check()
    fresh.check()
    for dq, dk, dv in runs:
        got = dict(o=o.float().cpu(), lse=lse.float().cpu(), dq=dq.float().cpu(),
                   dk=dk.float().cpu(), dv=dv.float().cpu())
        compare_full(w, inp, got)


def test_workspace_reused_across_problems():
    """One workspace, two packed batches of different lengths back to back
    (plan, forward, backward each): the second backward relies on the first
    leaving the dQ accumulator clear, as it does for every backward."""
    import diffusion_lm_block_bda_b300 as bda
    from diffusion_lm_block_bda_b300 import Problem
    ws_list = [W.custom(BC, 32, 8, 2, 128, [300, 64, 450], name="reuse_a"),
               W.custom(BC, 32, 8, 2, 128, [128, 513, 97], name="reuse_b"),
               W.custom(SC, 32, 8, 2, 128, [416, 160], prefix=[96, 64], name="reuse_c")]
    pbs = [Problem.from_workload(w) for w in ws_list]
    size = max(bda.bda_attn_workspace_size(pb, True) for pb in pbs)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for w, pb in zip(ws_list * 2, pbs * 2):
        inp = W.make_inputs(w, seed=7)
        host = torch.empty(bda.bda_attn_plan_size(pb), dtype=torch.uint8).pin_memory()
        bda.bda_attn_plan(pb, host, ws)
        q, k, v, dout = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.hq, pb.total_q), float("nan"), device="cuda")
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        bda.bda_attn_fwd(pb, q, k, v, o, lse, ws)
        bda.bda_attn_bwd(pb, q, k, v, o, lse, dout, dq, dk, dv, ws)
        torch.cuda.synchronize()
        assert bda.bda_attn_check_status(ws) == bda.BDA_OK
        got = {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
        compare_full(w, inp, got)


def test_forward_and_backward_replay_from_cuda_graph():
    """After bda_attn_plan, forward and backward are capturable: replaying the
    captured launches reproduces the eager results bit for bit (no kernel
    uses atomics whose order varies, except the dQ accumulation, compared
    within the parity tolerance)."""
    import diffusion_lm_block_bda_b300 as bda
    from diffusion_lm_block_bda_b300 import Problem
    for w, bwd in ((W.named("c2"), False),
                   (W.custom(SC, 32, 8, 2, 128, [416, 160], prefix=[96, 64], name="graph_sc"), True)):
        inp = W.make_inputs(w, seed=11)
        pb = Problem.from_workload(w)
        q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
        ws = torch.zeros(bda.bda_attn_workspace_size(pb, bwd), dtype=torch.uint8, device="cuda")
        host = torch.empty(bda.bda_attn_plan_size(pb), dtype=torch.uint8).pin_memory()
        bda.bda_attn_plan(pb, host, ws)
        outs = []
        for captured in (False, True):
            o = torch.full_like(q, float("nan"))
            lse = torch.full((w.hq, pb.total_q), float("nan"), device="cuda")
            grads = [torch.full_like(x, float("nan")) for x in (q, k, v)] if bwd else []
            dout = inp["dout"].cuda() if bwd else None

            def run(stream=None):
                bda.bda_attn_fwd(pb, q, k, v, o, lse, ws, stream)
                if bwd:
                    bda.bda_attn_bwd(pb, q, k, v, o, lse, dout, *grads, ws, stream)

            if captured:
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    run(s)
                g.replay()
                g.replay()
            else:
                run()
            torch.cuda.synchronize()
            assert bda.bda_attn_check_status(ws) == bda.BDA_OK
            outs.append([t.float().cpu() for t in [o, lse] + grads])
        eager, graphed = outs
        assert torch.equal(eager[0], graphed[0]) and torch.equal(eager[1], graphed[1])
        if bwd:
            assert torch.equal(eager[3], graphed[3]) and torch.equal(eager[4], graphed[4])
            got = dict(o=graphed[0], lse=graphed[1], dq=graphed[2], dk=graphed[3], dv=graphed[4])
            compare_full(w, inp, got)
        else:
            compare_full(w, inp, dict(o=graphed[0], lse=graphed[1]), with_bwd=False)


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
    # every key (and every query row) of the shortest and of the longest
    # sequence: the longest holds the longest dK/dV query loops of the batch
    compare_sampled(w, inp, got, seqs=[int(np.argmin(lens))], kv_heads=(7, 8),
                    qrows_fn=lambda L: list(range(L)), krows_fn=lambda L: list(range(L)))
    compare_sampled(w, inp, got, seqs=[int(np.argmax(lens))], kv_heads=(3, 4),
                    qrows_fn=lambda L: list(range(L)), krows_fn=lambda L: list(range(L)))
    check_sum_rules(w, inp, got)


def test_long_block_causal_c5():
    w = W.named("c5")
    inp = W.make_inputs(w, seed=0)
    got = gpu_run(w, inp)
    # dK/dV element by element on the first key tile (keys 0..127: every one
    # of the 32,768 query rows sees them, the dK/dV kernel's longest loop, 1,024
    # query tiles), on a mid-sequence tile and on the last keys
    L = w.seqlens_k[0]
    keys = list(range(128)) + list(range(L // 2, L // 2 + 128)) + _tail_keys(L, 96)
    compare_sampled(w, inp, got, seqs=[0], kv_heads=(0, 1),
                    qrows_fn=lambda n: _sample_rows(n, 24), krows_fn=lambda n: keys)
    check_sum_rules(w, inp, got)


def test_largest_sequence_128k():
    """One 131,072-token sequence, block 128, Hq=32, Hkv=8, d=128: every
    tensor is 4x that of the long-sequence workload and the fp32 dQ
    accumulator spans 2 GiB, so no byte offset or element index may wrap at
    32 bits.  O/LSE/dQ on sampled query rows, dK/dV on the last keys (few
    query rows see them, so the oracle stays cheap) and on a key tile in the
    middle, plus the sum rules over the whole sequence."""
    L = 131072
    w = W.custom(BC, 128, 32, 8, 128, [L], name="block_causal_128k")
    inp = W.make_inputs(w, seed=7)
    got = gpu_run(w, inp)
    keys = list(range(L - 640, L - 512)) + _tail_keys(L, 96)
    compare_sampled(w, inp, got, seqs=[0], kv_heads=(7, 8),
                    qrows_fn=lambda n: _sample_rows(n, 16), krows_fn=lambda n: keys)
    check_sum_rules(w, inp, got)
