"""GPU checks of the FP8 (e4m3) KV-cache path (the decode engine of the ORL
paper card runs its NVFP4 configurations with an FP8 KV cache, Table 11
caption), through the C ABI:
- bda_kv_fp8_scales equals max|x| / 448 per head, computed on the host;
- bda_kv_quantize_fp8's codes equal the oracle's e4m3 codes bit for bit
  (both divide in fp32 and round to nearest even, saturating at 448), on
  the decode step's K/V and on a tensor of edge values;
- bda_attn_fwd_fp8kv matches the fp64 oracle's attention over the
  dequantised K and V (the oracle's own codes times the scales) within the
  bf16 forward tolerances, on the decode step and on other mask shapes."""
import numpy as np
import pytest
import torch

import oracle
import diffusion_lm_block_bda_b300 as bda
from diffusion_lm_block_bda_b300 import Attention, Problem, workloads as W

from _parity import check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


def _host_scales(x):
    amax = x.float().abs().amax(dim=(0, 2)).numpy().astype(np.float32)
    return np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)


def test_scales_and_codes_match_the_oracle():
    w = W.named("c2")
    inp = W.make_inputs(w, seed=2, with_dout=False)
    for name in ("k", "v"):
        x = inp[name] * 3.0  # a range wider than N(0, 1)
        xd = x.cuda()
        scale = torch.empty(w.hkv, dtype=torch.float32, device="cuda")
        bda.bda_kv_fp8_scales(xd, scale)
        codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        bda.bda_kv_quantize_fp8(xd, codes, scale)
        torch.cuda.synchronize()
        s_host = _host_scales(x)
        assert np.array_equal(scale.cpu().numpy(), s_host)
        assert np.array_equal(codes.cpu().numpy(), oracle.quantize_kv_e4m3(x, s_host))


def test_codes_of_edge_values():
    vals = [0.0, -0.0, 1e-30, -1e-30, 2.0 ** -9, 1.5 * 2.0 ** -9, 2.0 ** -10, 1.0625, 1.1875,
            447.0, 448.0, 460.0, 464.0, 1e4, -1e4, 3.0e38, float("inf"), float("-inf")]
    x = torch.tensor(vals * 8, dtype=torch.float32)[:128].to(torch.bfloat16)
    x = x.reshape(1, 1, 128).repeat(16, 2, 1)
    scale = np.array([1.0, 0.5], dtype=np.float32)
    codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    bda.bda_kv_quantize_fp8(x.cuda(), codes, torch.from_numpy(scale).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), oracle.quantize_kv_e4m3(x, scale))


CASES = {
    "decode_c2": lambda: W.named("c2"),
    "tiny_d64": lambda: W.custom(W.BLOCK_CAUSAL, 32, 4, 2, 64, [256], name="fp8_tiny"),
    "decode_batch": lambda: W.custom(W.BLOCK_CAUSAL, 32, 32, 8, 128, [32, 32, 5],
                                     [2080, 700, 133], name="fp8_batch"),
    "staircase": lambda: W.custom(W.STAIRCASE, 32, 8, 2, 128, [1536, 700], prefix=[1024, 316],
                                  name="fp8_sc"),
    "multi": lambda: W.multi_staircase([1000, 130], [[(3, 0), (2, 640), (1, 1000)], [(4, 130)]],
                                       block_size=16, hq=8, hkv=2),
    "packed_long": lambda: W.custom(W.BLOCK_CAUSAL, 64, 8, 2, 128, [3000, 1100], name="fp8_pk"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_forward_matches_oracle(name):
    w = CASES[name]()
    inp = W.make_inputs(w, seed=23, with_dout=False)
    pb = Problem.from_workload(w)
    q = inp["q"].cuda()
    k8, v8, scales, deq = [], [], [], {}
    for n in ("k", "v"):
        s_host = _host_scales(inp[n])
        codes_o = oracle.quantize_kv_e4m3(inp[n], s_host)
        deq[n] = oracle.dequantize_kv_e4m3(codes_o, s_host)
        sd = torch.from_numpy(s_host).cuda()
        c = torch.empty(inp[n].shape, dtype=torch.uint8, device="cuda")
        bda.bda_kv_quantize_fp8(inp[n].cuda(), c, sd)
        scales.append(sd)
        (k8 if n == "k" else v8).append(c)
    att = Attention(pb, device="cuda", with_bwd=False)
    o = torch.full((pb.total_q, w.hq, w.head_dim), float("nan"), dtype=torch.bfloat16,
                   device="cuda")
    lse = torch.full((w.hq, pb.total_q), float("nan"), dtype=torch.float32, device="cuda")
    bda.bda_attn_fwd_fp8kv(pb, q, k8[0], v8[0], scales[0], scales[1], o, lse, att.ws)
    torch.cuda.synchronize()
    att.check()
    O, LSE = oracle.fwd(w.kind, w.block_size, w.cu_seqlens_q, w.cu_seqlens_k, w.prefix,
                        inp["q"], deq["k"], deq["v"], w.hq, w.hkv, w.softmax_scale,
                        groups=w.groups)
    check_o(o.float().cpu().numpy(), O, w.name)
    check_lse(lse.cpu().numpy(), LSE, w.name)
