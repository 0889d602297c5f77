"""Shared helpers for the GPU parity tests: run the CUDA path through the
C-ABI binding, run the fp64 oracle on the same seeded bf16 inputs, compare.

Tolerances (written here, used by every parity test):
  O    : max-abs <= 2e-2 and relative L2 <= 5e-3
  LSE  : max_i |LSE - LSE*| / max(|LSE*_i|, 1) <= 1e-3
  dQ, dK, dV : relative L2 <= 1e-2 each, the reference norm floored at
               1e-3 * sqrt(elements) (an RMS of 1e-3): relative L2 has no
               meaning for a zero reference, and a gradient can be exactly
               zero (a one-token sequence's softmax over a single key has
               zero derivative) while fp32 rounding of dP - D leaves ~1e-7.
"""
import numpy as np
import torch

import oracle
from diffusion_lm_block_bda_b300 import Attention, Problem, workloads as W

O_MAXABS, O_REL, LSE_REL, GRAD_REL, GRAD_RMS_FLOOR = 2e-2, 5e-3, 1e-3, 1e-2, 1e-3


def rel_l2(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30))


def lse_err(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref) / np.maximum(np.abs(ref), 1.0))) if x.size else 0.0


def check_o(o, ref, what=""):
    o, ref = np.asarray(o, np.float64), np.asarray(ref, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    ma = float(np.max(np.abs(o - ref))) if o.size else 0.0
    rl = rel_l2(o, ref)
    assert ma <= O_MAXABS and rl <= O_REL, f"{what}: O max-abs {ma:.3e}, rel-L2 {rl:.3e}"
    return ma, rl


def check_lse(lse, ref, what=""):
    e = lse_err(lse, ref)
    assert np.isfinite(np.asarray(lse)).all(), f"{what}: non-finite LSE"
    assert e <= LSE_REL, f"{what}: LSE rel err {e:.3e}"
    return e


def check_grad(g, ref, name, what=""):
    g, ref = np.asarray(g, np.float64), np.asarray(ref, np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite {name}"
    floor = GRAD_RMS_FLOOR * np.sqrt(max(ref.size, 1))
    e = float(np.linalg.norm((g - ref).ravel()) / max(np.linalg.norm(ref.ravel()), floor))
    assert e <= GRAD_REL, f"{what}: {name} rel-L2 {e:.3e}"
    return e


def gpu_run(w, inputs, with_bwd=True, device="cuda"):
    """Forward (+ backward) of workload `w` on the GPU.  Outputs are poisoned
    with NaN first so unwritten elements show up.  Returns CPU tensors."""
    pb = Problem.from_workload(w)
    att = Attention(pb, device=device, with_bwd=with_bwd)
    q, k, v = (inputs[n].to(device) for n in ("q", "k", "v"))
    o = torch.full((pb.total_q, w.hq, w.head_dim), float("nan"), dtype=torch.bfloat16,
                   device=device)
    lse = torch.full((w.hq, pb.total_q), float("nan"), dtype=torch.float32, device=device)
    att.forward(q, k, v, o, lse)
    out = dict(o=o, lse=lse)
    if with_bwd:
        dout = inputs["dout"].to(device)
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        att.backward(q, k, v, o, lse, dout, dq, dk, dv)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    att.check()
    return {n: t.float().cpu() for n, t in out.items()}


def oracle_full(w, inputs, with_bwd=True, kv_heads=None):
    """The fp64 oracle's outputs for a whole (small) workload."""
    heads = None
    G = w.hq // w.hkv
    if kv_heads is not None:
        heads = (kv_heads[0] * G, kv_heads[1] * G)
    ref = {}
    ref["o"], ref["lse"] = oracle.fwd(w.kind, w.block_size, w.cu_seqlens_q, w.cu_seqlens_k,
                                      w.prefix, inputs["q"], inputs["k"], inputs["v"], w.hq,
                                      w.hkv, w.softmax_scale, heads=heads, groups=w.groups)
    if with_bwd:
        ref["dq"], ref["dk"], ref["dv"] = oracle.bwd(
            w.kind, w.block_size, w.cu_seqlens_q, w.cu_seqlens_k, w.prefix, inputs["q"],
            inputs["k"], inputs["v"], inputs["dout"], w.hq, w.hkv, w.softmax_scale,
            kv_heads=kv_heads, groups=w.groups)
    return ref


def compare_full(w, inputs, got, with_bwd=True, kv_heads=None, ref=None):
    """Full oracle over every sequence (small workloads); `ref` reuses an
    oracle_full result."""
    heads = None
    G = w.hq // w.hkv
    if kv_heads is not None:
        heads = (kv_heads[0] * G, kv_heads[1] * G)
    if ref is None:
        ref = oracle_full(w, inputs, with_bwd, kv_heads)
    O, LSE = ref["o"], ref["lse"]
    hs = slice(None) if heads is None else slice(*heads)
    ks = slice(None) if kv_heads is None else slice(*kv_heads)
    res = {}
    res["o"] = check_o(got["o"][:, hs].numpy(), O[:, hs], w.name)
    res["lse"] = check_lse(got["lse"][hs].numpy(), LSE[hs], w.name)
    if with_bwd:
        dQ, dK, dV = ref["dq"], ref["dk"], ref["dv"]
        res["dq"] = check_grad(got["dq"][:, hs].numpy(), dQ[:, hs], "dQ", w.name)
        res["dk"] = check_grad(got["dk"][:, ks].numpy(), dK[:, ks], "dK", w.name)
        res["dv"] = check_grad(got["dv"][:, ks].numpy(), dV[:, ks], "dV", w.name)
    return res


def compare_sampled(w, inputs, got, seqs, kv_heads, qrows_fn, krows_fn, with_bwd=True):
    """Oracle on sampled outputs of selected sequences: fwd O/LSE and dQ on
    query rows qrows_fn(Lq), dK/dV on key rows krows_fn(Lk), heads of
    kv_heads = (lo, hi)."""
    G = w.hq // w.hkv
    hs = slice(kv_heads[0] * G, kv_heads[1] * G)
    ks = slice(*kv_heads)
    cq, ck = w.cu_seqlens_q, w.cu_seqlens_k
    acc = {n: ([], []) for n in ("o", "lse", "dq", "dk", "dv")}
    for s in seqs:
        q0, q1, k0, k1 = cq[s], cq[s + 1], ck[s], ck[s + 1]
        qr = qrows_fn(q1 - q0)
        Q, K, V = inputs["q"][q0:q1], inputs["k"][k0:k1], inputs["v"][k0:k1]
        if w.kind == W.STAIRCASE_MULTI:
            g = w.groups[s]
            lay = (w.block_size, w.prefix[s], [c for c, _ in g], [v for _, v in g])
            O, LSE = oracle.fwd_seq_multi(*lay, Q, K, V, w.hq, w.hkv, w.softmax_scale,
                                          heads=(hs.start, hs.stop), rows=qr)
        else:
            P = w.prefix[s] if w.kind == W.STAIRCASE else (k1 - k0)
            O, LSE = oracle.fwd_seq(w.kind, w.block_size, P, Q, K, V, w.hq, w.hkv,
                                    w.softmax_scale, heads=(hs.start, hs.stop), rows=qr)
        acc["o"][0].append(got["o"][q0:q1][qr][:, hs].numpy())
        acc["o"][1].append(O[:, hs])
        acc["lse"][0].append(got["lse"][hs, q0:q1][:, qr].numpy())
        acc["lse"][1].append(LSE[hs])
        if with_bwd:
            kr = krows_fn(k1 - k0)
            if w.kind == W.STAIRCASE_MULTI:
                dQ, dK, dV = oracle.bwd_seq_multi(*lay, Q, K, V, inputs["dout"][q0:q1], w.hq,
                                                  w.hkv, w.softmax_scale, kv_heads=kv_heads,
                                                  qrows=qr, krows=kr)
            else:
                dQ, dK, dV = oracle.bwd_seq(w.kind, w.block_size, P, Q, K, V,
                                            inputs["dout"][q0:q1], w.hq, w.hkv, w.softmax_scale,
                                            kv_heads=kv_heads, qrows=qr, krows=kr)
            acc["dq"][0].append(got["dq"][q0:q1][qr][:, hs].numpy())
            acc["dq"][1].append(dQ[:, hs])
            acc["dk"][0].append(got["dk"][k0:k1][kr][:, ks].numpy())
            acc["dk"][1].append(dK[:, ks])
            acc["dv"][0].append(got["dv"][k0:k1][kr][:, ks].numpy())
            acc["dv"][1].append(dV[:, ks])
    cat = {n: (np.concatenate([x.ravel() for x in a]), np.concatenate([x.ravel() for x in b]))
           for n, (a, b) in acc.items() if a}
    res = {"o": check_o(*cat["o"], w.name), "lse": check_lse(*cat["lse"], w.name)}
    if with_bwd:
        res["dq"] = check_grad(*cat["dq"], "dQ", w.name)
        res["dk"] = check_grad(*cat["dk"], "dK", w.name)
        res["dv"] = check_grad(*cat["dv"], "dV", w.name)
    return res


def check_sum_rules(w, inputs, got):
    """Sum rules that hold at any size (see the oracle's pins): per sequence and
    KV head, the keys' dK sum to zero and the keys' dV sum to the sum of dO over
    the group's query rows."""
    G = w.hq // w.hkv
    cq, ck = w.cu_seqlens_q, w.cu_seqlens_k
    dout = inputs["dout"].double()
    for s in range(w.nseq):
        q0, q1, k0, k1 = cq[s], cq[s + 1], ck[s], ck[s + 1]
        dk = got["dk"][k0:k1].double()
        dv = got["dv"][k0:k1].double()
        for g in range(w.hkv):
            sk = dk[:, g].sum(0)
            scale_k = dk[:, g].abs().sum(0).clamp_min(1e-6)
            assert float((sk.abs() / scale_k).max()) < 2e-2, (s, g, "dK sum")
            want = dout[q0:q1, g * G:(g + 1) * G].sum(dim=(0, 1))
            sv = dv[:, g].sum(0)
            err = float((sv - want).norm() / want.norm().clamp_min(1e-6))
            assert err < 1e-2, (s, g, "dV sum", err)
