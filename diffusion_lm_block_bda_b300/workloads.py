"""Seeded synthetic workloads (shapes and inputs only; no attention arithmetic).

Both the CUDA path's tests/benchmark and the CPU oracle consume these tensors;
this module computes nothing of the method itself.

Shapes follow the QwenDLM-4B attention of the ORL paper card
(thelatestinai.com), Table 9: QKV projection 2560 -> 6144 and O projection
4096 -> 2560, i.e. 32 query heads and 8 KV heads of head_dim 128.  Block sizes
32 and 64 are in the range the ORL announcement thread (24vids.com mirror),
Result 2, reports using (32 and 128).

Recipe: one CPU torch.Generator seeded with `seed` per workload; draws in the
order (1) packed lengths (only for the random-length workload), (2) Q, (3) K,
(4) V, (5) dO, each randn fp32 ~ N(0, 1) then cast to bf16.  The same bf16
tensors go to the GPU and to the oracle.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

BLOCK_CAUSAL = 0
STAIRCASE = 1
STAIRCASE_MULTI = 2


@dataclass
class Workload:
    name: str
    kind: int                      # BLOCK_CAUSAL, STAIRCASE or STAIRCASE_MULTI
    block_size: int
    hq: int
    hkv: int
    head_dim: int
    seqlens_q: List[int]
    seqlens_k: List[int]
    prefix: Optional[List[int]] = None   # staircase prefix length per sequence
    scale: Optional[float] = None        # None -> 1/sqrt(head_dim)
    with_bwd: bool = True
    note: str = ""
    extra: dict = field(default_factory=dict)
    # STAIRCASE_MULTI: per sequence, its copy groups in block order as
    # (copies, visible clean keys) pairs.
    groups: Optional[List[List[Tuple[int, int]]]] = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else self.head_dim ** -0.5

    @property
    def nseq(self) -> int:
        return len(self.seqlens_q)

    @property
    def cu_seqlens_q(self) -> List[int]:
        return _cumsum(self.seqlens_q)

    @property
    def cu_seqlens_k(self) -> List[int]:
        return _cumsum(self.seqlens_k)

    @property
    def total_q(self) -> int:
        return sum(self.seqlens_q)

    @property
    def total_k(self) -> int:
        return sum(self.seqlens_k)


def _cumsum(xs):
    out = [0]
    for x in xs:
        out.append(out[-1] + int(x))
    return out


def packed_lengths(gen: torch.Generator, n: int = 16, lo: int = 512, hi: int = 4096,
                   mult: int = 32) -> List[int]:
    """n lengths uniform in [lo, hi], rounded to a multiple of `mult`, clamped."""
    u = torch.rand(n, generator=gen, dtype=torch.float64)
    out = []
    for x in u.tolist():
        v = lo + (hi - lo) * x
        v = int(round(v / mult)) * mult
        out.append(min(max(v, lo), hi))
    return out


def tiny_block_causal() -> Workload:
    return Workload("tiny_block_causal_L256_B32_hq4_hkv2_d64", BLOCK_CAUSAL, 32, 4, 2, 64,
                    [256], [256], scale=1.0 / 8.0,
                    note="1 sequence L=256, block 32, Hq=4, Hkv=2, d=64, scale 1/8, fwd+bwd")


def decode_step() -> Workload:
    return Workload("decode_prefix2048_block32", BLOCK_CAUSAL, 32, 32, 8, 128, [32], [2080],
                    with_bwd=False,
                    note="32 active-block queries over 2048 committed keys + the block, fwd only")


def packed_replay(gen: Optional[torch.Generator] = None) -> Workload:
    lens = packed_lengths(gen if gen is not None else torch.Generator().manual_seed(0))
    return Workload("packed_block_causal_16xU512_4096_B32", BLOCK_CAUSAL, 32, 32, 8, 128, lens,
                    list(lens),
                    note="16 packed sequences, lengths U[512,4096] rounded to 32, block 32, fwd+bwd")


def staircase_replay() -> Workload:
    L = 1024 + 16 * 32
    return Workload("staircase_8x_prefix1024_16copies_B32", STAIRCASE, 32, 32, 8, 128, [L] * 8,
                    [L] * 8, prefix=[1024] * 8,
                    note="8 trajectories: 1024-token prefix + 16 copies of a 32-token block")


def long_block_causal() -> Workload:
    return Workload("long_block_causal_L32768_B64", BLOCK_CAUSAL, 64, 32, 8, 128, [32768],
                    [32768], note="1 sequence L=32768, block 64, fwd+bwd")


def named(name: str, seed: int = 0) -> Workload:
    """The five workloads by short name c1..c5."""
    if name == "c1":
        return tiny_block_causal()
    if name == "c2":
        return decode_step()
    if name == "c3":
        return packed_replay(torch.Generator().manual_seed(seed))
    if name == "c4":
        return staircase_replay()
    if name == "c5":
        return long_block_causal()
    raise KeyError(name)


WORKLOADS = ("c1", "c2", "c3", "c4", "c5")


def make_inputs(w: Workload, seed: int = 0, with_dout: Optional[bool] = None):
    """Seeded bf16 inputs on the CPU: dict(q, k, v, dout).  For the packed
    workload the generator first re-draws the lengths, so the draw order is
    lengths, Q, K, V, dO."""
    gen = torch.Generator().manual_seed(seed)
    if w.name.startswith("packed_block_causal"):
        packed_lengths(gen)
    tq, tk = w.total_q, w.total_k

    def draw(rows, heads):
        return torch.randn((rows, heads, w.head_dim), generator=gen,
                           dtype=torch.float32).to(torch.bfloat16)

    q = draw(tq, w.hq)
    k = draw(tk, w.hkv)
    v = draw(tk, w.hkv)
    want_do = w.with_bwd if with_dout is None else with_dout
    dout = draw(tq, w.hq) if want_do else None
    return dict(q=q, k=k, v=v, dout=dout)


def custom(kind, block_size, hq, hkv, head_dim, seqlens_q, seqlens_k=None, prefix=None,
           scale=None, name="custom", groups=None) -> Workload:
    """A workload of arbitrary shape (tests use these for ragged / edge cases)."""
    seqlens_k = list(seqlens_q) if seqlens_k is None else list(seqlens_k)
    return Workload(name, kind, block_size, hq, hkv, head_dim, list(seqlens_q), seqlens_k,
                    prefix=None if prefix is None else list(prefix), scale=scale,
                    groups=None if groups is None else [list(g) for g in groups])


def multi_staircase(prefix, groups, block_size=32, hq=32, hkv=8, head_dim=128,
                    name="staircase_multi") -> Workload:
    """Multi-block staircase trajectories: sequence s is a clean prefix of
    prefix[s] tokens followed by its copy groups groups[s] = [(copies,
    visible), ...] in block order; its length is prefix + sum(copies) * B."""
    lens = [int(p) + block_size * sum(int(c) for c, _ in g) for p, g in zip(prefix, groups)]
    return Workload(name, STAIRCASE_MULTI, block_size, hq, hkv, head_dim, lens, list(lens),
                    prefix=[int(p) for p in prefix],
                    groups=[[(int(c), int(v)) for c, v in g] for g in groups])
