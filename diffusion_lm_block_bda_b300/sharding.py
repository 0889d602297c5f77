"""Packed load balancing of whole sequences across data-parallel replicas.

The ORL paper card (thelatestinai.com), Figure 3 caption, packs verified
states and load-balances them across GPUs before replaying them with
staircase attention.  Attention over packed sequences needs no exchange
between GPUs: each replica runs the single-GPU library on its own sequences,
so the only decision is which sequences go where.  The cost of a sequence is
its useful attention work, the number of allowed (query, key) pairs, which
the library counts (bda_attn_count_pairs).  Sequences are assigned longest
first to the least-loaded replica (LPT), so the most loaded replica ends
within one sequence of the mean.
"""
from typing import List, Sequence

from . import Problem, bda_attn_count_pairs


def sequence_costs(w) -> List[int]:
    """Allowed (query, key) pairs of every sequence of workload `w`."""
    out = []
    for s in range(w.nseq):
        lq, lk = w.seqlens_q[s], w.seqlens_k[s]
        pb = Problem([0, lq], [0, lk], w.hq, w.hkv, w.head_dim, w.kind, w.block_size,
                     None if w.prefix is None else [w.prefix[s]])
        out.append(bda_attn_count_pairs(pb))
    return out


def lpt_shard(costs: Sequence[int], n_ranks: int) -> List[List[int]]:
    """Indices of the sequences each rank gets (each list in packing order)."""
    if n_ranks < 1:
        raise ValueError("n_ranks must be >= 1")
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    loads = [0] * n_ranks
    shards: List[List[int]] = [[] for _ in range(n_ranks)]
    for i in order:
        r = min(range(n_ranks), key=lambda k: (loads[k], k))
        shards[r].append(i)
        loads[r] += costs[i]
    return [sorted(s) for s in shards]


def subset(w, idx: Sequence[int], name_suffix: str = ""):
    """The workload restricted to sequences `idx` (re-packed)."""
    from .workloads import Workload
    return Workload(w.name + name_suffix, w.kind, w.block_size, w.hq, w.hkv, w.head_dim,
                    [w.seqlens_q[i] for i in idx], [w.seqlens_k[i] for i in idx],
                    None if w.prefix is None else [w.prefix[i] for i in idx], w.scale,
                    w.with_bwd, w.note)
