"""fp64 CPU oracle for block-causal / staircase attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product library and its Python
binding never do.  It shares no code with the CUDA path.

`oracle.c` holds the plain definition (explicit mask, dense rows, fp64); this
module marshals numpy/torch inputs into it, one packed sequence at a time.
The `*_multi` functions cover the multi-block staircase (several active
blocks per trajectory, each with its own group of copies).
`brute.py` holds an independent NumPy brute force for tiny inputs.

Mask kinds follow the ORL announcement thread (24vids.com mirror),
highlight 3 (block-causal) and Insight 3 (staircase), and the ORL paper card
(thelatestinai.com), Figure 3 caption.  Every array is THD:
Q/O/dO/dQ [T_q][Hq][d], K/V/dK/dV [T_k][Hkv][d], LSE [Hq][T_q].

Parity unpinned: none -- every function here is pinned by tests/test_oracle_*.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build

BLOCK_CAUSAL = 0
STAIRCASE = 1
STAIRCASE_MULTI = 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c_int, c_dbl = ctypes.c_int, ctypes.c_double
        pd = ctypes.POINTER(ctypes.c_double)
        pi = ctypes.POINTER(ctypes.c_int32)
        lib.oracle_allowed.argtypes = [c_int] * 7
        lib.oracle_allowed.restype = c_int
        lib.oracle_mask.argtypes = [c_int] * 5 + [ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_mask.restype = None
        lib.oracle_count_pairs.argtypes = [c_int] * 5
        lib.oracle_count_pairs.restype = ctypes.c_longlong
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = c_int
        lib.oracle_fwd_seq.argtypes = ([c_int] * 8 + [c_dbl, pd, pd, pd, c_int, c_int, pi, c_int,
                                                     pd, pd])
        lib.oracle_fwd_seq.restype = None
        lib.oracle_bwd_seq.argtypes = ([c_int] * 8 + [c_dbl, pd, pd, pd, pd, c_int, c_int, pi,
                                                     c_int, pi, c_int, pd, pd, pd])
        lib.oracle_bwd_seq.restype = None
        grp = [c_int, c_int, c_int, pi, pi, c_int]  # B, P, n_groups, copies, visible, L
        lib.oracle_allowed_multi.argtypes = grp + [c_int, c_int]
        lib.oracle_allowed_multi.restype = c_int
        lib.oracle_mask_multi.argtypes = grp + [ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_mask_multi.restype = None
        lib.oracle_count_pairs_multi.argtypes = grp
        lib.oracle_count_pairs_multi.restype = ctypes.c_longlong
        lib.oracle_fwd_seq_multi.argtypes = grp + [c_int, c_int, c_int, c_dbl, pd, pd, pd, c_int,
                                                   c_int, pi, c_int, pd, pd]
        lib.oracle_fwd_seq_multi.restype = None
        lib.oracle_bwd_seq_multi.argtypes = grp + [c_int, c_int, c_int, c_dbl, pd, pd, pd, pd,
                                                   c_int, c_int, pi, c_int, pi, c_int, pd, pd, pd]
        lib.oracle_bwd_seq_multi.restype = None
        pu8 = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_encode_array.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_long, pu8]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [pu8, ctypes.c_long, pd]
        lib.oracle_e4m3_decode_array.restype = None
        _lib = lib
    return _lib


def _f64(x):
    """Any array-like (numpy, torch CPU of any float dtype) -> C-contiguous fp64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    return r, int(r.size)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def allowed(kind, B, P, Lq, Lk, i, j) -> bool:
    return bool(_load().oracle_allowed(kind, B, P, Lq, Lk, i, j))


def mask(kind, B, P, Lq, Lk) -> np.ndarray:
    m = np.zeros((Lq, Lk), dtype=np.uint8)
    _load().oracle_mask(kind, B, P, Lq, Lk, _ptr(m, ctypes.c_uint8))
    return m.astype(bool)


def count_pairs(kind, B, P, Lq, Lk) -> int:
    return int(_load().oracle_count_pairs(kind, B, P, Lq, Lk))


def _prefix(kind, prefix, s, Lk):
    if kind == STAIRCASE:
        return int(prefix[s])
    return Lk  # unused by the block-causal predicate


def fwd_seq(kind, B, P, Q, K, V, hq, hkv, scale, heads=None, rows=None):
    """One sequence.  Q [Lq][Hq][d], K/V [Lk][Hkv][d] (any float type).
    Returns (O [n][Hq][d], LSE [Hq][n]) in fp64, n = Lq or len(rows); heads
    outside `heads` = (lo, hi) are left NaN."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    Lq, Lk, d = Q.shape[0], K.shape[0], Q.shape[2]
    h_lo, h_hi = heads if heads is not None else (0, hq)
    r, nr = _rows(rows)
    n = Lq if r is None else nr
    O = np.full((n, hq, d), np.nan)
    LSE = np.full((hq, n), np.nan)
    _load().oracle_fwd_seq(kind, B, P, Lq, Lk, hq, hkv, d, scale, _ptr(Q), _ptr(K), _ptr(V),
                           h_lo, h_hi, None if r is None else _ptr(r, ctypes.c_int32), n,
                           _ptr(O), _ptr(LSE))
    return O, LSE


def bwd_seq(kind, B, P, Q, K, V, dO, hq, hkv, scale, kv_heads=None, qrows=None, krows=None):
    """One sequence.  Returns (dQ [nq][Hq][d], dK [nk][Hkv][d], dV [nk][Hkv][d]),
    fp64; entries of heads outside `kv_heads` = (lo, hi) are left NaN."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    Lq, Lk, d = Q.shape[0], K.shape[0], Q.shape[2]
    lo, hi = kv_heads if kv_heads is not None else (0, hkv)
    qr, nq = _rows(qrows)
    kr, nk = _rows(krows)
    nq = Lq if qr is None else nq
    nk = Lk if kr is None else nk
    dQ = np.full((nq, hq, d), np.nan)
    dK = np.full((nk, hkv, d), np.nan)
    dV = np.full((nk, hkv, d), np.nan)
    _load().oracle_bwd_seq(kind, B, P, Lq, Lk, hq, hkv, d, scale, _ptr(Q), _ptr(K), _ptr(V),
                           _ptr(dO), lo, hi, None if qr is None else _ptr(qr, ctypes.c_int32), nq,
                           None if kr is None else _ptr(kr, ctypes.c_int32), nk, _ptr(dQ),
                           _ptr(dK), _ptr(dV))
    return dQ, dK, dV


def fwd(kind, B, cu_q, cu_k, prefix, Q, K, V, hq, hkv, scale, heads=None, groups=None):
    """Packed varlen forward: cu_q/cu_k int [nseq+1]; prefix [nseq] (staircase
    kinds) or None; groups (STAIRCASE_MULTI) per sequence a list of (copies,
    visible) pairs.  Returns (O [T_q][Hq][d], LSE [Hq][T_q]) fp64."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    cu_q = [int(x) for x in cu_q]
    cu_k = [int(x) for x in cu_k]
    Tq, d = Q.shape[0], Q.shape[2]
    O = np.full((Tq, hq, d), np.nan)
    LSE = np.full((hq, Tq), np.nan)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if q1 == q0:
            continue
        if kind == STAIRCASE_MULTI:
            g = groups[s]
            o, l = fwd_seq_multi(B, int(prefix[s]), [c for c, _ in g], [v for _, v in g],
                                 Q[q0:q1], K[k0:k1], V[k0:k1], hq, hkv, scale, heads)
        else:
            P = _prefix(kind, prefix, s, k1 - k0)
            o, l = fwd_seq(kind, B, P, Q[q0:q1], K[k0:k1], V[k0:k1], hq, hkv, scale, heads)
        O[q0:q1] = o
        LSE[:, q0:q1] = l
    return O, LSE


def bwd(kind, B, cu_q, cu_k, prefix, Q, K, V, dO, hq, hkv, scale, kv_heads=None, groups=None):
    """Packed varlen backward (arguments as for fwd).  Returns (dQ, dK, dV)
    fp64 in THD layout."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    cu_q = [int(x) for x in cu_q]
    cu_k = [int(x) for x in cu_k]
    dQ = np.full(Q.shape, np.nan)
    dK = np.full(K.shape, np.nan)
    dV = np.full(V.shape, np.nan)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if k1 == k0:
            continue
        if q1 == q0:
            dK[k0:k1] = 0.0
            dV[k0:k1] = 0.0
            continue
        if kind == STAIRCASE_MULTI:
            g = groups[s]
            dq, dk, dv = bwd_seq_multi(B, int(prefix[s]), [c for c, _ in g], [v for _, v in g],
                                       Q[q0:q1], K[k0:k1], V[k0:k1], dO[q0:q1], hq, hkv, scale,
                                       kv_heads)
        else:
            P = _prefix(kind, prefix, s, k1 - k0)
            dq, dk, dv = bwd_seq(kind, B, P, Q[q0:q1], K[k0:k1], V[k0:k1], dO[q0:q1], hq, hkv,
                                 scale, kv_heads)
        dQ[q0:q1] = dq
        dK[k0:k1] = dk
        dV[k0:k1] = dv
    return dQ, dK, dV


# ---------------------------------------------------- multi-block staircase
# One trajectory (Lq = Lk = L): a clean prefix [0, P), block-causal in blocks
# of B; then groups g = 0.. of copies[g] copies (B tokens each) of one active
# block, whose copies see the clean keys [0, visible[g]) and themselves.
# Requires sum(copies) * B == L - P and 0 <= visible[g] <= P.

def _groups(B, P, copies, visible, L):
    c = np.ascontiguousarray(np.asarray(copies, dtype=np.int32))
    v = np.ascontiguousarray(np.asarray(visible, dtype=np.int32))
    if c.shape != v.shape or c.ndim != 1:
        raise ValueError("copies and visible: one entry per group")
    if int(c.sum()) * B != L - P or (c < 0).any() or (v < 0).any() or (v > P).any():
        raise ValueError("groups do not tile [P, L) or see past the prefix")
    return (B, P, int(c.size), _ptr(c, ctypes.c_int32), _ptr(v, ctypes.c_int32), L), (c, v)


def allowed_multi(B, P, copies, visible, L, i, j) -> bool:
    g, keep = _groups(B, P, copies, visible, L)
    return bool(_load().oracle_allowed_multi(*g, i, j))


def mask_multi(B, P, copies, visible, L) -> np.ndarray:
    g, keep = _groups(B, P, copies, visible, L)
    m = np.zeros((L, L), dtype=np.uint8)
    _load().oracle_mask_multi(*g, _ptr(m, ctypes.c_uint8))
    return m.astype(bool)


def count_pairs_multi(B, P, copies, visible, L) -> int:
    g, keep = _groups(B, P, copies, visible, L)
    return int(_load().oracle_count_pairs_multi(*g))


def fwd_seq_multi(B, P, copies, visible, Q, K, V, hq, hkv, scale, heads=None, rows=None):
    """fwd_seq for one multi-block staircase trajectory."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    L, d = Q.shape[0], Q.shape[2]
    g, keep = _groups(B, P, copies, visible, L)
    h_lo, h_hi = heads if heads is not None else (0, hq)
    r, nr = _rows(rows)
    n = L if r is None else nr
    O = np.full((n, hq, d), np.nan)
    LSE = np.full((hq, n), np.nan)
    _load().oracle_fwd_seq_multi(*g, hq, hkv, d, scale, _ptr(Q), _ptr(K), _ptr(V), h_lo, h_hi,
                                 None if r is None else _ptr(r, ctypes.c_int32), n, _ptr(O),
                                 _ptr(LSE))
    return O, LSE


def bwd_seq_multi(B, P, copies, visible, Q, K, V, dO, hq, hkv, scale, kv_heads=None, qrows=None,
                  krows=None):
    """bwd_seq for one multi-block staircase trajectory."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    L, d = Q.shape[0], Q.shape[2]
    g, keep = _groups(B, P, copies, visible, L)
    lo, hi = kv_heads if kv_heads is not None else (0, hkv)
    qr, nq = _rows(qrows)
    kr, nk = _rows(krows)
    nq = L if qr is None else nq
    nk = L if kr is None else nk
    dQ = np.full((nq, hq, d), np.nan)
    dK = np.full((nk, hkv, d), np.nan)
    dV = np.full((nk, hkv, d), np.nan)
    _load().oracle_bwd_seq_multi(*g, hq, hkv, d, scale, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), lo,
                                 hi, None if qr is None else _ptr(qr, ctypes.c_int32), nq,
                                 None if kr is None else _ptr(kr, ctypes.c_int32), nk, _ptr(dQ),
                                 _ptr(dK), _ptr(dV))
    return dQ, dK, dV


def count_pairs_packed(kind, B, cu_q, cu_k, prefix, groups=None) -> int:
    """Allowed (i, j) pairs summed over the packed sequences (per head)."""
    n = 0
    for s in range(len(cu_q) - 1):
        Lq, Lk = int(cu_q[s + 1] - cu_q[s]), int(cu_k[s + 1] - cu_k[s])
        if kind == STAIRCASE_MULTI:
            g = groups[s]
            n += count_pairs_multi(B, int(prefix[s]), [c for c, _ in g], [v for _, v in g], Lq)
        else:
            n += count_pairs(kind, B, _prefix(kind, prefix, s, Lk), Lq, Lk)
    return n


# ------------------------------------------------------------ FP8 (e4m3)
# The KV-cache format of the decode engine on the ORL paper card (Table 11
# caption: NVFP4 configurations use an FP8 KV cache).  oracle.c holds the
# OCP E4M3 definition: encode = round to nearest, ties to even, saturating
# at 448; decode = the exact value of a code.

def e4m3_encode(x) -> np.ndarray:
    """fp32 values (any array-like; converted to float32 first) -> uint8 codes."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).ravel()
    out = np.zeros(a.size, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(a.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), a.size,
                                     _ptr(out, ctypes.c_uint8))
    return out.reshape(np.shape(x))


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> fp64 values (NaN for the NaN codes)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8)).ravel()
    out = np.zeros(c.size, dtype=np.float64)
    _load().oracle_e4m3_decode_array(_ptr(c, ctypes.c_uint8), c.size, _ptr(out))
    return out.reshape(np.shape(codes))


def quantize_kv_e4m3(x, scale) -> np.ndarray:
    """Codes of the FP8 KV cache: e4m3(fl32(x / scale[h])) for x [rows][heads][d]
    (bf16 or fp32 values) and fp32 scales [heads]; the quotient is the IEEE
    fp32 division."""
    xf = np.asarray(_f64(x), dtype=np.float32)
    s = np.asarray(scale, dtype=np.float32).reshape(1, -1, 1)
    return e4m3_encode(xf / s)


def dequantize_kv_e4m3(codes, scale) -> np.ndarray:
    """fp64 values code * scale[h] of an FP8 KV cache [rows][heads][d]."""
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64).reshape(1, -1, 1)
