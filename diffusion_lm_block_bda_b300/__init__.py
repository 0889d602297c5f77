"""Block-causal and staircase attention for B300 (sm_103a).

Python binding of libbda_attn.so (include/bda_attn.h).  The functions named
like the C entry points marshal arguments and call them; torch only provides
device memory and the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels: if the library is missing this module
raises instead of falling back to anything else.

Convenience layer: `Attention(...)` holds the problem description, plans once,
allocates the workspace with torch and exposes `forward` / `backward`.
"""
import ctypes
import os

import torch

from . import workloads  # noqa: F401  (seeded synthetic workloads)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbda_attn.so")

BDA_OK = 0
BDA_ERR_INVALID_ARG = 1
BDA_ERR_UNSUPPORTED = 2
BDA_ERR_WORKSPACE = 3
BDA_ERR_CUDA = 4
BDA_ERR_DEVICE_TIMEOUT = 5

BDA_MASK_BLOCK_CAUSAL = 0
BDA_MASK_STAIRCASE = 1
BDA_MASK_STAIRCASE_MULTI = 2

EXPORTED = (
    "bda_attn_plan_size", "bda_attn_workspace_size", "bda_attn_plan", "bda_attn_plan_host",
    "bda_attn_fwd",
    "bda_attn_bwd", "bda_attn_bwd_preprocess", "bda_attn_bwd_dkdv", "bda_attn_bwd_dq_convert",
    "bda_attn_count_pairs", "bda_attn_check_status", "bda_status_string",
    "bda_last_cuda_error", "bda_attn_fwd_noalloc", "bda_attn_fwd_noalloc_check_status",
    "bda_testing_arm_wait_timeout", "bda_attn_fwd_fp8kv", "bda_kv_quantize_fp8",
    "bda_kv_fp8_scales", "bda_testing_force_forward_kernel",
)


class BdaMaskDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("prefix_len_host", ctypes.POINTER(ctypes.c_int32)),
                ("group_offsets_host", ctypes.POINTER(ctypes.c_int32)),
                ("group_copies_host", ctypes.POINTER(ctypes.c_int32)),
                ("group_visible_host", ctypes.POINTER(ctypes.c_int32))]


class BdaProblem(ctypes.Structure):
    _fields_ = [("nseq", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("cu_seqlens_q_host", ctypes.POINTER(ctypes.c_int32)),
                ("cu_seqlens_k_host", ctypes.POINTER(ctypes.c_int32))]


class BdaError(RuntimeError):
    def __init__(self, status, where):
        self.status = int(status)
        msg = f"{where}: {string(self.status)} (status {self.status})"
        if self.status == BDA_ERR_CUDA:
            msg += f": {lib().bda_last_cuda_error().decode()}"
        super().__init__(msg)


_lib = None


def lib():
    """Load libbda_attn.so (build it with `python -m diffusion_lm_block_bda_b300.build`)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbda_attn.so not found at {LIB_PATH}; build it first "
                               "(python -m diffusion_lm_block_bda_b300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, M = ctypes.POINTER(BdaProblem), ctypes.POINTER(BdaMaskDesc)
        vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
        sig = {
            "bda_attn_plan_size": ([P, M], sz),
            "bda_attn_workspace_size": ([P, M, ctypes.c_int], sz),
            "bda_attn_plan": ([P, M, vp, sz, vp, sz, st], ctypes.c_int),
            "bda_attn_plan_host": ([P, M, vp, sz], ctypes.c_int),
            "bda_attn_fwd": ([P, M, vp, vp, vp, vp, vp, vp, sz, st], ctypes.c_int),
            "bda_attn_bwd": ([P, M, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, st], ctypes.c_int),
            "bda_attn_bwd_preprocess": ([P, M, vp, vp, vp, sz, st], ctypes.c_int),
            "bda_attn_bwd_dkdv": ([P, M, vp, vp, vp, vp, vp, vp, vp, vp, sz, st], ctypes.c_int),
            "bda_attn_bwd_dq_convert": ([P, M, vp, vp, sz, st], ctypes.c_int),
            "bda_attn_count_pairs": ([P, M], ctypes.c_longlong),
            "bda_attn_check_status": ([vp, sz, st], ctypes.c_int),
            "bda_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "bda_last_cuda_error": ([], ctypes.c_char_p),
            "bda_attn_fwd_noalloc": ([P, M, vp, vp, vp, vp, vp, st], ctypes.c_int),
            "bda_attn_fwd_noalloc_check_status": ([st], ctypes.c_int),
            "bda_testing_arm_wait_timeout": ([ctypes.c_int, ctypes.c_ulonglong], ctypes.c_int),
            "bda_attn_fwd_fp8kv": ([P, M, vp, vp, vp, vp, vp, vp, vp, vp, sz, st], ctypes.c_int),
            "bda_kv_quantize_fp8": ([vp, vp, vp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, st],
                                    ctypes.c_int),
            "bda_kv_fp8_scales": ([vp, vp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, st],
                                  ctypes.c_int),
            "bda_testing_force_forward_kernel": ([ctypes.c_int], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def string(status: int) -> str:
    return lib().bda_status_string(int(status)).decode()


def _check(status, where):
    if status != BDA_OK:
        raise BdaError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32(xs):
    xs = [int(x) for x in xs]
    return (ctypes.c_int32 * max(1, len(xs)))(*xs)


class Problem:
    """Host-side problem + mask description (keeps the ctypes arrays alive)."""

    def __init__(self, cu_seqlens_q, cu_seqlens_k, hq, hkv, head_dim, kind, block_size,
                 prefix_len=None, softmax_scale=0.0, groups=None):
        """groups (BDA_MASK_STAIRCASE_MULTI): per sequence a list of
        (copies, visible) pairs, one per active block, in order."""
        self.cu_q = [int(x) for x in cu_seqlens_q]
        self.cu_k = [int(x) for x in cu_seqlens_k]
        self.hq, self.hkv, self.head_dim = int(hq), int(hkv), int(head_dim)
        self.kind, self.block_size = int(kind), int(block_size)
        self.prefix_len = None if prefix_len is None else [int(x) for x in prefix_len]
        self._cq, self._ck = _i32(self.cu_q), _i32(self.cu_k)
        self._pf = _i32(self.prefix_len) if self.prefix_len is not None else None
        self.groups = None if groups is None else [[(int(c), int(v)) for c, v in g] for g in groups]
        self._go = self._gc = self._gv = None
        if self.groups is not None:
            offs = [0]
            for g in self.groups:
                offs.append(offs[-1] + len(g))
            self._go = _i32(offs)
            self._gc = _i32([c for g in self.groups for c, _ in g] or [0])
            self._gv = _i32([v for g in self.groups for _, v in g] or [0])
        self.prob = BdaProblem(len(self.cu_q) - 1, self.hq, self.hkv, self.head_dim,
                               float(softmax_scale or 0.0), self._cq, self._ck)
        self.mask = BdaMaskDesc(self.kind, self.block_size, self._pf, self._go, self._gc,
                                self._gv)

    @property
    def total_q(self):
        return self.cu_q[-1]

    @property
    def total_k(self):
        return self.cu_k[-1]

    @classmethod
    def from_workload(cls, w):
        return cls(w.cu_seqlens_q, w.cu_seqlens_k, w.hq, w.hkv, w.head_dim, w.kind, w.block_size,
                   w.prefix, w.scale or 0.0, getattr(w, "groups", None))

    def refs(self):
        return ctypes.byref(self.prob), ctypes.byref(self.mask)


# ------------------------------------------------ C-ABI mirrors (same names)

def bda_attn_plan_size(pb: Problem) -> int:
    return int(lib().bda_attn_plan_size(*pb.refs()))


def bda_attn_workspace_size(pb: Problem, with_bwd: bool) -> int:
    return int(lib().bda_attn_workspace_size(*pb.refs(), int(bool(with_bwd))))


def bda_attn_count_pairs(pb: Problem) -> int:
    return int(lib().bda_attn_count_pairs(*pb.refs()))


def bda_attn_plan(pb: Problem, host_plan, ws, stream=None):
    _check(lib().bda_attn_plan(*pb.refs(), _ptr(host_plan), host_plan.numel(), _ptr(ws),
                               ws.numel(), _stream(stream)), "bda_attn_plan")


def bda_attn_plan_host(pb: Problem, host_plan):
    _check(lib().bda_attn_plan_host(*pb.refs(), _ptr(host_plan), host_plan.numel()),
           "bda_attn_plan_host")


def bda_attn_fwd(pb: Problem, q, k, v, o, lse, ws, stream=None):
    _check(lib().bda_attn_fwd(*pb.refs(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws),
                              ws.numel(), _stream(stream)), "bda_attn_fwd")


def bda_attn_fwd_noalloc(pb: Problem, q, k, v, o, lse, stream=None):
    """Forward without a workspace (for callers that cannot allocate device
    memory where they run attention): the plan lives in a fixed 1 MiB array
    inside the library, shared by every call; overlapping calls race, and a
    stream under graph capture is refused."""
    _check(lib().bda_attn_fwd_noalloc(*pb.refs(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _stream(stream)), "bda_attn_fwd_noalloc")


def bda_attn_fwd_noalloc_check_status(stream=None) -> int:
    """Status of the latest no-alloc forward on the current device (syncs the stream)."""
    return int(lib().bda_attn_fwd_noalloc_check_status(_stream(stream)))


def bda_testing_arm_wait_timeout(stage: int, timeout_ns: int) -> int:
    """Testing only: the next launch of `stage` (1 forward, 2 dK/dV) lets one
    bounded wait run out after timeout_ns; 0 disarms."""
    return int(lib().bda_testing_arm_wait_timeout(int(stage), int(timeout_ns)))


def bda_attn_fwd_fp8kv(pb: Problem, q, k8, v8, k_scale, v_scale, o, lse, ws, stream=None):
    """Forward over an FP8 (e4m3) KV cache: k8/v8 uint8 codes [T_k][Hkv][d],
    k_scale/v_scale fp32 [Hkv] dequantisation scales (device)."""
    _check(lib().bda_attn_fwd_fp8kv(*pb.refs(), _ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale),
                                    _ptr(v_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(stream)), "bda_attn_fwd_fp8kv")


def bda_kv_quantize_fp8(x, x8, scale, stream=None):
    """e4m3 codes of x / scale[h] for bf16 x [rows][heads][d] into uint8 x8."""
    rows, heads, d = x.shape
    _check(lib().bda_kv_quantize_fp8(_ptr(x), _ptr(x8), _ptr(scale), rows, heads, d,
                                     _stream(stream)), "bda_kv_quantize_fp8")


def bda_kv_fp8_scales(x, scale, stream=None):
    """Per-head scales max|x| / 448 (1 for an all-zero head) into fp32 scale [heads]."""
    rows, heads, d = x.shape
    _check(lib().bda_kv_fp8_scales(_ptr(x), _ptr(scale), rows, heads, d, _stream(stream)),
           "bda_kv_fp8_scales")


def bda_testing_force_forward_kernel(which: int) -> int:
    """Testing only: 0 the plan's choice, 1 persistent forward, 2 split forward."""
    return int(lib().bda_testing_force_forward_kernel(int(which)))


def bda_attn_bwd(pb: Problem, q, k, v, o, lse, dout, dq, dk, dv, ws, stream=None):
    _check(lib().bda_attn_bwd(*pb.refs(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                              _stream(stream)), "bda_attn_bwd")


def bda_attn_bwd_preprocess(pb: Problem, o, dout, ws, stream=None):
    _check(lib().bda_attn_bwd_preprocess(*pb.refs(), _ptr(o), _ptr(dout), _ptr(ws), ws.numel(),
                                         _stream(stream)), "bda_attn_bwd_preprocess")


def bda_attn_bwd_dkdv(pb: Problem, q, k, v, lse, dout, dk, dv, ws, stream=None):
    _check(lib().bda_attn_bwd_dkdv(*pb.refs(), _ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(dout),
                                   _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)),
           "bda_attn_bwd_dkdv")


def bda_attn_bwd_dq_convert(pb: Problem, dq, ws, stream=None):
    _check(lib().bda_attn_bwd_dq_convert(*pb.refs(), _ptr(dq), _ptr(ws), ws.numel(),
                                         _stream(stream)), "bda_attn_bwd_dq_convert")


def bda_attn_check_status(ws, stream=None) -> int:
    return int(lib().bda_attn_check_status(_ptr(ws), ws.numel(), _stream(stream)))


# ------------------------------------------------------------ convenience

class Attention:
    """Plans once, owns the workspace (torch uint8 on `device`) and a pinned
    host plan buffer, and runs forward / backward through the C ABI."""

    def __init__(self, problem: Problem, device="cuda", with_bwd=True, stream=None):
        self.pb = problem
        self.device = torch.device(device)
        self.with_bwd = with_bwd
        n_ws = bda_attn_workspace_size(problem, with_bwd)
        n_plan = bda_attn_plan_size(problem)
        if n_ws == 0 or n_plan == 0:
            # The library validates; reproduce its status for a clear error.
            probe = torch.empty(16, dtype=torch.uint8)
            st = lib().bda_attn_plan(*problem.refs(), _ptr(probe), 16, None, 0, None)
            raise BdaError(st if st != BDA_OK else BDA_ERR_INVALID_ARG, "Attention")
        self.ws = torch.zeros(n_ws, dtype=torch.uint8, device=self.device)
        self.host_plan = torch.empty(n_plan, dtype=torch.uint8).pin_memory()
        self.plan(stream)

    def plan(self, stream=None):
        bda_attn_plan(self.pb, self.host_plan, self.ws, stream)

    def forward(self, q, k, v, o=None, lse=None, stream=None):
        pb = self.pb
        if o is None:
            o = torch.empty((pb.total_q, pb.hq, pb.head_dim), dtype=torch.bfloat16, device=q.device)
        if lse is None:
            lse = torch.empty((pb.hq, pb.total_q), dtype=torch.float32, device=q.device)
        bda_attn_fwd(pb, q, k, v, o, lse, self.ws, stream)
        return o, lse

    def backward(self, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, stream=None):
        if not self.with_bwd:
            raise RuntimeError("Attention was created with with_bwd=False")
        pb = self.pb
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        bda_attn_bwd(pb, q, k, v, o, lse, dout, dq, dk, dv, self.ws, stream)
        return dq, dk, dv

    def check(self, stream=None):
        st = bda_attn_check_status(self.ws, stream)
        _check(st, "device status")
