"""Python binding of the GB300 per-token adapter routing library (include/molora.h).

Argument marshalling only: every function here checks shapes and dtypes of torch CUDA
tensors, passes their device pointers and the current CUDA stream through ctypes to the
C ABI, and raises on a non-OK status.  All computation happens in the library's CUDA
kernels; there is no CPU or PyTorch fallback.  If the compiled library is missing the
first call raises: build it with ``token_adapter_routing_gb300.build.build()``.

Method: "MoLoRA: Composable Specialization via Per-Token Adapter Routing" -- vocabulary
routing and the learned top-k router (Table 1), dispatch by histogram / pointer arrays /
grouping (Table 1, Figure 2), and the batched LoRA apply over a GPU-resident hot set
(Figure 2, Figure 4, Table 10 shapes).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "molora_route_vocab", "molora_router_topk", "molora_dispatch", "molora_route_vocab_dispatch",
    "molora_lora_apply", "molora_lora_apply_masked_pass", "molora_select_path", "molora_selftest_bounded_wait", "library_path",
    "load_library",
    "MoloraError", "PATHS", "DEV_TOKEN_OUTSIDE_RANGES", "DEV_BAD_RANGES", "DEV_BAD_ADAPTER_ID",
    "DEV_BAD_PERMUTATION", "DEV_WAIT_TIMEOUT", "MAX_ADAPTERS", "ROUTER_HIDDEN",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3
F32, BF16 = 0, 1
PATHS = {"auto": 0, "scalar": 1, "grouped": 2, "dense": 3}
PATH_NAMES = {v: k for k, v in PATHS.items()}
DEV_TOKEN_OUTSIDE_RANGES = 0x1
DEV_BAD_RANGES = 0x2
DEV_BAD_ADAPTER_ID = 0x4
DEV_BAD_PERMUTATION = 0x8
DEV_WAIT_TIMEOUT = 0x10
MAX_ADAPTERS = 64
ROUTER_HIDDEN = 64

EXPORTED = ("molora_route_vocab", "molora_router_topk", "molora_dispatch", "molora_route_vocab_dispatch",
            "molora_lora_apply", "molora_router_lora_apply", "molora_route_vocab_lora_apply",
            "molora_lora_apply_ex", "molora_lora_apply_bf16y", "molora_lora_apply_indirect", "molora_lora_apply_masked_pass", "molora_select_path",
            "molora_status_string", "molora_version", "molora_selftest_bounded_wait")


class MoloraError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Loads the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: build it with token_adapter_routing_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I64, I32, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_int
    lib.molora_route_vocab.argtypes = [P, I64, P, I32, P, P, P]
    lib.molora_router_topk.argtypes = [P, S, I64, I32, P, P, P, P, I32, I32, P, P, P, P]
    lib.molora_dispatch.argtypes = [P, I64, I32, I32, P, P, P, P, P]
    lib.molora_route_vocab_dispatch.argtypes = [P, I64, P, I32, P, P, P, P, P, P]
    lib.molora_lora_apply.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, P]
    lib.molora_lora_apply_ex.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, S, P]
    lib.molora_lora_apply_bf16y.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, S, P]
    lib.molora_lora_apply_indirect.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, I32,
                                               P, S, P]
    lib.molora_router_lora_apply.argtypes = [P, S, I64, I32, I32, P, P, P, P, P, P, I32, I32, I32, F, P, P, P, P,
                                             I32, P, P]
    lib.molora_route_vocab_lora_apply.argtypes = [P, I64, P, I32, P, S, I32, I32, P, P, I32, F, P, I32, P, P, P, P,
                                                  P, P]
    lib.molora_lora_apply_masked_pass.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, I32, F, P, P, S, P]
    lib.molora_select_path.argtypes = [S, I64, I32, I32, I32, I32, I32]
    lib.molora_status_string.argtypes = [S]
    lib.molora_status_string.restype = ctypes.c_char_p
    lib.molora_version.argtypes = []
    lib.molora_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P, P]
    for name in ("molora_route_vocab", "molora_router_topk", "molora_dispatch", "molora_route_vocab_dispatch",
                 "molora_lora_apply", "molora_lora_apply_ex", "molora_lora_apply_bf16y", "molora_lora_apply_indirect",
                 "molora_lora_apply_masked_pass", "molora_select_path", "molora_version",
                 "molora_selftest_bounded_wait"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != OK:
        raise MoloraError(fn, status, load_library().molora_status_string(status).decode())


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def molora_route_vocab(tok, starts, adapter=None, err_word=None, stream=None):
    """adapter[t] = a with starts[a] <= tok[t] < starts[a+1], else -1 (int32 [N])."""
    _cuda(tok, "tok", torch.int32, 1)
    _cuda(starts, "starts", torch.int32, 1)
    N, K = tok.numel(), starts.numel() - 1
    if adapter is None:
        adapter = torch.empty(N, dtype=torch.int32, device=tok.device)
    _cuda(adapter, "adapter", torch.int32)
    _check("molora_route_vocab", load_library().molora_route_vocab(
        _p(tok), N, _p(starts), K, _p(adapter), _p(err_word), _stream(stream)))
    return adapter


def molora_router_topk(x, W1, W2, k, b1=None, b2=None, logits=None, ids=None, w=None, want_logits=True,
                       stream=None):
    """Learned router: returns (logits fp32 [N,K] or None, ids int32 [N,k], w fp32 [N,k])."""
    _cuda(x, "x", None, 2)
    N, d_in = x.shape
    _cuda(W1, "W1", x.dtype, 2)
    _cuda(W2, "W2", x.dtype, 2)
    if W1.shape != (d_in, ROUTER_HIDDEN) or W2.shape[0] != ROUTER_HIDDEN:
        raise ValueError("W1 must be [d_in, 64] and W2 [64, K]")
    K = W2.shape[1]
    dev = x.device
    if b1 is not None:
        _cuda(b1, "b1", torch.float32)
    if b2 is not None:
        _cuda(b2, "b2", torch.float32)
    if logits is None and want_logits:
        logits = torch.empty(N, K, dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty(N, k, dtype=torch.int32, device=dev)
    if w is None:
        w = torch.empty(N, k, dtype=torch.float32, device=dev)
    _check("molora_router_topk", load_library().molora_router_topk(
        _p(x), _dtype_code(x), N, d_in, _p(W1), _p(b1), _p(W2), _p(b2), K, k, _p(logits), _p(ids), _p(w),
        _stream(stream)))
    return logits, ids, w


def molora_dispatch(ids, K, counts=None, offsets=None, perm=None, err_word=None, stream=None):
    """Histogram, exclusive-scan offsets and stable slot permutation of ids [N] or [N, k]."""
    _cuda(ids, "ids", torch.int32)
    N = ids.shape[0]
    k = 1 if ids.dim() == 1 else ids.shape[1]
    dev = ids.device
    if counts is None:
        counts = torch.empty(K, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(N * k, dtype=torch.int32, device=dev)
    _check("molora_dispatch", load_library().molora_dispatch(
        _p(ids), N, k, K, _p(counts), _p(offsets), _p(perm), _p(err_word), _stream(stream)))
    return counts, offsets, perm


def molora_route_vocab_dispatch(tok, starts, adapter=None, counts=None, offsets=None, perm=None, err_word=None,
                                stream=None):
    """molora_route_vocab then molora_dispatch (k = 1) as one kernel: (adapter, counts, offsets, perm)."""
    _cuda(tok, "tok", torch.int32, 1)
    _cuda(starts, "starts", torch.int32, 1)
    N, K = tok.numel(), starts.numel() - 1
    dev = tok.device
    if adapter is None:
        adapter = torch.empty(N, dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(K, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(N, dtype=torch.int32, device=dev)
    for name, t in (("adapter", adapter), ("counts", counts), ("offsets", offsets), ("perm", perm)):
        _cuda(t, name, torch.int32)
    _check("molora_route_vocab_dispatch", load_library().molora_route_vocab_dispatch(
        _p(tok), N, _p(starts), K, _p(adapter), _p(counts), _p(offsets), _p(perm), _p(err_word), _stream(stream)))
    return adapter, counts, offsets, perm


def molora_lora_apply(x, A, B, ids, y, scale, w=None, counts=None, offsets=None, perm=None, err_word=None,
                      path="auto", stream=None):
    """y[t] += scale * sum_j w[t,j] (x[t] A_{ids[t,j]}) B_{ids[t,j]}, in place on y (fp32, or bf16
    through molora_lora_apply_bf16y).  A and B are the hot-set slabs [K, d_in, r] and
    [K, r, d_out], or lists of K per-adapter tensors [d_in, r] and [r, d_out] (the indirect
    layout, molora_lora_apply_indirect)."""
    _cuda(x, "x", None, 2)
    N, d_in = x.shape
    indirect = isinstance(A, (list, tuple))
    if indirect:
        if not isinstance(B, (list, tuple)) or len(A) != len(B) or not A:
            raise ValueError("indirect layout: A and B must be lists of the same nonzero length")
        for i, (a_i, b_i) in enumerate(zip(A, B)):
            _cuda(a_i, f"A[{i}]", x.dtype, 2)
            _cuda(b_i, f"B[{i}]", x.dtype, 2)
        K, r, d_out = len(A), A[0].shape[1], B[0].shape[1]
        if any(a_i.shape != (d_in, r) for a_i in A) or any(b_i.shape != (r, d_out) for b_i in B):
            raise ValueError("indirect layout: every A[i] must be [d_in, r] and every B[i] [r, d_out]")
    else:
        _cuda(A, "A", x.dtype, 3)
        _cuda(B, "B", x.dtype, 3)
        K, _, r = A.shape
        d_out = B.shape[2]
        if A.shape[1] != d_in or B.shape[:2] != (K, r):
            raise ValueError("A must be [K, d_in, r] and B [K, r, d_out]")
    _cuda(ids, "ids", torch.int32)
    k = 1 if ids.dim() == 1 else ids.shape[1]
    _cuda(y, "y", None, 2)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
    if w is not None:
        _cuda(w, "w", torch.float32)
    for name, t in (("counts", counts), ("offsets", offsets), ("perm", perm)):
        if t is not None:
            _cuda(t, name, torch.int32)
    lib = load_library()
    if indirect:
        a_ptrs = (ctypes.c_void_p * K)(*[t.data_ptr() for t in A])
        b_ptrs = (ctypes.c_void_p * K)(*[t.data_ptr() for t in B])
        _check("molora_lora_apply", lib.molora_lora_apply_indirect(
            _p(x), _dtype_code(x), N, d_in, d_out, ctypes.cast(a_ptrs, ctypes.c_void_p),
            ctypes.cast(b_ptrs, ctypes.c_void_p), K, r, _p(ids), _p(w), k, _p(counts), _p(offsets), _p(perm),
            float(scale), _p(y), 1 if y.dtype == torch.bfloat16 else 0, _p(err_word), PATHS[path], _stream(stream)))
        return y
    fn = lib.molora_lora_apply_bf16y if y.dtype == torch.bfloat16 else lib.molora_lora_apply_ex
    _check("molora_lora_apply", fn(
        _p(x), _dtype_code(x), N, d_in, d_out, _p(A), _p(B), K, r, _p(ids), _p(w), k, _p(counts), _p(offsets),
        _p(perm), float(scale), _p(y), _p(err_word), PATHS[path], _stream(stream)))
    return y


def molora_route_vocab_lora_apply(tok, starts, x, A, B, y, scale, adapter=None, counts=None, offsets=None,
                                  perm=None, err_word=None, stream=None):
    """The whole vocabulary-routed step in one call: routing, dispatch and the apply (k = 1).
    Returns (adapter, counts, offsets, perm); y (fp32 or bf16) is updated in place."""
    _cuda(tok, "tok", torch.int32, 1)
    _cuda(starts, "starts", torch.int32, 1)
    N, K = tok.numel(), starts.numel() - 1
    _cuda(x, "x", None, 2)
    if x.shape[0] != N:
        raise ValueError("x must have one row per token")
    d_in = x.shape[1]
    _cuda(A, "A", x.dtype, 3)
    _cuda(B, "B", x.dtype, 3)
    if A.shape[0] != K or A.shape[1] != d_in or B.shape[:2] != (K, A.shape[2]):
        raise ValueError("A must be [K, d_in, r] and B [K, r, d_out], with K = len(starts) - 1")
    r, d_out = A.shape[2], B.shape[2]
    _cuda(y, "y", None, 2)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
    dev = tok.device
    if adapter is None:
        adapter = torch.empty(N, dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(K, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(N, dtype=torch.int32, device=dev)
    for name, t in (("adapter", adapter), ("counts", counts), ("offsets", offsets), ("perm", perm)):
        _cuda(t, name, torch.int32)
    _check("molora_route_vocab_lora_apply", load_library().molora_route_vocab_lora_apply(
        _p(tok), N, _p(starts), K, _p(x), _dtype_code(x), d_in, d_out, _p(A), _p(B), r, float(scale), _p(y),
        1 if y.dtype == torch.bfloat16 else 0, _p(adapter), _p(counts), _p(offsets), _p(perm), _p(err_word),
        _stream(stream)))
    return adapter, counts, offsets, perm


def molora_router_lora_apply(x, W1, W2, A, B, k, y, scale, b1=None, b2=None, logits=None, ids=None, w=None,
                             want_logits=True, err_word=None, stream=None):
    """The learned router and the top-k apply in one kernel (x read once): returns
    (logits fp32 [N,K] or None, ids int32 [N,k], w fp32 [N,k]); y (fp32 or bf16) is updated in
    place exactly as molora_router_topk followed by molora_lora_apply would update it."""
    _cuda(x, "x", None, 2)
    N, d_in = x.shape
    _cuda(W1, "W1", x.dtype, 2)
    _cuda(W2, "W2", x.dtype, 2)
    if W1.shape != (d_in, ROUTER_HIDDEN) or W2.shape[0] != ROUTER_HIDDEN:
        raise ValueError("W1 must be [d_in, 64] and W2 [64, K]")
    K = W2.shape[1]
    _cuda(A, "A", x.dtype, 3)
    _cuda(B, "B", x.dtype, 3)
    if A.shape[0] != K or A.shape[1] != d_in or B.shape[:2] != (K, A.shape[2]):
        raise ValueError("A must be [K, d_in, r] and B [K, r, d_out], with K = W2.shape[1]")
    r, d_out = A.shape[2], B.shape[2]
    _cuda(y, "y", None, 2)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
    for name, t in (("b1", b1), ("b2", b2)):
        if t is not None:
            _cuda(t, name, torch.float32)
    dev = x.device
    if logits is None and want_logits:
        logits = torch.empty(N, K, dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty(N, k, dtype=torch.int32, device=dev)
    if w is None:
        w = torch.empty(N, k, dtype=torch.float32, device=dev)
    _cuda(ids, "ids", torch.int32)
    _cuda(w, "w", torch.float32)
    _check("molora_router_lora_apply", load_library().molora_router_lora_apply(
        _p(x), _dtype_code(x), N, d_in, d_out, _p(W1), _p(b1), _p(W2), _p(b2), _p(A), _p(B), K, r, k, float(scale),
        _p(logits), _p(ids), _p(w), _p(y), 1 if y.dtype == torch.bfloat16 else 0, _p(err_word), _stream(stream)))
    return logits, ids, w


def molora_lora_apply_masked_pass(x, A, B, adapter_of, a, y, scale, err_word=None, path="auto", stream=None):
    """One per-sequence pass: y[t] += [adapter_of[t] == a] * scale * (x[t] A_a) B_a for every t."""
    _cuda(x, "x", None, 2)
    N, d_in = x.shape
    _cuda(A, "A", x.dtype, 3)
    _cuda(B, "B", x.dtype, 3)
    K, _, r = A.shape
    d_out = B.shape[2]
    _cuda(adapter_of, "adapter_of", torch.int32, 1)
    _cuda(y, "y", torch.float32, 2)
    _check("molora_lora_apply_masked_pass", load_library().molora_lora_apply_masked_pass(
        _p(x), _dtype_code(x), N, d_in, d_out, _p(A), _p(B), K, r, _p(adapter_of), int(a), float(scale), _p(y),
        _p(err_word), PATHS[path], _stream(stream)))
    return y


def molora_selftest_bounded_wait(err_word, limit_us=1000, stream=None):
    """Runs one CTA whose mbarrier wait can never complete; it must give up after limit_us and
    set DEV_WAIT_TIMEOUT in err_word (a device int32 tensor)."""
    _cuda(err_word, "err_word", torch.int32)
    _check("molora_selftest_bounded_wait", load_library().molora_selftest_bounded_wait(
        int(limit_us), _p(err_word), _stream(stream)))
    return err_word


def molora_select_path(dtype: torch.dtype, N: int, d_in: int, d_out: int, K: int, r: int, k: int) -> str:
    """The kernel family molora_lora_apply picks for this shape ("scalar" or "grouped")."""
    code = BF16 if dtype == torch.bfloat16 else F32
    return PATH_NAMES[load_library().molora_select_path(code, N, d_in, d_out, K, r, k)]
