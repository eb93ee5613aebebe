"""Python binding of the GB300 per-token adapter routing library (include/molora.h).

Argument marshalling only: every function here checks the shapes, dtypes and devices of
torch CUDA tensors against the sizes the call implies, passes their device pointers and
the tensors' current CUDA stream through ctypes to the C ABI, and raises on a non-OK
status.  A mis-sized tensor raises ValueError before anything is launched.  All
computation happens in the library's CUDA kernels; there is no CPU or PyTorch fallback.  If
the compiled library is missing the first call raises: build it with
``token_adapter_routing_gb300.build.build()``.

Method: "MoLoRA: Composable Specialization via Per-Token Adapter Routing" -- vocabulary
routing and the learned top-k router (Table 1), dispatch by histogram / pointer arrays /
grouping (Table 1, Figure 2), and the batched LoRA apply over a GPU-resident hot set
(Figure 2, Figure 4, Table 10 shapes).
"""

from __future__ import annotations

import ctypes
import functools
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "molora_route_vocab", "molora_router_topk", "molora_dispatch", "molora_route_vocab_dispatch",
    "molora_lora_apply", "molora_lora_apply_masked_pass", "molora_route_vocab_lora_apply",
    "molora_router_lora_apply", "molora_select_path", "molora_workspace_bytes", "molora_lora_apply_static_ws",
    "molora_selftest_bounded_wait", "library_path", "load_library",
    "MoloraError", "PATHS", "DEV_TOKEN_OUTSIDE_RANGES", "DEV_BAD_RANGES", "DEV_BAD_ADAPTER_ID",
    "DEV_BAD_PERMUTATION", "DEV_WAIT_TIMEOUT", "MAX_ADAPTERS", "ROUTER_HIDDEN",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_SCRATCH_TOO_SMALL = 0, 1, 2, 3, 4
STATIC_SCRATCH_BYTES = 16 << 20
F32, BF16 = 0, 1
PATHS = {"auto": 0, "scalar": 1, "grouped": 2, "dense": 3, "stacked": 4}
PATH_NAMES = {v: k for k, v in PATHS.items()}
DEV_TOKEN_OUTSIDE_RANGES = 0x1
DEV_BAD_RANGES = 0x2
DEV_BAD_ADAPTER_ID = 0x4
DEV_BAD_PERMUTATION = 0x8
DEV_WAIT_TIMEOUT = 0x10
INPUTS_READY = 0x1  # molora_route_vocab_dispatch_ex flag
MAX_ADAPTERS = 64
ROUTER_HIDDEN = 64

EXPORTED = ("molora_route_vocab", "molora_route_vocab_ex", "molora_router_topk", "molora_dispatch", "molora_route_vocab_dispatch",
            "molora_route_vocab_dispatch_ex", "molora_route_vocab_lora_apply_ex",
            "molora_lora_apply", "molora_router_lora_apply", "molora_route_vocab_lora_apply",
            "molora_lora_apply_ex", "molora_lora_apply_bf16y", "molora_lora_apply_indirect",
            "molora_lora_apply_masked_pass", "molora_select_path", "molora_status_string", "molora_version",
            "molora_selftest_bounded_wait", "molora_lora_apply_static_ws")


class MoloraError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(path=None):
    """Loads the compiled library (raises if it has not been built).  ``path``: another build of
    it (the tuning build of build.build(tuning=True)); only the first load in a process counts."""
    global _lib
    if _lib is not None:
        if path is not None and os.path.realpath(path) != os.path.realpath(_lib._name):
            raise RuntimeError(f"a different CUDA library ({_lib._name}) is already loaded")
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: build it with token_adapter_routing_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I64, I32, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_int
    lib.molora_route_vocab.argtypes = [P, I64, P, I32, P, P, P]
    lib.molora_route_vocab_ex.argtypes = [P, I64, P, I32, P, P, ctypes.c_uint32, P]
    lib.molora_router_topk.argtypes = [P, S, I64, I32, P, P, P, P, I32, I32, P, P, P, P]
    lib.molora_dispatch.argtypes = [P, I64, I32, I32, P, P, P, P, P]
    lib.molora_route_vocab_dispatch.argtypes = [P, I64, P, I32, P, P, P, P, P, P]
    lib.molora_route_vocab_dispatch_ex.argtypes = [P, I64, P, I32, P, P, P, P, P, ctypes.c_uint32, P]
    lib.molora_lora_apply.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, P, P, P]
    lib.molora_lora_apply_ex.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, P, P, S,
                                         P]
    lib.molora_lora_apply_bf16y.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, S, P]
    lib.molora_lora_apply_indirect.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, I32,
                                               P, S, P]
    lib.molora_router_lora_apply.argtypes = [P, S, I64, I32, I32, P, P, P, P, P, P, I32, I32, I32, F, P, P, P, P,
                                             I32, P, P, P, P]
    lib.molora_route_vocab_lora_apply.argtypes = [P, I64, P, I32, P, S, I32, I32, P, P, I32, F, P, I32, P, P, P, P,
                                                  P, P]
    lib.molora_route_vocab_lora_apply_ex.argtypes = [P, I64, P, I32, P, S, I32, I32, P, P, I32, F, P, I32, P, P, P,
                                                     P, P, ctypes.c_uint32, P]
    lib.molora_lora_apply_masked_pass.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, I32, F, P, P, S, P]
    lib.molora_lora_apply_static_ws.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, F, P, P, P]
    lib.molora_select_path.argtypes = [S, I64, I32, I32, I32, I32, I32]
    lib.molora_status_string.argtypes = [S]
    lib.molora_status_string.restype = ctypes.c_char_p
    lib.molora_version.argtypes = []
    lib.molora_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P, P]
    for name in ("molora_route_vocab", "molora_route_vocab_ex", "molora_router_topk", "molora_dispatch", "molora_route_vocab_dispatch",
                 "molora_route_vocab_dispatch_ex", "molora_route_vocab_lora_apply_ex", "molora_lora_apply", "molora_lora_apply_ex", "molora_lora_apply_bf16y", "molora_lora_apply_indirect",
                 "molora_router_lora_apply", "molora_route_vocab_lora_apply", "molora_lora_apply_masked_pass",
                 "molora_select_path", "molora_version", "molora_selftest_bounded_wait",
                 "molora_lora_apply_static_ws"):
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


def _stream(stream, device) -> ctypes.c_void_p:
    """The given stream, else the current stream of `device` (the tensors' device, which may
    differ from the current device)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t: torch.Tensor, name: str, dtype=None, ndim=None, device=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device} (all tensors of a call share one device)")
    return t


def _sized(t: Optional[torch.Tensor], name: str, numel: int, dtype, device, shape=None):
    """A caller-supplied output or index tensor: CUDA, contiguous, the right dtype, device and
    element count (and exact shape when given)."""
    if t is None:
        return None
    _cuda(t, name, dtype, device=device)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return t


def _need(t: Optional[torch.Tensor], name: str, numel: int, rows: Optional[int] = None):
    """Shape-only check of an optional tensor (before any device check, so that a mis-sized
    argument is reported as such): `numel` elements and, when given, `rows` rows."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()} (shape {tuple(t.shape)})")
    if rows is not None and (t.dim() == 0 or t.shape[0] != rows):
        raise ValueError(f"{name} must have {rows} rows, got shape {tuple(t.shape)}")


def _err_word(err_word: Optional[torch.Tensor], device):
    if err_word is None:
        return None
    _cuda(err_word, "err_word", torch.int32, device=device)
    if err_word.numel() < 1:
        raise ValueError("err_word must hold at least one int32")
    return err_word


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def _slots(ids: torch.Tensor, N: int, name: str = "ids"):
    """k for ids of shape [N] (k = 1) or [N, k]; raises unless ids has N rows."""
    if ids.dim() not in (1, 2) or ids.shape[0] != N:
        raise ValueError(f"{name} must be [N] or [N, k] with N = {N}, got {tuple(ids.shape)}")
    return 1 if ids.dim() == 1 else ids.shape[1]


def _workspace(ws: Optional[torch.Tensor], device, call) -> int:
    """Runs `call(ws_ptr, ws_bytes_ptr)` under the library's workspace convention and returns
    its status: with no caller buffer it first queries the size and, if one is needed,
    allocates it on `device` (torch's caching allocator; inside a CUDA graph capture the
    graph's pool)."""
    size = ctypes.c_size_t(0)
    if ws is None:
        status = call(None, ctypes.byref(size))
        if status != OK:
            return status
        if size.value == 0:
            return call(None, None)
        ws = torch.empty(size.value, dtype=torch.uint8, device=device)
    else:
        _cuda(ws, "ws", torch.uint8, device=device)
    size.value = ws.numel()
    return call(_p(ws), ctypes.byref(size))


def _on_tensor_device(fn):
    """Runs a launching call with the device of its first CUDA tensor argument current, so that
    the library launches on the device that holds the tensors (and their stream), whichever
    device the caller has current.  The call itself checks that all tensors share that device."""
    @functools.wraps(fn)
    def call(*args, **kwargs):
        for a in (*args, *kwargs.values()):
            if isinstance(a, (list, tuple)) and a and isinstance(a[0], torch.Tensor):
                a = a[0]
            if isinstance(a, torch.Tensor) and a.is_cuda:
                with torch.cuda.device(a.device):
                    return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return call


def molora_workspace_bytes(N, d_in, d_out, K, r, k, dtype=torch.bfloat16, path="auto", router=False) -> int:
    """Bytes of workspace molora_lora_apply (or, with router=True, molora_router_lora_apply)
    needs for these sizes (a query: nothing is launched).  Allocate them once, e.g. before
    capturing a CUDA graph, and pass the uint8 buffer as ``ws``."""
    size = ctypes.c_size_t(0)
    lib = load_library()
    code = BF16 if dtype == torch.bfloat16 else F32
    if router:
        _check("molora_router_lora_apply", lib.molora_router_lora_apply(
            None, code, N, d_in, d_out, None, None, None, None, None, None, K, r, k, 1.0, None, None, None, None, 0,
            None, ctypes.byref(size), None, None))
    else:
        _check("molora_lora_apply", lib.molora_lora_apply_ex(
            None, code, N, d_in, d_out, None, None, K, r, None, None, k, None, None, None, 1.0, None, None,
            ctypes.byref(size), None, PATHS[path], None))
    return size.value


@_on_tensor_device
def molora_route_vocab(tok, starts, adapter=None, err_word=None, stream=None):
    """adapter[t] = a with starts[a] <= tok[t] < starts[a+1], else -1 (int32 [N])."""
    return _route_vocab(tok, starts, adapter, err_word, stream, None)


@_on_tensor_device
def molora_route_vocab_ex(tok, starts, flags, adapter=None, err_word=None, stream=None):
    """molora_route_vocab with flags (INPUTS_READY: tok and starts are not written by the kernel
    enqueued just before, so each token is routed before waiting on it)."""
    return _route_vocab(tok, starts, adapter, err_word, stream, int(flags))


def _route_vocab(tok, starts, adapter, err_word, stream, flags):
    _need(adapter, "adapter", tok.numel())
    _cuda(tok, "tok", torch.int32, 1)
    dev = tok.device
    _cuda(starts, "starts", torch.int32, 1, device=dev)
    N, K = tok.numel(), starts.numel() - 1
    if adapter is None:
        adapter = torch.empty(N, dtype=torch.int32, device=dev)
    _sized(adapter, "adapter", N, torch.int32, dev)
    args = (_p(tok), N, _p(starts), K, _p(adapter), _p(_err_word(err_word, dev)))
    if flags is None:
        _check("molora_route_vocab", load_library().molora_route_vocab(*args, _stream(stream, dev)))
    else:
        _check("molora_route_vocab_ex", load_library().molora_route_vocab_ex(*args, flags, _stream(stream, dev)))
    return adapter


@_on_tensor_device
def molora_router_topk(x, W1, W2, k, b1=None, b2=None, logits=None, ids=None, w=None, want_logits=True,
                       stream=None):
    """Learned router: returns (logits fp32 [N,K] or None, ids int32 [N,k], w fp32 [N,k])."""
    if x.dim() != 2 or W1.dim() != 2 or W2.dim() != 2:
        raise ValueError("x must be [N, d_in], W1 [d_in, 64] and W2 [64, K]")
    N, d_in = x.shape
    if tuple(W1.shape) != (d_in, ROUTER_HIDDEN) or W2.shape[0] != ROUTER_HIDDEN:
        raise ValueError("W1 must be [d_in, 64] and W2 [64, K]")
    K = W2.shape[1]
    _need(logits, "logits", N * K, rows=N)
    _need(ids, "ids", N * k, rows=N)
    _need(w, "w", N * k, rows=N)
    _need(b1, "b1", ROUTER_HIDDEN)
    _need(b2, "b2", K)
    _cuda(x, "x", None, 2)
    dev = x.device
    _cuda(W1, "W1", x.dtype, 2, device=dev)
    _cuda(W2, "W2", x.dtype, 2, device=dev)
    _sized(b1, "b1", ROUTER_HIDDEN, torch.float32, dev)
    _sized(b2, "b2", K, torch.float32, dev)
    if logits is None and want_logits:
        logits = torch.empty(N, K, dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty(N, k, dtype=torch.int32, device=dev)
    if w is None:
        w = torch.empty(N, k, dtype=torch.float32, device=dev)
    _sized(logits, "logits", N * K, torch.float32, dev)
    _sized(ids, "ids", N * k, torch.int32, dev)
    _sized(w, "w", N * k, torch.float32, dev)
    _check("molora_router_topk", load_library().molora_router_topk(
        _p(x), _dtype_code(x), N, d_in, _p(W1), _p(b1), _p(W2), _p(b2), K, k, _p(logits), _p(ids), _p(w),
        _stream(stream, dev)))
    return logits, ids, w


@_on_tensor_device
def molora_dispatch(ids, K, counts=None, offsets=None, perm=None, err_word=None, stream=None):
    """Histogram, exclusive-scan offsets and stable slot permutation of ids [N] or [N, k]."""
    N = ids.shape[0]
    k = _slots(ids, N)
    _need(counts, "counts", K)
    _need(offsets, "offsets", K + 1)
    _need(perm, "perm", N * k)
    _cuda(ids, "ids", torch.int32)
    dev = ids.device
    if counts is None:
        counts = torch.empty(K, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(N * k, dtype=torch.int32, device=dev)
    _sized(counts, "counts", K, torch.int32, dev)
    _sized(offsets, "offsets", K + 1, torch.int32, dev)
    _sized(perm, "perm", N * k, torch.int32, dev)
    _check("molora_dispatch", load_library().molora_dispatch(
        _p(ids), N, k, K, _p(counts), _p(offsets), _p(perm), _p(_err_word(err_word, dev)), _stream(stream, dev)))
    return counts, offsets, perm


@_on_tensor_device
def molora_route_vocab_dispatch(tok, starts, adapter=None, counts=None, offsets=None, perm=None, err_word=None,
                                stream=None):
    """molora_route_vocab then molora_dispatch (k = 1) as one kernel: (adapter, counts, offsets, perm)."""
    return _route_vocab_dispatch(tok, starts, adapter, counts, offsets, perm, err_word, stream, None)


@_on_tensor_device
def molora_route_vocab_dispatch_ex(tok, starts, flags, adapter=None, counts=None, offsets=None, perm=None,
                                   err_word=None, stream=None):
    """molora_route_vocab_dispatch with flags (INPUTS_READY: tok and starts are not written by the
    kernel enqueued just before, so the kernel reads them before waiting on it)."""
    return _route_vocab_dispatch(tok, starts, adapter, counts, offsets, perm, err_word, stream, int(flags))


def _route_vocab_dispatch(tok, starts, adapter, counts, offsets, perm, err_word, stream, flags):
    N, K = tok.numel(), starts.numel() - 1
    for name, t, n in (("adapter", adapter, N), ("counts", counts, K), ("offsets", offsets, K + 1), ("perm", perm, N)):
        _need(t, name, n)
    _cuda(tok, "tok", torch.int32, 1)
    dev = tok.device
    _cuda(starts, "starts", torch.int32, 1, device=dev)
    if adapter is None:
        adapter = torch.empty(N, dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(K, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(N, dtype=torch.int32, device=dev)
    _sized(adapter, "adapter", N, torch.int32, dev)
    _sized(counts, "counts", K, torch.int32, dev)
    _sized(offsets, "offsets", K + 1, torch.int32, dev)
    _sized(perm, "perm", N, torch.int32, dev)
    args = (_p(tok), N, _p(starts), K, _p(adapter), _p(counts), _p(offsets), _p(perm), _p(_err_word(err_word, dev)))
    if flags is None:
        _check("molora_route_vocab_dispatch", load_library().molora_route_vocab_dispatch(*args, _stream(stream, dev)))
    else:
        _check("molora_route_vocab_dispatch_ex",
               load_library().molora_route_vocab_dispatch_ex(*args, flags, _stream(stream, dev)))
    return adapter, counts, offsets, perm


@_on_tensor_device
def molora_lora_apply(x, A, B, ids, y, scale, w=None, counts=None, offsets=None, perm=None, err_word=None,
                      path="auto", ws=None, stream=None):
    """y[t] += scale * sum_j w[t,j] (x[t] A_{ids[t,j]}) B_{ids[t,j]}, in place on y (fp32, or bf16
    through molora_lora_apply_bf16y).  A and B are the hot-set slabs [K, d_in, r] and
    [K, r, d_out], or lists of K per-adapter tensors [d_in, r] and [r, d_out] (the indirect
    layout, molora_lora_apply_indirect).  ``ws``: an optional uint8 workspace of
    molora_workspace_bytes bytes; without one, a path that needs it gets a fresh buffer."""
    # shapes first: a mis-sized argument raises before anything else is looked at
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a 2-D tensor [N, d_in]")
    N, d_in = x.shape
    indirect = isinstance(A, (list, tuple))
    if indirect:
        if not isinstance(B, (list, tuple)) or len(A) != len(B) or not A:
            raise ValueError("indirect layout: A and B must be lists of the same nonzero length")
        K, r, d_out = len(A), A[0].shape[1], B[0].shape[1]
        if any(tuple(a_i.shape) != (d_in, r) for a_i in A) or any(tuple(b_i.shape) != (r, d_out) for b_i in B):
            raise ValueError("indirect layout: every A[i] must be [d_in, r] and every B[i] [r, d_out]")
    else:
        if A.dim() != 3 or B.dim() != 3:
            raise ValueError("A must be [K, d_in, r] and B [K, r, d_out]")
        K, _, r = A.shape
        d_out = B.shape[2]
        if A.shape[1] != d_in or tuple(B.shape[:2]) != (K, r):
            raise ValueError("A must be [K, d_in, r] and B [K, r, d_out]")
    k = _slots(ids, N)
    if y.dim() != 2 or tuple(y.shape) != (N, d_out):
        raise ValueError(f"y must be [N, d_out] = {(N, d_out)}, got {tuple(y.shape)}")
    _need(w, "w", N * k, rows=N)
    _need(counts, "counts", K)
    _need(offsets, "offsets", K + 1)
    _need(perm, "perm", N * k)
    # then devices, dtypes and layout
    _cuda(x, "x", None, 2)
    dev = x.device
    if indirect:
        for i, (a_i, b_i) in enumerate(zip(A, B)):
            _cuda(a_i, f"A[{i}]", x.dtype, 2, device=dev)
            _cuda(b_i, f"B[{i}]", x.dtype, 2, device=dev)
    else:
        _cuda(A, "A", x.dtype, 3, device=dev)
        _cuda(B, "B", x.dtype, 3, device=dev)
    _cuda(ids, "ids", torch.int32, device=dev)
    _cuda(y, "y", None, 2, device=dev)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
    _sized(w, "w", N * k, torch.float32, dev)
    _sized(counts, "counts", K, torch.int32, dev)
    _sized(offsets, "offsets", K + 1, torch.int32, dev)
    _sized(perm, "perm", N * k, torch.int32, dev)
    e = _p(_err_word(err_word, dev))
    s = _stream(stream, dev)
    lib = load_library()
    if indirect:
        a_ptrs = (ctypes.c_void_p * K)(*[t.data_ptr() for t in A])
        b_ptrs = (ctypes.c_void_p * K)(*[t.data_ptr() for t in B])
        _check("molora_lora_apply", lib.molora_lora_apply_indirect(
            _p(x), _dtype_code(x), N, d_in, d_out, ctypes.cast(a_ptrs, ctypes.c_void_p),
            ctypes.cast(b_ptrs, ctypes.c_void_p), K, r, _p(ids), _p(w), k, _p(counts), _p(offsets), _p(perm),
            float(scale), _p(y), 1 if y.dtype == torch.bfloat16 else 0, e, PATHS[path], s))
        return y
    if y.dtype == torch.bfloat16:
        _check("molora_lora_apply", lib.molora_lora_apply_bf16y(
            _p(x), _dtype_code(x), N, d_in, d_out, _p(A), _p(B), K, r, _p(ids), _p(w), k, _p(counts), _p(offsets),
            _p(perm), float(scale), _p(y), e, PATHS[path], s))
        return y

    def call(ws_ptr, ws_bytes):
        return lib.molora_lora_apply_ex(
            _p(x), _dtype_code(x), N, d_in, d_out, _p(A), _p(B), K, r, _p(ids), _p(w), k, _p(counts), _p(offsets),
            _p(perm), float(scale), _p(y), ws_ptr, ws_bytes, e, PATHS[path], s)
    if path in ("auto", "stacked") or ws is not None:
        _check("molora_lora_apply", _workspace(ws, dev, call))
    else:
        _check("molora_lora_apply", call(None, None))
    return y


@_on_tensor_device
def molora_route_vocab_lora_apply(tok, starts, x, A, B, y, scale, adapter=None, counts=None, offsets=None,
                                  perm=None, err_word=None, stream=None):
    """The whole vocabulary-routed step in one call: routing, dispatch and the apply (k = 1).
    Returns (adapter, counts, offsets, perm); y (fp32 or bf16) is updated in place."""
    return _route_vocab_lora_apply(tok, starts, x, A, B, y, scale, adapter, counts, offsets, perm, err_word, stream,
                                   None)


@_on_tensor_device
def molora_route_vocab_lora_apply_ex(tok, starts, x, A, B, y, scale, flags, adapter=None, counts=None, offsets=None,
                                     perm=None, err_word=None, stream=None):
    """molora_route_vocab_lora_apply with flags (INPUTS_READY: as for molora_route_vocab_dispatch_ex)."""
    return _route_vocab_lora_apply(tok, starts, x, A, B, y, scale, adapter, counts, offsets, perm, err_word, stream,
                                   int(flags))


def _route_vocab_lora_apply(tok, starts, x, A, B, y, scale, adapter, counts, offsets, perm, err_word, stream, flags):
    N, K = tok.numel(), starts.numel() - 1
    if x.dim() != 2 or x.shape[0] != N:
        raise ValueError("x must be [N, d_in] with one row per token")
    d_in = x.shape[1]
    if A.dim() != 3 or B.dim() != 3 or A.shape[0] != K or A.shape[1] != d_in or tuple(B.shape[:2]) != (K, A.shape[2]):
        raise ValueError("A must be [K, d_in, r] and B [K, r, d_out], with K = len(starts) - 1")
    r, d_out = A.shape[2], B.shape[2]
    if y.dim() != 2 or tuple(y.shape) != (N, d_out):
        raise ValueError(f"y must be [N, d_out] = {(N, d_out)}, got {tuple(y.shape)}")
    for name, t, n in (("adapter", adapter, N), ("counts", counts, K), ("offsets", offsets, K + 1), ("perm", perm, N)):
        _need(t, name, n)
    _cuda(tok, "tok", torch.int32, 1)
    dev = tok.device
    _cuda(starts, "starts", torch.int32, 1, device=dev)
    _cuda(x, "x", None, 2, device=dev)
    _cuda(A, "A", x.dtype, 3, device=dev)
    _cuda(B, "B", x.dtype, 3, device=dev)
    _cuda(y, "y", None, 2, device=dev)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
    if adapter is None:
        adapter = torch.empty(N, dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(K, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(N, dtype=torch.int32, device=dev)
    _sized(adapter, "adapter", N, torch.int32, dev)
    _sized(counts, "counts", K, torch.int32, dev)
    _sized(offsets, "offsets", K + 1, torch.int32, dev)
    _sized(perm, "perm", N, torch.int32, dev)
    args = (_p(tok), N, _p(starts), K, _p(x), _dtype_code(x), d_in, d_out, _p(A), _p(B), r, float(scale), _p(y),
            1 if y.dtype == torch.bfloat16 else 0, _p(adapter), _p(counts), _p(offsets), _p(perm),
            _p(_err_word(err_word, dev)))
    if flags is None:
        _check("molora_route_vocab_lora_apply",
               load_library().molora_route_vocab_lora_apply(*args, _stream(stream, dev)))
    else:
        _check("molora_route_vocab_lora_apply_ex",
               load_library().molora_route_vocab_lora_apply_ex(*args, flags, _stream(stream, dev)))
    return adapter, counts, offsets, perm


@_on_tensor_device
def molora_router_lora_apply(x, W1, W2, A, B, k, y, scale, b1=None, b2=None, logits=None, ids=None, w=None,
                             want_logits=True, err_word=None, ws=None, use_ws=True, stream=None):
    """The learned router and the top-k apply with one pass over x: returns
    (logits fp32 [N,K] or None, ids int32 [N,k], w fp32 [N,k]); y (fp32 or bf16) is updated in
    place.  ``use_ws=False`` restricts it to the one-kernel family (no workspace); otherwise a
    workspace is used where the library prefers the stacked pair (``ws`` if given, else a
    fresh buffer)."""
    if x.dim() != 2 or W1.dim() != 2 or W2.dim() != 2:
        raise ValueError("x must be [N, d_in], W1 [d_in, 64] and W2 [64, K]")
    N, d_in = x.shape
    if tuple(W1.shape) != (d_in, ROUTER_HIDDEN) or W2.shape[0] != ROUTER_HIDDEN:
        raise ValueError("W1 must be [d_in, 64] and W2 [64, K]")
    K = W2.shape[1]
    if A.dim() != 3 or B.dim() != 3 or A.shape[0] != K or A.shape[1] != d_in or tuple(B.shape[:2]) != (K, A.shape[2]):
        raise ValueError("A must be [K, d_in, r] and B [K, r, d_out], with K = W2.shape[1]")
    r, d_out = A.shape[2], B.shape[2]
    if y.dim() != 2 or tuple(y.shape) != (N, d_out):
        raise ValueError(f"y must be [N, d_out] = {(N, d_out)}, got {tuple(y.shape)}")
    _need(logits, "logits", N * K, rows=N)
    _need(ids, "ids", N * k, rows=N)
    _need(w, "w", N * k, rows=N)
    _need(b1, "b1", ROUTER_HIDDEN)
    _need(b2, "b2", K)
    _cuda(x, "x", None, 2)
    dev = x.device
    _cuda(W1, "W1", x.dtype, 2, device=dev)
    _cuda(W2, "W2", x.dtype, 2, device=dev)
    _cuda(A, "A", x.dtype, 3, device=dev)
    _cuda(B, "B", x.dtype, 3, device=dev)
    _cuda(y, "y", None, 2, device=dev)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
    _sized(b1, "b1", ROUTER_HIDDEN, torch.float32, dev)
    _sized(b2, "b2", K, torch.float32, dev)
    if logits is None and want_logits:
        logits = torch.empty(N, K, dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty(N, k, dtype=torch.int32, device=dev)
    if w is None:
        w = torch.empty(N, k, dtype=torch.float32, device=dev)
    _sized(logits, "logits", N * K, torch.float32, dev)
    _sized(ids, "ids", N * k, torch.int32, dev)
    _sized(w, "w", N * k, torch.float32, dev)
    e = _p(_err_word(err_word, dev))
    s = _stream(stream, dev)
    lib = load_library()

    def call(ws_ptr, ws_bytes):
        return lib.molora_router_lora_apply(
            _p(x), _dtype_code(x), N, d_in, d_out, _p(W1), _p(b1), _p(W2), _p(b2), _p(A), _p(B), K, r, k,
            float(scale), _p(logits), _p(ids), _p(w), _p(y), 1 if y.dtype == torch.bfloat16 else 0, ws_ptr,
            ws_bytes, e, s)
    if use_ws:
        _check("molora_router_lora_apply", _workspace(ws, dev, call))
    else:
        _check("molora_router_lora_apply", call(None, None))
    return logits, ids, w


@_on_tensor_device
def molora_lora_apply_static_ws(x, A, B, ids, y, scale, w=None, err_word=None, stream=None):
    """The stacked apply for callers that cannot allocate device memory: the workspace is a
    fixed scratch buffer inside the library (STATIC_SCRATCH_BYTES; N*K*r up to 4M), shared by
    every call on the device -- calls that may overlap on the GPU must be serialised.  The
    first call on a device looks the buffer up; make it before capturing a CUDA graph.
    Same results as molora_lora_apply(..., path="stacked"); y (fp32) is updated in place."""
    if x.dim() != 2 or A.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [N, d_in], A [K, d_in, r] and B [K, r, d_out]")
    N, d_in = x.shape
    K, _, r = A.shape
    d_out = B.shape[2]
    if A.shape[1] != d_in or tuple(B.shape[:2]) != (K, r):
        raise ValueError("A must be [K, d_in, r] and B [K, r, d_out]")
    k = _slots(ids, N)
    if y.dim() != 2 or tuple(y.shape) != (N, d_out):
        raise ValueError(f"y must be [N, d_out] = {(N, d_out)}, got {tuple(y.shape)}")
    _need(w, "w", N * k, rows=N)
    _cuda(x, "x", None, 2)
    dev = x.device
    _cuda(A, "A", x.dtype, 3, device=dev)
    _cuda(B, "B", x.dtype, 3, device=dev)
    _cuda(ids, "ids", torch.int32, device=dev)
    _cuda(y, "y", torch.float32, 2, device=dev)
    _sized(w, "w", N * k, torch.float32, dev)
    _check("molora_lora_apply_static_ws", load_library().molora_lora_apply_static_ws(
        _p(x), _dtype_code(x), N, d_in, d_out, _p(A), _p(B), K, r, _p(ids), _p(w), k, float(scale), _p(y),
        _p(_err_word(err_word, dev)), _stream(stream, dev)))
    return y


@_on_tensor_device
def molora_lora_apply_masked_pass(x, A, B, adapter_of, a, y, scale, err_word=None, path="auto", stream=None):
    """One per-sequence pass: y[t] += [adapter_of[t] == a] * scale * (x[t] A_a) B_a for every t."""
    if x.dim() != 2 or A.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [N, d_in], A [K, d_in, r] and B [K, r, d_out]")
    N, d_in = x.shape
    K, _, r = A.shape
    d_out = B.shape[2]
    if A.shape[1] != d_in or tuple(B.shape[:2]) != (K, r):
        raise ValueError("A must be [K, d_in, r] and B [K, r, d_out]")
    if adapter_of.dim() != 1 or adapter_of.numel() != N:
        raise ValueError(f"adapter_of must be [N] with N = {N}, got {tuple(adapter_of.shape)}")
    if y.dim() != 2 or tuple(y.shape) != (N, d_out):
        raise ValueError(f"y must be [N, d_out] = {(N, d_out)}, got {tuple(y.shape)}")
    _cuda(x, "x", None, 2)
    dev = x.device
    _cuda(A, "A", x.dtype, 3, device=dev)
    _cuda(B, "B", x.dtype, 3, device=dev)
    _cuda(adapter_of, "adapter_of", torch.int32, 1, device=dev)
    _cuda(y, "y", torch.float32, 2, device=dev)
    _check("molora_lora_apply_masked_pass", load_library().molora_lora_apply_masked_pass(
        _p(x), _dtype_code(x), N, d_in, d_out, _p(A), _p(B), K, r, _p(adapter_of), int(a), float(scale), _p(y),
        _p(_err_word(err_word, dev)), PATHS[path], _stream(stream, dev)))
    return y


@_on_tensor_device
def molora_selftest_bounded_wait(err_word, limit_us=1000, stream=None):
    """Runs one CTA whose mbarrier wait can never complete; it must give up after limit_us and
    set DEV_WAIT_TIMEOUT in err_word (a device int32 tensor)."""
    _cuda(err_word, "err_word", torch.int32)
    dev = err_word.device
    _err_word(err_word, dev)
    _check("molora_selftest_bounded_wait", load_library().molora_selftest_bounded_wait(
        int(limit_us), _p(err_word), _stream(stream, dev)))
    return err_word


def molora_select_path(dtype: torch.dtype, N: int, d_in: int, d_out: int, K: int, r: int, k: int) -> str:
    """The kernel family molora_lora_apply picks for this shape when it may use a workspace
    ("scalar", "grouped", "dense" or "stacked")."""
    code = BF16 if dtype == torch.bfloat16 else F32
    return PATH_NAMES[load_library().molora_select_path(code, N, d_in, d_out, K, r, k)]
