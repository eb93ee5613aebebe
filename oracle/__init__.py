"""CPU oracle for per-token adapter routing and the batched LoRA apply.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or executes anything here, and this package
never imports the product.

The arithmetic lives in ``molora_oracle.c``: plain loops, double accumulation, one final
rounding, written from "MoLoRA: Composable Specialization via Per-Token Adapter Routing"
(Table 1: the routing decisions and the shared histogram / pointer-array / grouped-GEMM
dispatch; Figure 2: the top-k weighted sum and grouping by adapter; Table 10: weight shapes;
Tables 3 and 7: K masked per-sequence passes).  This module only marshals arguments.

Inputs are torch CPU tensors (contiguous).  bf16 tensors are handed over as raw bits and
decoded exactly in C.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "molora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmolora_oracle.so")

F32 = 0
BF16 = 1
ROUTER_HIDDEN = 64

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no CUDA).  Returns the library path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    lib.oracle_route_vocab.argtypes = [P, I64, P, I32, P]
    lib.oracle_route_vocab.restype = I64
    lib.oracle_router_topk.argtypes = [P, ctypes.c_int, I64, I32, P, P, P, P, I32, I32, P, P, P]
    lib.oracle_router_topk.restype = None
    lib.oracle_dispatch.argtypes = [P, I64, I32, I32, P, P, P]
    lib.oracle_dispatch.restype = I64
    lib.oracle_lora_apply.argtypes = [P, ctypes.c_int, I64, I32, I32, P, P, I32, I32, P, P, I32, F, P, P]
    lib.oracle_lora_apply.restype = None
    lib.oracle_masked_pass.argtypes = [P, ctypes.c_int, I64, I32, I32, P, P, I32, I32, P, I32, F, P, P]
    lib.oracle_masked_pass.restype = None
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous(), "oracle takes contiguous CPU tensors"
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"oracle supports float32 and bfloat16 inputs, got {t.dtype}")


def route_vocab(tok: torch.Tensor, starts: torch.Tensor):
    """adapter[t] = a with starts[a] <= tok[t] < starts[a+1], else -1.  Returns (adapter, n_outside)."""
    tok = tok.to(torch.int32).contiguous()
    starts = starts.to(torch.int32).contiguous()
    K = starts.numel() - 1
    out = torch.empty(tok.numel(), dtype=torch.int32)
    n_out = _load().oracle_route_vocab(_ptr(tok), tok.numel(), _ptr(starts), K, _ptr(out))
    return out, int(n_out)


def router_topk(x, W1, W2, k, b1=None, b2=None):
    """Learned router: returns (logits fp32 [N,K], ids int32 [N,k], w fp32 [N,k])."""
    x = x.contiguous()
    N, d_in = x.shape
    K = W2.shape[1]
    assert W1.shape == (d_in, ROUTER_HIDDEN) and W2.shape[0] == ROUTER_HIDDEN
    assert W1.dtype == x.dtype and W2.dtype == x.dtype
    b1 = None if b1 is None else b1.to(torch.float32).contiguous()
    b2 = None if b2 is None else b2.to(torch.float32).contiguous()
    logits = torch.empty(N, K, dtype=torch.float32)
    ids = torch.empty(N, k, dtype=torch.int32)
    w = torch.empty(N, k, dtype=torch.float32)
    _load().oracle_router_topk(_ptr(x), _dtype_code(x), N, d_in, _ptr(W1.contiguous()), _ptr(b1),
                               _ptr(W2.contiguous()), _ptr(b2), K, k, _ptr(logits), _ptr(ids), _ptr(w))
    return logits, ids, w


def dispatch(ids: torch.Tensor, K: int):
    """Histogram, exclusive-scan offsets and stable permutation of the slots.

    ids is [N, k] (or [N] for k=1).  Returns (counts [K], offsets [K+1], perm [N*k], n_invalid).
    """
    ids2 = ids.to(torch.int32)
    ids2 = (ids2.reshape(-1, 1) if ids2.dim() == 1 else ids2).contiguous()
    N, k = ids2.shape
    counts = torch.empty(K, dtype=torch.int32)
    offsets = torch.empty(K + 1, dtype=torch.int32)
    perm = torch.empty(N * k, dtype=torch.int32)
    n_inv = _load().oracle_dispatch(_ptr(ids2), N, k, K, _ptr(counts), _ptr(offsets), _ptr(perm))
    return counts, offsets, perm, int(n_inv)


def lora_apply(x, A, B, ids, y0, scale, w=None):
    """y = y0 + scale * sum_j w[t,j] (x[t] A_{ids[t,j]}) B_{ids[t,j]}, token-major, double.

    x [N, d_in], A [K, d_in, r], B [K, r, d_out] (same dtype), ids [N, k] int, y0 [N, d_out] fp32,
    w [N, k] fp32 or None (all ones).  Returns (y, adapter_rows_evaluated).
    """
    x = x.contiguous()
    N, d_in = x.shape
    K, _, r = A.shape
    d_out = B.shape[2]
    assert A.dtype == x.dtype and B.dtype == x.dtype and B.shape[:2] == (K, r)
    ids2 = ids.to(torch.int32)
    ids2 = (ids2.reshape(-1, 1) if ids2.dim() == 1 else ids2).contiguous()
    k = ids2.shape[1]
    wc = None if w is None else w.to(torch.float32).reshape(N, k).contiguous()
    y = y0.to(torch.float32).clone().contiguous()
    work = ctypes.c_int64(0)
    _load().oracle_lora_apply(_ptr(x), _dtype_code(x), N, d_in, d_out, _ptr(A.contiguous()),
                              _ptr(B.contiguous()), K, r, _ptr(ids2), _ptr(wc), k, float(scale),
                              _ptr(y), ctypes.byref(work))
    return y, int(work.value)


def masked_pass(x, A, B, adapter_of, a, y, scale):
    """One per-sequence pass of adapter a over every token, masked by adapter_of == a.

    Updates y (fp32, contiguous CPU) in place and returns the adapter-rows evaluated (N).
    """
    x = x.contiguous()
    N, d_in = x.shape
    K, _, r = A.shape
    d_out = B.shape[2]
    assert y.dtype == torch.float32 and y.is_contiguous()
    adapter_of = adapter_of.to(torch.int32).contiguous()
    work = ctypes.c_int64(0)
    _load().oracle_masked_pass(_ptr(x), _dtype_code(x), N, d_in, d_out, _ptr(A.contiguous()),
                               _ptr(B.contiguous()), K, r, _ptr(adapter_of), int(a), float(scale),
                               _ptr(y), ctypes.byref(work))
    return int(work.value)


def per_sequence_apply(x, A, B, adapter_of, y0, scale):
    """The per-sequence baseline: K masked passes, one per adapter.  Returns (y, rows = K*N)."""
    K = A.shape[0]
    y = y0.to(torch.float32).clone().contiguous()
    work = 0
    for a in range(K):
        work += masked_pass(x, A, B, adapter_of, a, y, scale)
    return y, work
