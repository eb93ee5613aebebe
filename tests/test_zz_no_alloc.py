"""The allocation-free entry point, molora_lora_apply_static_ws, called through the C ABI.

It serves callers that cannot allocate device memory (an allocator that owns all of it, a
path that may not risk cudaMalloc/cudaFree synchronising the device, or a caller holding only
raw pointers and a stream): the stacked apply then takes its workspace from a fixed scratch
buffer inside the library instead of from the caller.  These tests check that two calls in a
row give the same y as the workspace-taking entry point (molora_lora_apply_ex on the stacked
path) within the tolerance the parity tests use, and that a problem too large for the
buffer is refused before any launch.  The file is collected last, and it needs nothing from
the other test files, so it passes alone in a fresh process as well as after them.
"""

import ctypes
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

STACKED = 4
OK, ERR_SCRATCH_TOO_SMALL = 0, 4
TOL = 2e-4  # relative to rms(y): the tight bound of the apply parity tests


@pytest.fixture(scope="module")
def lib():
    from token_adapter_routing_gb300 import build
    lib = ctypes.CDLL(build.build())
    P, I64, I32, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_int
    lib.molora_lora_apply_static_ws.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, F, P, P, P]
    lib.molora_lora_apply_static_ws.restype = ctypes.c_int
    lib.molora_lora_apply_ex.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, P, P, S, P]
    lib.molora_lora_apply_ex.restype = ctypes.c_int
    return lib


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def inputs(N, d_in, d_out, K, r, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(N, d_in, generator=g).to(torch.bfloat16).cuda()
    A = (torch.randn(K, d_in, r, generator=g) / math.sqrt(d_in)).to(torch.bfloat16).cuda()
    B = (torch.randn(K, r, d_out, generator=g) / math.sqrt(r)).to(torch.bfloat16).cuda()
    y0 = torch.randn(N, d_out, generator=g).cuda()
    ids = torch.stack([torch.randperm(K, generator=g)[:k] for _ in range(N)]).to(torch.int32).cuda()
    w = torch.softmax(torch.randn(N, k, generator=g), dim=1).cuda()
    return x, A, B, y0, ids, w


@pytest.mark.parametrize("N,d_in,d_out,K,r,k", [(1000, 1024, 1536, 8, 64, 2),
                                                # N*K*r = 4M: the largest problem the buffer holds
                                                (8192, 4096, 4096, 8, 64, 4)])
def test_static_scratch_matches_workspace_entry_point(lib, N, d_in, d_out, K, r, k):
    x, A, B, y0, ids, w = inputs(N, d_in, d_out, K, r, k, seed=N + k)
    stream = torch.cuda.current_stream().cuda_stream
    # the existing entry point with a caller-owned workspace
    need = ctypes.c_size_t(0)
    assert lib.molora_lora_apply_ex(None, 1, N, d_in, d_out, None, None, K, r, None, None, k, None, None, None,
                                    2.0, None, None, ctypes.byref(need), None, STACKED, None) == OK
    ws = torch.empty(need.value, dtype=torch.uint8, device="cuda")
    size = ctypes.c_size_t(need.value)
    y_ref = y0.clone()
    assert lib.molora_lora_apply_ex(ptr(x), 1, N, d_in, d_out, ptr(A), ptr(B), K, r, ptr(ids), ptr(w), k, None, None,
                                    None, 2.0, ptr(y_ref), ptr(ws), ctypes.byref(size), None, STACKED, stream) == OK
    # two calls in a row of the allocation-free entry point, each on a fresh copy of y0
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for _ in range(2):
        y = y0.clone()
        assert lib.molora_lora_apply_static_ws(ptr(x), 1, N, d_in, d_out, ptr(A), ptr(B), K, r, ptr(ids), ptr(w), k,
                                               2.0, ptr(y), ptr(e), stream) == OK
        ys.append(y)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    rms = y_ref.double().pow(2).mean().sqrt().item()
    for y in ys:
        err = (y.double() - y_ref.double()).abs().max().item()
        assert err <= TOL * rms, f"max|dy| {err:.3e} > {TOL} rms ({rms:.3e})"


def test_static_scratch_refuses_problems_beyond_its_size(lib):
    # N*K*r = 4M + 64: one token more than the buffer holds at K*r = 512; refused on the host,
    # so the pointers are never looked at
    fake = ctypes.c_void_p(0x10000)
    st = lib.molora_lora_apply_static_ws(fake, 1, 8193, 4096, 4096, fake, fake, 8, 64, fake, None, 2, 2.0, fake, None,
                                         None)
    assert st == ERR_SCRATCH_TOO_SMALL
