"""The C-ABI library builds, loads and exports every entry point include/molora.h declares;
host-side validation rejects bad arguments before any launch (no GPU needed: every call
here returns before touching the CUDA runtime)."""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "molora.h")

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOLORA_API\s+[\w\s\*]+?\b(molora_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from token_adapter_routing_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for name in ("molora_route_vocab", "molora_router_topk", "molora_dispatch", "molora_lora_apply"):
        assert name in syms


@needs_nvcc
def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    import token_adapter_routing_gb300 as m
    assert set(m.EXPORTED) == set(declared_symbols())


@needs_nvcc
def test_only_the_c_abi_is_exported(lib):
    import subprocess
    from token_adapter_routing_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    text_syms = [ln.split()[-1] for ln in out.splitlines() if " T " in ln]
    assert sorted(text_syms) == declared_symbols()


@needs_nvcc
def test_host_validation_rejects_bad_arguments_without_launching(lib):
    P, I64, I32, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_int
    lib.molora_route_vocab.argtypes = [P, I64, P, I32, P, P, P]
    lib.molora_dispatch.argtypes = [P, I64, I32, I32, P, P, P, P, P]
    lib.molora_lora_apply_ex.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, P, P, S,
                                         P]
    lib.molora_router_topk.argtypes = [P, S, I64, I32, P, P, P, P, I32, I32, P, P, P, P]
    lib.molora_status_string.restype = ctypes.c_char_p
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x10004)   # not 16-byte aligned
    INVALID, UNSUPPORTED = 1, 2
    # route_vocab: K out of range, null pointers; N == 0 is a valid no-op
    assert lib.molora_route_vocab(fake, 10, fake, 0, fake, None, None) == INVALID
    assert lib.molora_route_vocab(fake, 10, fake, 65, fake, None, None) == INVALID
    assert lib.molora_route_vocab(None, 10, fake, 4, fake, None, None) == INVALID
    assert lib.molora_route_vocab(None, 0, None, 4, None, None, None) == 0
    lib.molora_route_vocab_ex.argtypes = [P, I64, P, I32, P, P, ctypes.c_uint32, P]
    assert lib.molora_route_vocab_ex(fake, 10, fake, 4, fake, None, 2, None) == INVALID
    assert lib.molora_route_vocab_ex(fake, 10, fake, 0, fake, None, 1, None) == INVALID
    assert lib.molora_route_vocab_ex(None, 10, fake, 4, fake, None, 1, None) == INVALID
    assert lib.molora_route_vocab_ex(None, 0, None, 4, None, None, 1, None) == 0
    # dispatch: k > K, k < 1, K > 64, null outputs
    assert lib.molora_dispatch(fake, 8, 5, 4, fake, fake, fake, None, None) == INVALID
    assert lib.molora_dispatch(fake, 8, 0, 4, fake, fake, fake, None, None) == INVALID
    assert lib.molora_dispatch(fake, 8, 1, 65, fake, fake, fake, None, None) == INVALID
    assert lib.molora_dispatch(fake, 8, 1, 4, None, fake, fake, None, None) == INVALID
    # fused routing + dispatch: K out of range, null pointers; N == 0 still needs counts/offsets
    lib.molora_route_vocab_dispatch.argtypes = [P, I64, P, I32, P, P, P, P, P, P]
    assert lib.molora_route_vocab_dispatch(fake, 8, fake, 0, fake, fake, fake, fake, None, None) == INVALID
    assert lib.molora_route_vocab_dispatch(fake, 8, fake, 65, fake, fake, fake, fake, None, None) == INVALID
    assert lib.molora_route_vocab_dispatch(None, 8, fake, 4, fake, fake, fake, fake, None, None) == INVALID
    assert lib.molora_route_vocab_dispatch(fake, 8, None, 4, fake, fake, fake, fake, None, None) == INVALID
    assert lib.molora_route_vocab_dispatch(fake, 8, fake, 4, fake, fake, None, fake, None, None) == INVALID
    assert lib.molora_route_vocab_dispatch(fake, -1, fake, 4, fake, fake, fake, fake, None, None) == INVALID
    # the flags variant: the same checks, and any flag bit other than INPUTS_READY (1) is refused
    lib.molora_route_vocab_dispatch_ex.argtypes = [P, I64, P, I32, P, P, P, P, P, ctypes.c_uint32, P]
    rvd_ex = lib.molora_route_vocab_dispatch_ex
    assert rvd_ex(fake, 8, fake, 4, fake, fake, fake, fake, None, 2, None) == INVALID
    assert rvd_ex(fake, 8, fake, 4, fake, fake, fake, fake, None, 0x80000001, None) == INVALID
    assert rvd_ex(fake, 8, fake, 0, fake, fake, fake, fake, None, 1, None) == INVALID
    assert rvd_ex(None, 8, fake, 4, fake, fake, fake, fake, None, 1, None) == INVALID
    assert rvd_ex(fake, 8, fake, 4, fake, fake, None, fake, None, 0, None) == INVALID
    assert rvd_ex(fake, -1, fake, 4, fake, fake, fake, fake, None, 1, None) == INVALID
    lib.molora_route_vocab_lora_apply_ex.argtypes = [P, I64, P, I32, P, S, I32, I32, P, P, I32, F, P, I32, P, P, P,
                                                     P, P, ctypes.c_uint32, P]

    def step_ex(flags=1, K=4, y=fake, adapter=fake):
        return lib.molora_route_vocab_lora_apply_ex(fake, 16, fake, K, fake, 1, 64, 64, fake, fake, 16, 2.0, y, 0,
                                                    adapter, fake, fake, fake, None, flags, None)

    assert step_ex(flags=4) == INVALID and step_ex(flags=0xFFFFFFFF) == INVALID
    assert step_ex(K=0) == INVALID and step_ex(y=None) == INVALID and step_ex(adapter=None) == INVALID

    def apply(x=fake, dtype=1, N=16, d_in=64, d_out=64, A=fake, B=fake, K=4, r=16, ids=fake, k=1, y=fake, path=0,
              ws=None, ws_bytes=None):
        return lib.molora_lora_apply_ex(x, dtype, N, d_in, d_out, A, B, K, r, ids, None, k, fake, fake, fake,
                                        2.0, y, ws, ws_bytes, None, path, None)

    assert apply(r=12) == INVALID
    assert apply(K=0) == INVALID and apply(K=65) == INVALID
    assert apply(k=5) == INVALID and apply(k=0) == INVALID
    assert apply(dtype=7) == INVALID
    assert apply(x=None) == INVALID and apply(y=None) == INVALID and apply(ids=None) == INVALID
    assert apply(x=odd) == INVALID and apply(A=odd) == INVALID and apply(B=odd) == INVALID and apply(y=odd) == INVALID
    assert apply(N=-1) == INVALID and apply(d_in=0) == INVALID
    assert apply(path=9) == INVALID and apply(path=-1) == INVALID
    # the stacked path needs a workspace: without ws_bytes it is an invalid request, and an
    # empty batch is a no-op on every path
    assert apply(path=4) == INVALID
    assert apply(N=0, path=4) == 0
    # a query looks at sizes only: bad sizes are still rejected, null pointers are not
    size = ctypes.c_size_t(12345)
    assert apply(x=None, A=None, B=None, ids=None, y=None, ws_bytes=ctypes.byref(size)) == 0
    assert size.value == 0  # no workspace path without the driver's tensor-map encoder
    assert apply(K=0, ws_bytes=ctypes.byref(size)) == INVALID and apply(r=12, ws_bytes=ctypes.byref(size)) == INVALID
    # the grouped tensor-core path needs bf16 and r >= 16
    assert apply(dtype=0, path=2) == UNSUPPORTED
    assert apply(r=8, path=2) == UNSUPPORTED
    assert apply(N=0) == 0
    # bf16 y: the same checks through the bf16-y entry point
    lib.molora_lora_apply_bf16y.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P, P, S, P]

    def apply16(y=fake, r=16, path=0):
        return lib.molora_lora_apply_bf16y(fake, 1, 16, 64, 64, fake, fake, 4, r, fake, None, 1, fake, fake, fake,
                                           2.0, y, None, path, None)

    assert apply16(y=None) == INVALID and apply16(y=odd) == INVALID and apply16(r=12) == INVALID
    assert apply16(r=8, path=2) == UNSUPPORTED
    # indirect layout: per-adapter address tables; a null or unaligned entry is rejected
    lib.molora_lora_apply_indirect.argtypes = [P, S, I64, I32, I32, P, P, I32, I32, P, P, I32, P, P, P, F, P,
                                               I32, P, S, P]
    good = (ctypes.c_void_p * 4)(0x10000, 0x20000, 0x30000, 0x40000)
    with_null = (ctypes.c_void_p * 4)(0x10000, None, 0x30000, 0x40000)
    with_odd = (ctypes.c_void_p * 4)(0x10000, 0x20008, 0x30000, 0x40000)

    def ind(a_tab, b_tab, K=4):
        return lib.molora_lora_apply_indirect(fake, 1, 16, 64, 64, ctypes.cast(a_tab, P), ctypes.cast(b_tab, P), K,
                                              16, fake, None, 1, fake, fake, fake, 2.0, fake, 0, None, 0, None)

    assert ind(with_null, good) == INVALID and ind(good, with_odd) == INVALID
    assert ind(good, good, K=0) == INVALID and ind(good, good, K=65) == INVALID
    assert lib.molora_lora_apply_indirect(fake, 1, 16, 64, 64, None, ctypes.cast(good, P), 4, 16, fake, None, 1,
                                          fake, fake, fake, 2.0, fake, 0, None, 0, None) == INVALID
    # router: k > K, K > 64, null outputs
    assert lib.molora_router_topk(fake, 1, 8, 64, fake, None, fake, None, 4, 5, None, fake, fake, None) == INVALID
    assert lib.molora_router_topk(fake, 1, 8, 64, fake, None, fake, None, 65, 1, None, fake, fake, None) == INVALID
    assert lib.molora_router_topk(fake, 1, 8, 64, fake, None, fake, None, 4, 1, None, None, fake, None) == INVALID
    # router + apply in one kernel: bad k, null or unaligned W1, null w; fp32 and K*r > 128 unsupported
    lib.molora_router_lora_apply.argtypes = [P, S, I64, I32, I32, P, P, P, P, P, P, I32, I32, I32, F, P, P, P, P,
                                             I32, P, P, P, P]

    def fused(dtype=1, K=4, r=16, k=2, W1=fake, w=fake, y=fake):
        return lib.molora_router_lora_apply(fake, dtype, 64, 512, 512, W1, None, fake, None, fake, fake, K, r, k,
                                            2.0, None, fake, w, y, 0, None, None, None, None)

    assert fused(k=5) == INVALID and fused(k=0) == INVALID and fused(W1=None) == INVALID
    assert fused(W1=odd) == INVALID and fused(w=None) == INVALID and fused(y=odd) == INVALID
    assert fused(dtype=0) == UNSUPPORTED and fused(K=16, r=16) == UNSUPPORTED and fused(r=8) == UNSUPPORTED
    assert lib.molora_router_lora_apply(None, 1, 0, 512, 512, None, None, None, None, None, None, 4, 16, 2, 2.0,
                                        None, None, None, None, 0, None, None, None, None) == 0
    # the whole vocabulary-routed step: null outputs, bad K, odd y
    lib.molora_route_vocab_lora_apply.argtypes = [P, I64, P, I32, P, S, I32, I32, P, P, I32, F, P, I32, P, P, P, P,
                                                  P, P]

    def step(K=4, starts=fake, counts=fake, perm=fake, y=fake):
        return lib.molora_route_vocab_lora_apply(fake, 64, starts, K, fake, 1, 512, 512, fake, fake, 16, 2.0, y, 0,
                                                 fake, counts, fake, perm, None, None)

    assert step(starts=None) == INVALID and step(counts=None) == INVALID and step(perm=None) == INVALID
    assert step(K=0) == INVALID and step(K=65) == INVALID and step(y=odd) == INVALID
    assert lib.molora_status_string(1) == b"invalid argument"


def test_binding_has_no_cpu_fallback():
    import torch
    # every entry point refuses host tensors outright: the product path is the CUDA library
    import token_adapter_routing_gb300 as m
    x = torch.zeros(8, 64, dtype=torch.bfloat16)
    A = torch.zeros(4, 64, 16, dtype=torch.bfloat16)
    B = torch.zeros(4, 16, 64, dtype=torch.bfloat16)
    W1 = torch.zeros(64, 64, dtype=torch.bfloat16)
    W2 = torch.zeros(64, 4, dtype=torch.bfloat16)
    ids = torch.zeros(8, 1, dtype=torch.int32)
    tok = torch.zeros(8, dtype=torch.int32)
    starts = torch.tensor([0, 10, 20, 30, 40], dtype=torch.int32)
    y = torch.zeros(8, 64)
    calls = [
        lambda: m.molora_route_vocab(tok, starts),
        lambda: m.molora_router_topk(x, W1, W2, 2),
        lambda: m.molora_dispatch(ids, 4),
        lambda: m.molora_route_vocab_dispatch(tok, starts),
        lambda: m.molora_lora_apply(x, A, B, ids, y, 2.0),
        lambda: m.molora_route_vocab_lora_apply(tok, starts, x, A, B, y, 2.0),
        lambda: m.molora_router_lora_apply(x, W1, W2, A, B, 2, y, 2.0),
        lambda: m.molora_lora_apply_masked_pass(x, A, B, tok, 0, y, 2.0),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def test_binding_rejects_mis_sized_tensors_before_any_launch():
    """The Python binding checks every tensor's size against N, d_out, K and k before it looks
    at devices (so these CPU tensors fail on their sizes, with the argument named), and a
    correctly sized CPU tensor fails only for not being on a GPU: nothing reaches the library."""
    import torch
    import token_adapter_routing_gb300 as m
    N, d_in, d_out, K, r, k = 8, 64, 32, 4, 16, 2
    x = torch.zeros(N, d_in, dtype=torch.bfloat16)
    A = torch.zeros(K, d_in, r, dtype=torch.bfloat16)
    B = torch.zeros(K, r, d_out, dtype=torch.bfloat16)
    ids = torch.zeros(N, k, dtype=torch.int32)
    w = torch.zeros(N, k)
    y = torch.zeros(N, d_out)
    counts = torch.zeros(K, dtype=torch.int32)
    offsets = torch.zeros(K + 1, dtype=torch.int32)
    perm = torch.zeros(N * k, dtype=torch.int32)
    ok = dict(w=w, counts=counts, offsets=offsets, perm=perm)

    def apply(**kw):
        args = dict(ok)
        args.update(kw)
        yy = args.pop("y", y)
        ii = args.pop("ids", ids)
        return m.molora_lora_apply(x, A, B, ii, yy, 2.0, **args)

    with pytest.raises(ValueError, match="y must be"):
        apply(y=torch.zeros(N, d_out + 1))
    with pytest.raises(ValueError, match="y must be"):
        apply(y=torch.zeros(N + 1, d_out))
    with pytest.raises(ValueError, match="ids must be"):
        apply(ids=torch.zeros(N + 1, k, dtype=torch.int32))
    with pytest.raises(ValueError, match="w must"):
        apply(w=torch.zeros(N, k + 1))
    with pytest.raises(ValueError, match="counts must"):
        apply(counts=torch.zeros(K + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="offsets must"):
        apply(offsets=torch.zeros(K, dtype=torch.int32))
    with pytest.raises(ValueError, match="perm must"):
        apply(perm=torch.zeros(N, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        apply()
    with pytest.raises(ValueError, match="perm must"):
        m.molora_dispatch(ids, K, perm=torch.zeros(N * k - 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="offsets must"):
        m.molora_dispatch(ids, K, offsets=torch.zeros(K + 2, dtype=torch.int32))
    W1 = torch.zeros(d_in, 64, dtype=torch.bfloat16)
    W2 = torch.zeros(64, K, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="logits must"):
        m.molora_router_topk(x, W1, W2, k, logits=torch.zeros(N, K + 1))
    with pytest.raises(ValueError, match="ids must"):
        m.molora_router_topk(x, W1, W2, k, ids=torch.zeros(N, k + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="y must be"):
        m.molora_router_lora_apply(x, W1, W2, A, B, k, torch.zeros(N, d_out - 1), 2.0)
    with pytest.raises(ValueError, match="w must"):
        m.molora_router_lora_apply(x, W1, W2, A, B, k, y, 2.0, w=torch.zeros(N, k + 1))
    tok = torch.zeros(N, dtype=torch.int32)
    starts = torch.arange(K + 1, dtype=torch.int32)
    with pytest.raises(ValueError, match="perm must"):
        m.molora_route_vocab_dispatch(tok, starts, perm=torch.zeros(N + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="counts must"):
        m.molora_route_vocab_dispatch_ex(tok, starts, m.INPUTS_READY, counts=torch.zeros(K + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="adapter must"):
        m.molora_route_vocab(tok, starts, adapter=torch.zeros(N - 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="adapter_of must"):
        m.molora_lora_apply_masked_pass(x, A, B, torch.zeros(N + 1, dtype=torch.int32), 0, y, 2.0)


def test_launching_calls_run_on_the_tensors_device():
    """Every launching binding runs with its tensors' device current (a device guard), so a
    caller whose current device differs still launches where the data lives."""
    import token_adapter_routing_gb300 as m
    for name in ("molora_route_vocab", "molora_route_vocab_ex", "molora_router_topk", "molora_dispatch",
                 "molora_route_vocab_dispatch", "molora_route_vocab_dispatch_ex", "molora_lora_apply",
                 "molora_route_vocab_lora_apply",
                 "molora_route_vocab_lora_apply_ex", "molora_router_lora_apply",
                 "molora_lora_apply_static_ws", "molora_lora_apply_masked_pass", "molora_selftest_bounded_wait"):
        fn = getattr(m, name)
        assert getattr(fn, "__wrapped__", None) is not None, f"{name} has no device guard"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_header_compiles_as_c99(tmp_path):
    """include/molora.h is a C ABI: a C99 translation unit that includes it and takes the
    address of every declared entry point compiles without warnings from the header itself."""
    import subprocess
    cuda_inc = "/usr/local/cuda/include"
    if not os.path.isdir(cuda_inc):
        pytest.skip("CUDA headers not available")
    body = "\n".join(f"  (void)&{name};" for name in declared_symbols())
    src = tmp_path / "abi.c"
    src.write_text(f'#include "molora.h"\nint main(void) {{\n  uint32_t f = MOLORA_INPUTS_READY;\n  (void)f;\n{body}\n'
                   "  return 0;\n}\n")
    out = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                          "-c", str(src), "-o", str(tmp_path / "abi.o")], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "molora.h" not in out.stderr, out.stderr
