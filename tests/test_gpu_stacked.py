"""GPU parity of the stacked top-k path (shrink into a workspace, then the expand GEMM), called
through the C ABI, against the CPU oracle.

Same bars as test_gpu_parity.py: max|dy| <= 1e-2 * rms(oracle y) with the tight 2e-4 check
(the shrink output reaches the expand as two bf16 terms, relative error 2^-17); small-integer
inputs bit-exact; learned top-k ids exact on clear tokens and weights within 1e-5.  Every
y element receives one addition, so two runs agree bit for bit for any k.
"""

import pytest
import torch

import oracle
import workloads
from test_gpu_parity import (TOL_CONTRACT, assert_apply_close, check_learned_apply, dev, err_word, make_adapters,
                             random_topk, small_int_case)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from token_adapter_routing_gb300 import build
    build.build()
    import token_adapter_routing_gb300 as mod
    mod.load_library()
    return mod


def ws_bytes(N, K, r):
    g = (N * K * r * 2 + 255) // 256 * 256
    return 2 * g


# K*r from 64 to 1024 (one, two or four CTAs per tile), ragged N, d_out that is not a multiple
# of the 256-column tile, and d_out below 256 (128-column tiles)
CASES = [(8, 64, 2, 700, 1024, 1536), (4, 16, 1, 300, 512, 512), (16, 16, 3, 513, 1024, 1000),
         (4, 64, 4, 129, 2048, 320), (16, 64, 2, 257, 512, 768), (8, 32, 1, 1, 256, 200),
         (2, 16, 2, 640, 128, 128), (8, 64, 4, 128, 4096, 4096),
         # an odd K and K = 1 (plain LoRA) keep the whole stacked operand in one CTA per tile
         (3, 64, 2, 300, 512, 512), (1, 64, 1, 100, 256, 256)]


@pytest.mark.parametrize("K,r,k,N,d_in,d_out", CASES)
def test_stacked_apply_vs_oracle(m, K, r, k, N, d_in, d_out):
    x, A, B, y0 = make_adapters(N, d_in, d_out, K, r, seed=N + K * r + k)
    ids, w = random_topk(N, K, k, seed=k + 11)
    y, y2 = dev(y0).clone(), dev(y0).clone()
    e = err_word()
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(ids), y, 2.0, w=dev(w), err_word=e, path="stacked")
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(ids), y2, 2.0, w=dev(w), path="stacked")
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(y.cpu(), y2.cpu())  # one addition per y element: reproducible for any k
    y_ref, _ = oracle.lora_apply(x, A, B, ids, y0, 2.0, w)
    assert_apply_close(y, y_ref)


@pytest.mark.parametrize("N,d_in,d_out,K,r,k", [(200, 128, 256, 4, 16, 1), (130, 256, 384, 8, 64, 3),
                                                (64, 64, 64, 8, 64, 4), (301, 192, 320, 16, 16, 2)])
def test_stacked_small_integers_bitexact(m, N, d_in, d_out, K, r, k):
    # every partial sum is an exact fp32 integer (or dyadic): any summation order gives the
    # oracle's bits, so the stacked path must reproduce them exactly
    x, A, B, y0, ids, w = small_int_case(N, d_in, d_out, K, r, k, N + d_in + r)
    y_ref, _ = oracle.lora_apply(x, A, B, ids, y0, 0.5, w)
    y = dev(y0).clone()
    e = err_word()
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(ids), y, 0.5, w=dev(w), err_word=e, path="stacked")
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(y.cpu(), y_ref)


def test_stacked_degenerate_and_invalid_ids(m):
    N, d_in, d_out, K, r, k = 300, 512, 640, 8, 32, 2
    x, A, B, y0 = make_adapters(N, d_in, d_out, K, r, seed=5)
    ids, w = random_topk(N, K, k, seed=6)
    # B = 0 and w = 0 leave y at y0 bit for bit
    y = dev(y0).clone()
    m.molora_lora_apply(dev(x), dev(A), dev(torch.zeros_like(B)), dev(ids), y, 2.0, w=dev(w), path="stacked")
    assert torch.equal(y.cpu(), y0)
    y = dev(y0).clone()
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(ids), y, 2.0, w=torch.zeros(N, k, device="cuda"), path="stacked")
    assert torch.equal(y.cpu(), y0)
    # k = K with uniform weights: the dense sum of all adapters
    idsK = torch.stack([torch.randperm(K) for _ in range(N)]).to(torch.int32)
    wK = torch.full((N, K), 1.0 / K)
    y = dev(y0).clone()
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(idsK), y, 2.0, w=dev(wK), path="stacked")
    y_ref, _ = oracle.lora_apply(x, A, B, idsK, y0, 2.0, wK)
    assert_apply_close(y, y_ref)
    # ids outside [0, K) are skipped and reported, as by the oracle
    bad = ids.clone()
    bad[5, 0], bad[77, 1], bad[299, 0] = -1, K, 1000
    y = dev(y0).clone()
    e = err_word()
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(bad), y, 2.0, w=dev(w), err_word=e, path="stacked")
    torch.cuda.synchronize()
    assert int(e.item()) == m.DEV_BAD_ADAPTER_ID
    y_ref, _ = oracle.lora_apply(x, A, B, bad, y0, 2.0, w)
    assert_apply_close(y, y_ref)
    # w = None means weight one per slot
    y = dev(y0).clone()
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(ids), y, 2.0, path="stacked")
    y_ref, _ = oracle.lora_apply(x, A, B, ids, y0, 2.0, None)
    assert_apply_close(y, y_ref)


def test_stacked_workspace_convention_and_graph(m):
    N, d_in, d_out, K, r, k = 1100, 1024, 1024, 8, 64, 2
    need = m.molora_workspace_bytes(N, d_in, d_out, K, r, k, path="stacked")
    assert need == ws_bytes(N, K, r)
    assert m.molora_workspace_bytes(N, d_in, d_out, K, r, k, path="grouped") == 0
    assert m.molora_select_path(torch.bfloat16, N, d_in, d_out, K, r, k) == "stacked"
    assert m.molora_workspace_bytes(N, d_in, d_out, K, r, k) == need  # AUTO picks the stacked pair
    x, A, B, y0 = make_adapters(N, d_in, d_out, K, r, seed=7)
    ids, w = random_topk(N, K, k, seed=8)
    xd, Ad, Bd, idsd, wd = dev(x), dev(A), dev(B), dev(ids), dev(w)
    # a workspace one byte short, or not 256-byte aligned, is rejected before any launch
    small = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoloraError):
        m.molora_lora_apply(xd, Ad, Bd, idsd, dev(y0), 2.0, w=wd, path="stacked", ws=small)
    big = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoloraError):
        m.molora_lora_apply(xd, Ad, Bd, idsd, dev(y0), 2.0, w=wd, path="stacked", ws=big[16:])
    # a caller-owned workspace, reused, inside a captured CUDA graph
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = dev(y0).clone()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            m.molora_lora_apply(xd, Ad, Bd, idsd, y, 2.0, w=wd, ws=ws)
    for _ in range(3):
        y.copy_(dev(y0))
        graph.replay()
    torch.cuda.synchronize()
    y_ref, _ = oracle.lora_apply(x, A, B, ids, y0, 2.0, w)
    assert_apply_close(y, y_ref)


# learned router + apply through the stacked pair: K*r = 512 (two CTAs per tile), 1024 (four),
# 64 and 256 (one or two), ragged N
ROUTER_CASES = [({"N": 700, "d_in": 1024, "d_out": 1536}, 2), ({"N": 300, "d_in": 512, "d_out": 512, "K": 16}, 3),
                ({"N": 333, "d_in": 1024, "d_out": 768, "K": 4, "r": 16}, 2),
                ({"N": 129, "d_in": 2048, "d_out": 512, "K": 4}, 4), ({"N": 257, "d_in": 256, "d_out": 256}, 1),
                # K = 5: no even split, one CTA per tile carries all 80 adapter and 64 router columns
                ({"N": 200, "d_in": 512, "d_out": 512, "K": 5, "r": 16}, 2)]


@pytest.mark.parametrize("kw,k", ROUTER_CASES)
def test_stacked_router_apply_vs_oracle(m, kw, k):
    wl = workloads.make("topk_scaling", k=k, **kw)
    x, W1, W2, A, B = dev(wl.x), dev(wl.W1), dev(wl.W2), dev(wl.A), dev(wl.B)
    need = m.molora_workspace_bytes(wl.N, wl.d_in, wl.d_out, wl.K, wl.r, k, router=True)
    ws = torch.empty(max(need, ws_bytes(wl.N, wl.K, wl.r)), dtype=torch.uint8, device="cuda")
    y, y2 = dev(wl.y0).clone(), dev(wl.y0).clone()
    e = err_word()
    # an explicit workspace forces the stacked pair wherever it applies
    logits, ids, w = m.molora_router_lora_apply(x, W1, W2, A, B, k, y, wl.scale, err_word=e, ws=ws)
    logits2, ids2, w2 = m.molora_router_lora_apply(x, W1, W2, A, B, k, y2, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    for a_, b_ in ((y, y2), (logits, logits2), (ids, ids2), (w, w2)):
        assert torch.equal(a_.cpu(), b_.cpu())
    check_learned_apply(wl, k, logits, ids, w, y)


def test_stacked_router_biases_and_graph(m):
    wl = workloads.make("topk_scaling", N=515, d_in=1024, d_out=1024, k=2)
    g = torch.Generator().manual_seed(9)
    b1 = torch.randn(64, generator=g) * 0.1
    b2 = torch.randn(wl.K, generator=g) * 0.1
    x, W1, W2, A, B = dev(wl.x), dev(wl.W1), dev(wl.W2), dev(wl.A), dev(wl.B)
    need = m.molora_workspace_bytes(wl.N, wl.d_in, wl.d_out, wl.K, wl.r, 2, router=True)
    assert need == ws_bytes(wl.N, wl.K, wl.r)  # K*r = 512: only the stacked pair applies
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = dev(wl.y0).clone()
    logits, ids, w = m.molora_router_lora_apply(x, W1, W2, A, B, 2, y, wl.scale, b1=dev(b1), b2=dev(b2), ws=ws)
    torch.cuda.synchronize()
    check_learned_apply(wl, 2, logits, ids, w, y, b1=b1, b2=b2)
    # without logits, captured in a CUDA graph and replayed
    yg = dev(wl.y0).clone()
    ids_g = torch.empty(wl.N, 2, dtype=torch.int32, device="cuda")
    w_g = torch.empty(wl.N, 2, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            m.molora_router_lora_apply(x, W1, W2, A, B, 2, yg, wl.scale, ids=ids_g, w=w_g, want_logits=False, ws=ws)
    for _ in range(3):
        yg.copy_(dev(wl.y0))
        graph.replay()
    torch.cuda.synchronize()
    lg = m.molora_router_lora_apply(x, W1, W2, A, B, 2, dev(wl.y0).clone(), wl.scale, ws=ws)[0]
    check_learned_apply(wl, 2, lg, ids_g, w_g, yg)
    # no workspace allowed: K*r = 512 has no one-kernel path
    with pytest.raises(m.MoloraError):
        m.molora_router_lora_apply(x, W1, W2, A, B, 2, dev(wl.y0).clone(), wl.scale, use_ws=False)


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_full_size_topk_scaling_stacked(m, k):
    # N=8192, d=4096, K=8, r=64: the fused router + stacked apply at full size, twice (bit-equal),
    # against the oracle on sampled tokens that cover every 128-row tile and the last row
    wl = workloads.make("topk_scaling", k=k)
    x, W1, W2, A, B = dev(wl.x), dev(wl.W1), dev(wl.W2), dev(wl.A), dev(wl.B)
    ws = torch.empty(ws_bytes(wl.N, wl.K, wl.r), dtype=torch.uint8, device="cuda")
    y, y2 = dev(wl.y0).clone(), dev(wl.y0).clone()
    e = err_word()
    logits, ids, w = m.molora_router_lora_apply(x, W1, W2, A, B, k, y, wl.scale, err_word=e, ws=ws)
    m.molora_router_lora_apply(x, W1, W2, A, B, k, y2, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(y.cpu(), y2.cpu())
    g = torch.Generator().manual_seed(100 + k)
    tiles = wl.N // 128
    rows = torch.cat([torch.arange(tiles) * 128 + torch.randint(0, 128, (tiles,), generator=g),
                      torch.tensor([0, wl.N - 1])])
    check_learned_apply(wl, k, logits, ids, w, y, rows=rows)
    # the apply alone on the oracle's own routing of the same rows agrees too
    ys = dev(wl.y0).clone()
    m.molora_lora_apply(x, A, B, ids, ys, wl.scale, w=w, ws=ws, path="stacked")
    torch.cuda.synchronize()
    assert torch.equal(ys.cpu(), y.cpu())  # same G, same expand: the router's choice drives both


@pytest.mark.parametrize("N,K,r,k,want", [(2048, 16, 16, 1, "grouped"), (2048, 16, 16, 4, "stacked"),
                                          (8192, 8, 64, 1, "stacked"), (1024, 4, 64, 1, "grouped"),
                                          (1024, 4, 64, 2, "stacked"), (4096, 64, 16, 4, "stacked"),
                                          (2048, 64, 16, 2, "grouped"), (8192, 16, 64, 1, "grouped"),
                                          (2048, 8, 64, 1, "grouped"), (4096, 8, 64, 1, "stacked"),
                                          (2048, 64, 16, 4, "stacked")])
def test_auto_stacked_or_grouped_follows_the_measured_crossover(m, N, K, r, k, want):
    """At d = 4096 AUTO (with a workspace) takes the stacked pair only where it measured faster
    than dispatch + grouped apply: few adapters per selected one, enough tokens."""
    assert m.molora_select_path(torch.bfloat16, N, 4096, 4096, K, r, k) == want


@pytest.mark.parametrize("N,K,r,want", [(128, 8, 64, "scalar"), (160, 8, 64, "grouped"), (384, 16, 64, "scalar"),
                                        (512, 16, 64, "grouped"), (512, 32, 64, "scalar"), (768, 32, 64, "grouped"),
                                        (768, 64, 64, "scalar"), (1024, 64, 64, "grouped"), (512, 16, 32, "scalar"),
                                        (768, 16, 32, "grouped"), (1024, 32, 32, "scalar"), (1536, 32, 32, "grouped"),
                                        (512, 8, 16, "scalar"), (768, 8, 16, "grouped"), (768, 16, 16, "scalar"),
                                        (2048, 64, 16, "scalar")])
def test_auto_scalar_or_grouped_by_rank(m, N, K, r, want):
    """Top-1 at d = 4096: the scalar path re-reads a token's adapter from L2 per token, so the
    measured crossover to the grouped path falls with the rank (near batch 160 for 8 adapters of
    rank 64, as Figures 5 and 9 find)."""
    assert m.molora_select_path(torch.bfloat16, N, 4096, 4096, K, r, 1) == want


@pytest.mark.parametrize("with_ws", [True, False])
def test_auto_without_dispatch_outputs_picks_a_path_that_needs_none(m, with_ws):
    """A shape where AUTO prefers the grouped path, called without counts/offsets/perm: AUTO
    runs the stacked pair when a workspace is given and the scalar path otherwise, and either
    matches the oracle."""
    N, d_in, d_out, K, r, k = 2048, 1024, 1024, 16, 16, 1
    assert m.molora_select_path(torch.bfloat16, N, d_in, d_out, K, r, k) == "grouped"
    x, A, B, y0 = make_adapters(N, d_in, d_out, K, r, seed=31)
    ids, w = random_topk(N, K, k, seed=32)
    y = dev(y0).clone()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    if with_ws:
        ws = torch.empty(m.molora_workspace_bytes(N, d_in, d_out, K, r, k, path="stacked"), dtype=torch.uint8,
                         device="cuda")
    m.molora_lora_apply(dev(x), dev(A), dev(B), dev(ids), y, 2.0, w=dev(w), err_word=e, ws=ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    y_ref, _ = oracle.lora_apply(x, A, B, ids, y0, 2.0, w)
    assert_apply_close(y, y_ref)
