"""Pins for the CPU oracle, checked against things other than the oracle itself.

Source: "MoLoRA: Composable Specialization via Per-Token Adapter Routing".  The pages print
no input/output values, so the pins are: hand-worked examples (tests/golden), library
routines for the special cases that reduce to them (searchsorted, argmax, softmax, stable
argsort, float64 matmul), closed forms (k = K with uniform weights is the dense sum of all
adapters; K = 1 is textbook LoRA), invariants stated by the pages (per-token routing equals
K masked per-sequence passes while evaluating N instead of K*N adapter-rows, Tables 3 and 7),
degenerate cases (B = 0, w = 0, no valid id leave y at the base output) and brute force on
tiny small-integer inputs, where every partial sum is exact so any order gives the same bits.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_molora.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- route_vocab

def test_route_vocab_golden():
    g = _golden()["vocab"]
    adapter, n_out = oracle.route_vocab(torch.tensor(g["tok"]), torch.tensor(g["starts"]))
    assert adapter.tolist() == g["expected_adapter"]
    assert n_out == sum(1 for a in g["expected_adapter"] if a < 0)


@pytest.mark.parametrize("K", [1, 3, 4, 64])
def test_route_vocab_matches_searchsorted(K):
    gen = torch.Generator().manual_seed(7 + K)
    # unequal, strictly increasing ranges that do not start at 0
    widths = torch.randint(1, 500, (K,), generator=gen)
    starts = torch.cat([torch.tensor([100]), 100 + torch.cumsum(widths, 0)]).to(torch.int32)
    tok = torch.randint(0, int(starts[-1]) + 200, (5000,), generator=gen, dtype=torch.int32)
    adapter, n_out = oracle.route_vocab(tok, starts)
    s = starts.numpy()
    idx = np.searchsorted(s, tok.numpy(), side="right") - 1
    inside = (tok.numpy() >= s[0]) & (tok.numpy() < s[-1])
    expect = np.where(inside, idx, -1)
    assert np.array_equal(adapter.numpy(), expect)
    assert n_out == int((~inside).sum())
    # both ends of every range map to that range
    lo = starts[:-1]
    hi = starts[1:] - 1
    a_lo, _ = oracle.route_vocab(lo, starts)
    a_hi, _ = oracle.route_vocab(hi, starts)
    assert a_lo.tolist() == list(range(K)) and a_hi.tolist() == list(range(K))


# ----------------------------------------------------------------------------- router

def _router_case(N, d_in, K, seed, dtype=torch.float32):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(N, d_in, generator=gen).to(dtype)
    W1 = (torch.randn(d_in, 64, generator=gen) / math.sqrt(d_in)).to(dtype)
    W2 = (torch.randn(64, K, generator=gen) / 8.0).to(dtype)
    b1 = torch.randn(64, generator=gen) * 0.1
    b2 = torch.randn(K, generator=gen) * 0.1
    return x, W1, W2, b1, b2


def _router_logits_f64(x, W1, W2, b1, b2):
    h = torch.relu(x.double() @ W1.double() + (0 if b1 is None else b1.double()))
    return h @ W2.double() + (0 if b2 is None else b2.double())


def test_router_golden():
    g = _golden()["router"]
    W1 = torch.zeros(2, 64)
    W1[:, 0] = torch.tensor(g["W1_nonzero"]["col0"], dtype=torch.float32)
    W1[:, 1] = torch.tensor(g["W1_nonzero"]["col1"], dtype=torch.float32)
    W1[:, 2] = torch.tensor(g["W1_nonzero"]["col2"], dtype=torch.float32)
    W2 = torch.zeros(64, 3)
    W2[0] = torch.tensor(g["W2_nonzero_rows"]["row0"])
    W2[1] = torch.tensor(g["W2_nonzero_rows"]["row1"])
    x = torch.tensor(g["x"], dtype=torch.float32)
    for k in (1, 2, 3):
        logits, ids, w = oracle.router_topk(x, W1, W2, k)
        assert logits[0].tolist() == g["expected_logits"]
        assert ids[0].tolist() == g[f"k{k}"]["ids"]
        assert torch.allclose(w[0].double(), torch.tensor(g[f"k{k}"]["w"], dtype=torch.float64), rtol=1e-7, atol=0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_router_logits_match_float64_matmul(dtype):
    x, W1, W2, b1, b2 = _router_case(64, 96, 8, 11, dtype)
    logits, _, _ = oracle.router_topk(x, W1, W2, 2, b1, b2)
    ref = _router_logits_f64(x, W1, W2, b1, b2)
    assert torch.allclose(logits.double(), ref, rtol=1e-6, atol=1e-6)
    # without biases the bias terms must vanish
    logits0, _, _ = oracle.router_topk(x, W1, W2, 2)
    assert torch.allclose(logits0.double(), _router_logits_f64(x, W1, W2, None, None), rtol=1e-6, atol=1e-6)


def test_router_top1_is_argmax_and_topK_is_full_softmax():
    x, W1, W2, b1, b2 = _router_case(200, 32, 6, 3)
    logits, ids, w = oracle.router_topk(x, W1, W2, 1, b1, b2)
    assert np.array_equal(ids[:, 0].numpy(), np.argmax(logits.numpy(), axis=1))
    assert torch.all(w == 1.0)
    logits, ids, w = oracle.router_topk(x, W1, W2, 6, b1, b2)
    l64 = logits.double().numpy()
    sm = np.exp(l64 - l64.max(1, keepdims=True))
    sm /= sm.sum(1, keepdims=True)
    order = np.argsort(-logits.numpy(), axis=1, kind="stable")
    assert np.array_equal(ids.numpy(), order)
    assert np.allclose(w.double().numpy(), np.take_along_axis(sm, order, 1), rtol=1e-6, atol=0)
    assert np.allclose(w.double().sum(1).numpy(), 1.0, atol=1e-6)


@pytest.mark.parametrize("K,k", [(4, 2), (5, 3), (8, 2), (8, 4)])
def test_router_topk_brute_force_subsets(K, k):
    x, W1, W2, b1, b2 = _router_case(60, 24, K, 100 + K * 10 + k)
    logits, ids, w = oracle.router_topk(x, W1, W2, k, b1, b2)
    for t in range(x.shape[0]):
        lt = logits[t].tolist()
        best = max(itertools.combinations(range(K), k), key=lambda c: (sum(lt[a] for a in c), [-a for a in c]))
        chosen = ids[t].tolist()
        assert sorted(chosen) == sorted(best)
        assert all(lt[chosen[i]] >= lt[chosen[i + 1]] for i in range(k - 1))
        e = [math.exp(lt[a] - lt[chosen[0]]) for a in chosen]
        assert np.allclose(w[t].tolist(), [v / sum(e) for v in e], rtol=1e-6, atol=0)


def test_router_ties_go_to_lower_index():
    x, W1, W2, _, _ = _router_case(50, 16, 6, 5)
    W2[:, 4] = W2[:, 1]  # adapters 1 and 4 always tie
    W2[:, 5] = W2[:, 1]
    logits, ids, w = oracle.router_topk(x, W1, W2, 3)
    assert torch.equal(logits[:, 1], logits[:, 4])
    for t in range(50):
        chosen = ids[t].tolist()
        for a, b in ((1, 4), (1, 5), (4, 5)):
            if b in chosen:
                assert a in chosen and chosen.index(a) < chosen.index(b)


# ----------------------------------------------------------------------------- dispatch

def test_dispatch_golden():
    g = _golden()["dispatch"]
    counts, offsets, perm, n_inv = oracle.dispatch(torch.tensor(g["ids"]), g["K"])
    assert counts.tolist() == g["expected_counts"]
    assert offsets.tolist() == g["expected_offsets"]
    assert perm.tolist() == g["expected_perm"]
    assert n_inv == 0


@pytest.mark.parametrize("N,k,K", [(1, 1, 1), (777, 1, 4), (300, 3, 8), (1000, 2, 64), (0, 2, 4)])
def test_dispatch_matches_stable_argsort(N, k, K):
    gen = torch.Generator().manual_seed(N + 31 * k + K)
    ids = torch.randint(-1, K + 1, (N, k), generator=gen, dtype=torch.int32)  # includes invalid ids
    counts, offsets, perm, n_inv = oracle.dispatch(ids, K)
    flat = ids.reshape(-1).numpy()
    valid = (flat >= 0) & (flat < K)
    assert np.array_equal(counts.numpy(), np.bincount(flat[valid], minlength=K))
    assert offsets[0] == 0 and np.array_equal(offsets[1:].numpy(), np.cumsum(counts.numpy()))
    nv = int(valid.sum())
    assert n_inv == N * k - nv
    order = np.argsort(np.where(valid, flat, K + 1), kind="stable")[:nv]
    assert np.array_equal(perm[:nv].numpy(), order)
    assert np.all(perm[nv:].numpy() == -1)
    for a in range(K):
        grp = perm[offsets[a]:offsets[a + 1]].numpy()
        assert np.all(flat[grp] == a) and np.all(np.diff(grp) > 0)


# ----------------------------------------------------------------------------- lora apply

def test_apply_golden():
    g = _golden()["apply"]
    y, rows = oracle.lora_apply(torch.tensor(g["x"], dtype=torch.float32),
                                torch.tensor(g["A"], dtype=torch.float32),
                                torch.tensor(g["B"], dtype=torch.float32),
                                torch.tensor(g["ids"]), torch.tensor(g["y0"], dtype=torch.float32),
                                g["scale"], torch.tensor(g["w"], dtype=torch.float32))
    assert y.tolist() == g["expected_y"]
    assert rows == 6


def _small_int_case(N, d_in, d_out, K, r, k, seed, dtype):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randint(-3, 4, (N, d_in), generator=gen).to(dtype)
    A = torch.randint(-2, 3, (K, d_in, r), generator=gen).to(dtype)
    B = torch.randint(-2, 3, (K, r, d_out), generator=gen).to(dtype)
    y0 = torch.randint(-8, 9, (N, d_out), generator=gen).to(torch.float32)
    ids = torch.stack([torch.randperm(K, generator=gen)[:k] for _ in range(N)]).to(torch.int32)
    w = (2.0 ** torch.randint(-3, 1, (N, k), generator=gen)).to(torch.float32)
    return x, A, B, y0, ids, w


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,d_in,d_out,K,r,k", [(8, 8, 8, 4, 2, 2), (5, 7, 3, 3, 2, 3), (6, 4, 9, 4, 1, 1)])
def test_apply_brute_force_small_integers(dtype, N, d_in, d_out, K, r, k):
    x, A, B, y0, ids, w = _small_int_case(N, d_in, d_out, K, r, k, N * 100 + d_in, dtype)
    scale = 0.5
    y, rows = oracle.lora_apply(x, A, B, ids, y0, scale, w)
    # hand-unrolled triple loop in plain Python floats: every value is a small dyadic
    # rational, so the result is exact and order-free
    X, AA, BB, Y0, I, W = (x.float().tolist(), A.float().tolist(), B.float().tolist(),
                            y0.tolist(), ids.tolist(), w.tolist())
    expect = [row[:] for row in Y0]
    for t in range(N):
        for j in range(k):
            a = I[t][j]
            h = [sum(X[t][i] * AA[a][i][q] for i in range(d_in)) for q in range(r)]
            for o in range(d_out):
                expect[t][o] += scale * W[t][j] * sum(h[q] * BB[a][q][o] for q in range(r))
    assert y.tolist() == expect
    assert rows == N * k


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_apply_single_adapter_is_textbook_lora(dtype):
    gen = torch.Generator().manual_seed(21)
    N, d_in, d_out, r = 40, 48, 24, 6  # every dimension distinct: a transposed operand fails
    x = torch.randn(N, d_in, generator=gen).to(dtype)
    A = (torch.randn(1, d_in, r, generator=gen) / 7).to(dtype)
    B = (torch.randn(1, r, d_out, generator=gen) / 2).to(dtype)
    y0 = torch.randn(N, d_out, generator=gen)
    y, _ = oracle.lora_apply(x, A, B, torch.zeros(N, 1, dtype=torch.int32), y0, 2.0)
    ref = y0.double() + 2.0 * (x.double() @ A[0].double()) @ B[0].double()
    assert torch.allclose(y.double(), ref, rtol=2e-7, atol=2e-7)


def test_apply_topK_uniform_is_dense_sum():
    gen = torch.Generator().manual_seed(22)
    N, d_in, d_out, K, r = 30, 20, 28, 5, 3
    x = torch.randn(N, d_in, generator=gen).to(torch.bfloat16)
    A = (torch.randn(K, d_in, r, generator=gen) / 4).to(torch.bfloat16)
    B = (torch.randn(K, r, d_out, generator=gen) / 2).to(torch.bfloat16)
    y0 = torch.randn(N, d_out, generator=gen)
    ids = torch.stack([torch.randperm(K, generator=gen) for _ in range(N)]).to(torch.int32)
    w = torch.full((N, K), 1.0 / K)
    y, rows = oracle.lora_apply(x, A, B, ids, y0, 1.5, w)
    dense = sum(x.double() @ A[a].double() @ B[a].double() for a in range(K))
    ref = y0.double() + (1.5 * w[0, 0].double()) * dense
    assert torch.allclose(y.double(), ref, rtol=2e-7, atol=2e-7)
    assert rows == N * K


def test_apply_degenerate_cases_leave_base_output():
    wl = workloads.make("tiny_vocab", N=40, d_in=32, d_out=24, r=4)
    ids = torch.randint(0, wl.K, (wl.N, 2), generator=torch.Generator().manual_seed(1), dtype=torch.int32)
    y, _ = oracle.lora_apply(wl.x, wl.A, torch.zeros_like(wl.B), ids, wl.y0, wl.scale)
    assert torch.equal(y, wl.y0)
    y, _ = oracle.lora_apply(wl.x, wl.A, wl.B, ids, wl.y0, wl.scale, torch.zeros(wl.N, 2))
    assert torch.equal(y, wl.y0)
    bad = torch.full((wl.N, 2), -1, dtype=torch.int32)
    bad[::2, 1] = wl.K  # out of range above too
    y, rows = oracle.lora_apply(wl.x, wl.A, wl.B, bad, wl.y0, wl.scale)
    assert torch.equal(y, wl.y0) and rows == 0


def test_per_sequence_golden():
    g = _golden()["per_sequence"]
    args = (torch.tensor(g["x"], dtype=torch.float32), torch.tensor(g["A"], dtype=torch.float32),
            torch.tensor(g["B"], dtype=torch.float32))
    y0 = torch.tensor(g["y0"], dtype=torch.float32)
    adapter_of = torch.tensor(g["adapter_of"])
    y_tok, rows_tok = oracle.lora_apply(*args, adapter_of.reshape(-1, 1), y0, g["scale"])
    y_seq, rows_seq = oracle.per_sequence_apply(*args, adapter_of, y0, g["scale"])
    assert y_tok.tolist() == g["expected_y"] and y_seq.tolist() == g["expected_y"]
    assert rows_tok == g["expected_rows_per_token"] and rows_seq == g["expected_rows_per_sequence"]


@pytest.mark.parametrize("name", ["tiny_vocab", "modality4"])
def test_per_token_equals_K_masked_passes(name):
    wl = workloads.make(name, N=96, d_in=64, d_out=48)
    adapter, _ = oracle.route_vocab(wl.tok, wl.starts)
    y_tok, rows_tok = oracle.lora_apply(wl.x, wl.A, wl.B, adapter.reshape(-1, 1), wl.y0, wl.scale)
    y_seq, rows_seq = oracle.per_sequence_apply(wl.x, wl.A, wl.B, adapter, wl.y0, wl.scale)
    assert torch.equal(y_tok, y_seq)  # masked rows add an exact zero
    assert rows_tok == wl.N and rows_seq == wl.K * wl.N
