"""The seeded input generators (CPU): deterministic, shaped as stated, and drawing the
modality shares asked for.  They hold no method arithmetic; these checks only make sure
the inputs the parity tests and the benchmark consume are the ones described."""

import torch

import workloads


def test_same_seed_same_inputs_and_different_seed_differs():
    a, b = workloads.make("modality4", N=300, d_in=256), workloads.make("modality4", N=300, d_in=256)
    assert torch.equal(a.tok, b.tok) and torch.equal(a.x, b.x) and torch.equal(a.A, b.A)
    c = workloads.make("modality4", seed=99, N=300, d_in=256)
    assert not torch.equal(a.x, c.x)


def test_shapes_and_dtypes_follow_the_workloads():
    for name in workloads.WORKLOADS:
        wl = workloads.make(name, N=64, d_in=256, d_out=384)
        assert wl.x.shape == (64, 256) and wl.y0.shape == (64, 384) and wl.y0.dtype == torch.float32
        assert wl.A.shape == (wl.K, 256, wl.r) and wl.B.shape == (wl.K, wl.r, 384)
        assert wl.A.dtype == wl.x.dtype == wl.B.dtype
        if wl.routing == "vocab":
            assert wl.tok.shape == (64,) and wl.starts.shape == (wl.K + 1,)
            assert bool((wl.tok >= 0).all() and (wl.tok < workloads.VOCAB).all())
        else:
            assert wl.W1.shape == (256, workloads.ROUTER_HIDDEN) and wl.W2.shape == (workloads.ROUTER_HIDDEN, wl.K)


def modality_of(wl):
    return torch.bucketize(wl.tok.long(), wl.starts.long(), right=True) - 1


def test_runs_have_one_modality_and_geometric_mean_length():
    wl = workloads.make("modality4", N=20000, d_in=64, d_out=64)
    m = modality_of(wl)
    changes = int((m[1:] != m[:-1]).sum())
    # runs of mean 64 with a uniform modality per run: a new run keeps the previous
    # modality with probability 1/4, so modality changes come about every 64 / (3/4) tokens
    assert 20000 / (changes + 1) > 40 and 20000 / (changes + 1) < 140


def test_skewed_shares_are_drawn_per_run():
    for dist, top in (("80-10-5-5", 0.8), ("95-2-2-1", 0.95), ("70-10-10-10", 0.7)):
        wl = workloads.make("modality4", N=60000, d_in=64, d_out=64, dist=dist)
        share = torch.bincount(modality_of(wl), minlength=4).double() / wl.N
        assert abs(share[0].item() - top) < 0.12, (dist, share.tolist())
        assert share[0] == share.max()


def test_zipf_prefers_low_ranks():
    wl = workloads.make("decode_sweep", N=20000, K=8, d_in=64, d_out=64, dist="zipf")
    counts = torch.bincount(modality_of(wl), minlength=8)
    assert counts[0] > counts[1] > counts[3] > counts[7]
