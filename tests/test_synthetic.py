"""Host-side checks of the seeded input generators (shapes, determinism, recipe)."""

import numpy as np
import torch

from post_weight_quantization_03_gb300 import synthetic as S


def test_deterministic_and_prefix():
    spec = S.ActivationSpec(d_in=64, n_tok=6144, dtype="f16", n_dead=3, n_outlier=2, seed=7)
    a = S.activations(spec)
    b = S.activations(spec)
    assert a.shape == (6144, 64) and a.dtype == torch.float16
    assert torch.equal(a, b)
    # the first 2048-token chunk of a long draw is a short draw
    c = S.activations(spec, n_tok=2048)
    assert torch.equal(a[:2048], c)
    # tokens [2048, 4096) can be drawn on their own
    d = S.activations(spec, n_tok=2048, tok_start=2048)
    assert torch.equal(a[2048:4096], d)


def test_dead_and_outlier_channels():
    spec = S.ActivationSpec(d_in=128, n_tok=2048, dtype="f32", n_dead=5, n_outlier=4, seed=9)
    X = S.activations(spec).numpy()
    dead, outl = S.channel_roles(spec)
    assert np.all(X[:, dead.numpy()] == 0)
    live = np.setdiff1d(np.arange(128), np.concatenate([dead.numpy(), outl.numpy()]))
    ratio = X[:, outl.numpy()].std() / X[:, live].std()
    assert 12 < ratio < 30
    assert np.count_nonzero(X.std(axis=0) == 0) == 5


def test_relu_t4_sparsity():
    spec = S.ActivationSpec(d_in=256, n_tok=4096, dtype="f16", relu_t4=True, seed=11)
    X = S.activations(spec).float().numpy()
    zero_frac = np.mean(X == 0)
    assert 0.57 < zero_frac < 0.63
    assert X.min() >= 0


def test_correlated_channels():
    spec = S.ActivationSpec(d_in=64, n_tok=4096, dtype="f32", seed=3)
    X = S.activations(spec).numpy().astype(np.float64)
    C = np.corrcoef(X.T)
    off = np.abs(C[~np.eye(64, dtype=bool)])
    assert off.mean() > 0.05          # mixing correlates the channels


def test_weights_recipe():
    W = S.weights(300, 200, 0.02, "bf16", 5)
    assert W.dtype == torch.bfloat16 and W.shape == (300, 200)
    assert abs(W.float().std().item() - 0.02) < 0.001
    assert torch.equal(W, S.weights(300, 200, 0.02, "bf16", 5))


def test_workload_table():
    w = S.WORKLOADS
    assert set(w) == {"layer256_n512", "layer4096_n262144", "mlp11008_n131072",
                      "block7b_n131072", "downproj28672_n65536"}
    l = w["layer4096_n262144"].layers[0]
    assert (l.d_out, l.act.d_in, l.act.n_tok, l.act.n_dead, l.act.n_outlier) == \
        (4096, 4096, 262144, 41, 8)
    assert len(w["block7b_n131072"].layers) == 7 and w["block7b_n131072"].bits == (3, 4)
