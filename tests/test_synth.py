"""The seeded input recipe (CPU)."""
import numpy as np
import torch

import synth


def test_dense_shapes_and_determinism():
    a = synth.make_dense(2, 3, 70, 16, 24, io="bf16", h0_std=0.02, seed=3)
    b = synth.make_dense(2, 3, 70, 16, 24, io="bf16", h0_std=0.02, seed=3)
    c = synth.make_dense(2, 3, 70, 16, 24, io="bf16", h0_std=0.02, seed=4)
    assert a.q.shape == (2, 3, 70, 16) and a.v.shape == (2, 3, 70, 24)
    assert a.h0.shape == (2, 3, 24, 16) and a.log_alpha.shape == (2, 3, 70)
    assert a.q.dtype == torch.bfloat16 and a.beta.dtype == torch.float32
    for x, y in zip(a.tensors().values(), b.tensors().values()):
        assert torch.equal(x, y)
    assert not torch.equal(a.v, c.v)


def test_distributions():
    x = synth.make_dense(1, 4, 4096, 64, 64, io="f32", seed=1)
    n = x.k.norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-5)
    assert (x.beta > 0).all() and (x.beta < 1).all()
    assert (x.log_alpha < 0).all()
    assert abs(float(x.v.mean())) < 0.01 and abs(float(x.v.std()) - 1) < 0.01
    # -0.5 softplus(N(0,1)) has mean about -0.40
    assert abs(float(x.log_alpha.mean()) + 0.40) < 0.02
    y = synth.make_dense(1, 2, 4096, 8, 8, io="f32", decay="slow", seed=1)
    # -softplus(N(-1,1)) has mean about -0.42
    assert abs(float(y.log_alpha.mean()) + 0.42) < 0.03
    assert synth.make_dense(1, 1, 4, 8, 8, seed=0).h0 is None


def test_varlen_recipe():
    lens = synth.varlen_lengths(64, 128, 16384, 5)
    assert lens.min() >= 128 and lens.max() <= 16384 and len(lens) == 64
    assert np.array_equal(lens, synth.varlen_lengths(64, 128, 16384, 5))
    y = synth.make_varlen([3, 0, 5], 2, 8, 16, h0_std=0.02, seed=2)
    assert y.cu_seqlens.tolist() == [0, 3, 3, 8]
    assert y.q.shape == (2, 8, 8) and y.v.shape == (2, 8, 16) and y.h0.shape == (3, 2, 16, 8)
    w = synth.make_workload("gdn_fwd_varlen_n64_h32_dk128_dv256_bf16", H=1, dk=8, dv=8)
    assert int(w.cu_seqlens[-1]) == int(lens.sum())
