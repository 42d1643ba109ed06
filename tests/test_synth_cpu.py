"""The seeded input generator that feeds both the oracle and the GPU path:
determinism, bf16 rounding, and the recipe's stated structure (unit-RMS
locality field, hot key tiles with strength s_h, per-head strength range of
the skewed workload, the extra tensors of backward and low-rank workloads)."""
import numpy as np
import pytest
import torch

import synth


def _small(**over):
    base = dict(name="synth-test", B=2, H=3, d=32, T=4, Y=8, X=8, ta=2, tb=4, tc=4, dtype="bf16",
                estimator="mean", top_p=0.9, k_floor=2, P=2, n_hot=3, skew=False, backward=False, seed=11)
    base.update(over)
    return synth.Workload(**base)


def test_same_seed_same_tensors_other_seed_other_tensors():
    wl = synth.WORKLOADS["tiny"]
    a, b = synth.make(wl), synth.make(wl)
    for key in ("q", "k", "v", "hot", "strength"):
        assert np.array_equal(a[key], b[key]), key
    c = synth.make(_small(seed=12))
    d = synth.make(_small(seed=13))
    assert not np.array_equal(c["q"], d["q"])


def test_round_bf16_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    # exact halfway cases between neighbouring bf16 values: ties go to the even one
    halfway = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3 + 2.0 ** -7], dtype=np.float32)
    for arr in (x, halfway):
        ours = synth.round_bf16(arr.copy())
        ref = torch.from_numpy(arr.copy()).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(ours, ref)
    assert synth.round_bf16(halfway.copy()).tolist() == [1.0, 1.015625, -1.0, 3.0]


def test_bf16_workloads_hold_bf16_values_and_shapes():
    wl = _small(backward=True, estimator="lowrank")
    data = synth.make(wl)
    shape = (wl.B, wl.N, wl.H, wl.d)
    for key in ("q", "k", "v", "do"):
        x = data[key]
        assert x.shape == shape and x.dtype == np.float32
        assert not (x.view(np.uint32) & np.uint32(0xFFFF)).any(), key   # exactly representable in bf16
    assert data["wq"].shape == data["wk"].shape == (wl.H, wl.d, wl.rank)
    assert "do" not in synth.make(_small())
    assert "wq" not in synth.make(_small())


def test_locality_field_has_unit_rms_and_hot_tiles_carry_the_query_direction():
    # without the N(0, I) noise: Q = F + u, K = F (+ 2 s_h u on the hot tiles)
    wl = _small(H=8, d=64, n_hot=2)
    data = synth.make(wl, with_noise=False)
    q, k = data["q"].astype(np.float64), data["k"].astype(np.float64)
    hot = data["hot"]
    assert hot.shape == (wl.B, wl.H, wl.n_hot)
    nT, nY, nX = wl.tiles
    rms = []
    for b in range(wl.B):
        for h in range(wl.H):
            assert len(set(hot[b, h].tolist())) == wl.n_hot and hot[b, h].min() >= 0 and hot[b, h].max() < wl.nb
            mask = np.zeros((wl.T, wl.Y, wl.X), bool)
            for tid in hot[b, h]:
                bt, rem = divmod(int(tid), nY * nX)
                by, bx = divmod(rem, nX)
                mask[bt * wl.ta:(bt + 1) * wl.ta, by * wl.tb:(by + 1) * wl.tb, bx * wl.tc:(bx + 1) * wl.tc] = True
            mask = mask.ravel()
            u = q[b, :, h, :] - k[b, :, h, :]          # on the cold tokens: u exactly (up to bf16)
            u0 = u[~mask][0]
            assert np.allclose(u[~mask], u0, atol=0.02)
            # hot tokens: K - F = 2 s_h u with s_h = 1 here, so Q - K = -u
            assert np.allclose(u[mask], -u0, atol=0.02)
            field = k[b, ~mask, h, :]
            rms.append(np.mean(np.sum(field ** 2, axis=1)))
    # E|F|^2 = 8 features x E|c|^2 (1/4) x E cos^2 (1/2) = 1, averaged over heads
    assert 0.75 < float(np.mean(rms)) < 1.25


def test_skewed_strength_is_log_uniform_in_its_range():
    wl = _small(skew=True, H=16, seed=21)
    data = synth.make(wl, with_noise=False)
    s = data["strength"]
    assert s.shape == (wl.B, wl.H)
    assert (s >= 0.25).all() and (s <= 8.0).all()
    assert s.max() / s.min() > 4.0          # spread over the range, not a constant
    assert np.array_equal(synth.make(_small())["strength"], np.ones((2, 3)))


@pytest.mark.parametrize("name", ["wan", "skewed", "training"])
def test_named_workloads_tile_their_grids(name):
    wl = synth.WORKLOADS[name]
    assert wl.T % wl.ta == 0 and wl.Y % wl.tb == 0 and wl.X % wl.tc == 0
    assert wl.nb == int(np.prod(wl.tiles)) and wl.N == wl.nb * wl.Bt
    assert wl.n_hot <= wl.nb
