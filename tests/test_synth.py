"""The synthetic generator's two implementations agree bit for bit: the
tensor path (what fills device buffers) and the host C path (what the CPU
side of every parity check regenerates inputs with)."""
import numpy as np
import pytest
import torch

import synth
from synth import workloads as W

RECIPES = [W.WEIGHT_RECIPE, W.GRAD_NORMAL, W.GRAD_T3_OUTLIERS, W.MOMENT_M_RECIPE,
           W.MOMENT_V_RECIPE,
           synth.Recipe(synth.Dist("normal", 1e-3), outlier_block=64, outlier_prob=0.05,
                        outlier_factor=100.0)]


def _torch_fill(recipe, seed, stream, start, count):
    out = torch.empty(count, dtype=torch.bfloat16)
    return synth.bf16_to_u16(synth._fill_torch(recipe, seed, stream, start, count, out, 1 << 20))


def test_host_generator_builds():
    assert synth._host_lib() is not None


@pytest.mark.parametrize("recipe", RECIPES, ids=lambda r: f"{r.dist.kind}-{r.outlier_block}")
@pytest.mark.parametrize("start,count", [(0, 1 << 16), (12345, 70001),
                                         ((1 << 32) - 3000, 7000),     # crosses 2^32
                                         (7 * 10 ** 9 - 5000, 5000)])
def test_host_fill_equals_tensor_path(recipe, start, count):
    for seed, stream in [(0, synth.WEIGHTS), (3, synth.grad_stream(5)),
                         (17, synth.grad_stream(127, 2))]:
        want = _torch_fill(recipe, seed, stream, start, count)
        got = synth.fill_u16(recipe, seed, stream, start, count)
        assert np.array_equal(got, want), (recipe, seed, stream, start)
        # the CPU tensor API goes through the same host path
        assert np.array_equal(synth.bf16_to_u16(synth.fill(recipe, seed, stream, start, count)),
                              want)


@pytest.mark.parametrize("recipe", RECIPES, ids=lambda r: f"{r.dist.kind}-{r.outlier_block}")
def test_host_at_equals_tensor_path(recipe):
    rng = np.random.default_rng(1)
    idx = np.concatenate([rng.integers(0, 1 << 40, 5000), np.arange(1 << 32, (1 << 32) + 300),
                          rng.integers(0, 4096, 3000)])
    want = synth.bf16_to_u16(synth._values_at(recipe, 2, synth.grad_stream(3),
                                              torch.from_numpy(idx.copy())))
    assert np.array_equal(synth.at_u16(recipe, 2, synth.grad_stream(3), idx), want)
    assert np.array_equal(synth.bf16_to_u16(synth.at(recipe, 2, synth.grad_stream(3), idx)), want)


def test_outliers_are_one_element_of_a_picked_block():
    r = synth.Recipe(synth.Dist("normal", 1e-3), outlier_block=256, outlier_prob=0.01,
                     outlier_factor=100.0)
    n = 1 << 22
    plain = synth.fill_u16(synth.Recipe(r.dist), 0, 9, 0, n)
    boosted = synth.fill_u16(r, 0, 9, 0, n)
    diff = np.flatnonzero(plain != boosted)
    blocks = diff // 256
    assert np.unique(blocks).size == blocks.size          # at most one element a block
    assert 0.5 * 0.01 * n / 256 < blocks.size < 1.5 * 0.01 * n / 256
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32)
    assert np.allclose(f(boosted[diff]), 100.0 * f(plain[diff]), rtol=2 ** -8)
