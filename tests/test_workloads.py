"""The seeded input generators: storage format and workload structure."""

import numpy as np
import torch

from workloads import (CONFIGS, bf16_bits_to_f32, f32_to_bf16_bits, make_random,
                       make_workload, workload_name)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 65504.0,
                                  1e-30, -3.3e-39], dtype=np.float32)])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_small_fp32_config():
    wl = make_workload("c1")
    assert wl.q.shape == (1, 1, 256, 64) and wl.q.dtype == np.float32
    assert wl.centroids.shape == (1, 4, 64)
    np.testing.assert_allclose(np.linalg.norm(wl.centroids, axis=-1), 1.0, atol=1e-6)
    again = make_workload("c1")
    assert np.array_equal(wl.q, again.q) and np.array_equal(wl.centroids, again.centroids)


def test_mixture_tokens_are_layer_normalised():
    wl = make_workload("c3", H=2, n=512)
    x = wl.q_f32().astype(np.float64)
    assert wl.q.dtype == np.uint16
    np.testing.assert_allclose(x.mean(-1), 0.0, atol=2e-2)
    np.testing.assert_allclose(x.std(-1), 1.0, atol=2e-2)
    assert wl.centroids.shape == (2, 128, 128)
    np.testing.assert_allclose(np.linalg.norm(wl.centroids, axis=-1), 1.0, atol=1e-6)


def test_raster_and_noise_configs_draw():
    wl4 = make_workload("c4", B=1, H=1)
    assert wl4.q.shape == (1, 1, 12288, 64)
    wl5 = make_workload("c5", H=1, n=4096)
    assert wl5.q.shape == (1, 1, 4096, 128)
    assert workload_name("c3") == "mix128_bf16_b1h8_n8192_d128_k128_w64"
    for cid, c in CONFIGS.items():
        assert c["k"] * c["w"] == c["n"], cid


def test_random_free_shape():
    wl = make_random(2, 3, 77, 64, 5, 9, dtype="bf16", seed=3)
    assert wl.q.shape == (2, 3, 77, 64) and wl.centroids.shape == (3, 5, 64)
