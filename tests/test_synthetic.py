"""The seeded input generators (no GPU): the recipe the design states for the
synthetic stand-ins of the pages' Llama-2 workloads, pinned here so that the
parity tests, the full-size tests and the bench all see the inputs it
describes."""
import numpy as np

import synthetic


def test_workloads_match_their_description():
    counts = {w.name: len(w.cases()) for w in synthetic.WORKLOADS}
    assert counts == {"single-4096x4096-m1": 1, "llama2-7b-decode": 16, "llama2-13b-mid": 16,
                      "llama2-7b-prefill": 8, "llama2-70b-sweep": 40}
    # the 70B sweep runs every layer with g = 128 and with one group per column
    groups = {(layer, g) for (layer, M, K, N, g) in synthetic.workload(4).cases()}
    assert ("down", 128) in groups and ("down", 28672) in groups
    # only the prefill workload has outlier channels
    assert [w.outliers for w in synthetic.WORKLOADS] == [False, False, False, True, False]
    # every shape fits the packed format: N % 16, K % 64, K % group
    for w in synthetic.WORKLOADS:
        for (layer, M, K, N, g) in w.cases():
            assert N % 16 == 0 and K % 64 == 0 and K % g == 0


def test_weights_are_seeded_normal():
    a = synthetic.weights(1, 512, 256)
    b = synthetic.weights(1, 512, 256)
    assert a.dtype == np.float32 and a.shape == (512, 256) and np.array_equal(a, b)
    assert not np.array_equal(a, synthetic.weights(2, 512, 256))   # depends on the workload
    assert abs(float(a.mean())) < 2e-4 and abs(float(a.std()) - 0.02) < 5e-4


def test_activations_and_outlier_channels():
    for K in (4096, 11008):
        A = synthetic.activations(3, 64, K, 12288, outliers=True).astype(np.float64)
        plain = synthetic.activations(3, 64, K, 12288, outliers=False).astype(np.float64)
        assert A.dtype == np.float64 and A.shape == (64, K)
        # round(0.01 K) whole columns are 20x larger (the same draws otherwise)
        big = np.where(np.abs(A).max(axis=0) > 6.5)[0]
        ratio = np.abs(A).mean(axis=0) / np.abs(plain).mean(axis=0)
        scaled = np.where(ratio > 10)[0]
        assert len(scaled) == round(0.01 * K)
        assert set(big) <= set(scaled)
        assert np.allclose(ratio[scaled], 20, rtol=2e-3)
        assert np.allclose(ratio[np.setdiff1d(np.arange(K), scaled)], 1, rtol=2e-3)
    a = synthetic.activations(1, 16, 4096, 4096)
    assert a.dtype == np.float16 and abs(float(a.astype(np.float64).std()) - 1) < 0.02


def test_sample_indices():
    s = synthetic.sample_indices(22016, 24, seed=1, salt=7)
    assert len(s) == 24 and len(set(s)) == 24 and np.all(np.diff(s) > 0)
    assert s.min() >= 0 and s.max() < 22016
    assert np.array_equal(s, synthetic.sample_indices(22016, 24, seed=1, salt=7))
    assert len(synthetic.sample_indices(10, 50, seed=0, salt=0)) == 10


def test_random_codes_cover_every_nibble():
    q, s, z = synthetic.random_codes(256, 64, 128, seed=3)
    assert set(np.unique(q)) == set(range(16)) and set(np.unique(z)) == set(range(16))
    sv = s.view(np.float16).astype(np.float64)
    assert np.all(sv >= 2.0 ** -10) and np.all(sv <= 2.0 ** -4)
