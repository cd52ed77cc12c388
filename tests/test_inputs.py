"""The seeded synthetic generators: deterministic, correctly rounded to bf16, and shaped as the
workloads they stand in for."""
import numpy as np
import torch

from verified_kv_cache_poissoncomp_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 65504.0, 1e-30, 3.0e38], np.float32)])
    want = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(I.f32_to_bf16(x), want)
    back = torch.tensor(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(I.bf16_to_f32(I.f32_to_bf16(x)), back)


def test_tiny_is_deterministic_and_shaped():
    a, b = I.tiny(), I.tiny()
    assert a.kv.shape == (1, 1, 1, 1024, 2, 64) and a.queries.shape == (16, 1, 4, 64)
    for f in ["tau", "kv", "queries", "plant_pos"]:
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert a.tau.dtype == np.float32 and np.all(a.tau > 0) and np.all(a.tau <= 1)
    assert a.planted.sum() == 8
    c = I.tiny(data_seed=99)
    assert not np.array_equal(a.kv, c.kv)


def test_planted_keys_have_the_smallest_importance():
    w = I.make_workload("t", B=1, L=2, h_kv=2, G=4, d=64, n=4096, eta=1 / 16, n_local=128,
                        n_queries=8)
    for l in range(2):
        for h in range(2):
            t = w.tau[0, l, h]
            for p in w.plant_pos[0, l, h]:
                assert t[p] == t.min()
    assert list(w.query_layer) == [0, 1, 0, 1, 0, 1, 0, 1]
    assert w.planted.tolist() == [False, False, False, True] * 2
