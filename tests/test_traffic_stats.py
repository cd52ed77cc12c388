"""Host-side traffic statistics of the tolerance sweep (bench.py) on hand-made inputs."""
import numpy as np

import bench


def test_traffic_stats_on_a_hand_made_case():
    n = 1000
    st = np.zeros((2, 4, 16), dtype=np.int32)
    # query 0: heads 0, 1 certified; heads 2, 3 fetch 100 and 50 rows
    st[0, :2, 10] = 1
    st[0, 2, 13], st[0, 3, 13] = 100, 50
    # query 1: every head fetches 10 rows
    st[1, :, 13] = 10
    fetched = np.array([[120, 0], [30, 10]])        # per KV head
    counts = np.array([60, 70, 80, 90])             # |H u S| per unit
    s = bench.traffic_stats(st, fetched, counts, n)
    assert s["decisions_fetching_frac"] == 6 / 8
    assert np.isclose(s["context_frac_per_fetching_decision"], (100 + 50 + 4 * 10) / 6 / n)
    assert np.isclose(s["resident_frac"], 75 / n)
    assert np.isclose(s["overall_read_frac"], 75 / n + (150 + 40) / 8 / n)
    assert np.isclose(s["kv_head_transfer_frac"], 160 / 4 / n)
    assert s["shortlist_exhausted_frac"] == 0.0
    st[1, 0, 15] = 4
    assert bench.traffic_stats(st, fetched, counts, n)["shortlist_exhausted_frac"] == 1 / 8


def test_estimator_bytes_on_a_hand_made_case():
    # two units: 3 rows (one sampled) and 2 rows (both sampled); rows past the count are ignored
    r = np.array([[1.0, 0.5, 1.0, 0.1], [0.2, 0.3, 0.9, 0.9]], dtype=np.float32)
    count = np.array([3, 2])
    nbytes, n_l = bench.estimator_bytes(count, r, d=128, G=4)
    assert n_l == 3
    assert nbytes == 5 * (4 * 128 + 8)
    # with a 2-bit sketch each sampled row also reads the sketch logit of its 4 query heads
    nbytes, n_l = bench.estimator_bytes(count, r, d=128, G=4, sketch_logits=True)
    assert nbytes == 5 * (4 * 128 + 8) + 3 * 4 * 4
