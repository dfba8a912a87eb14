"""The seeded input generator: determinism, stream independence, distribution."""
import numpy as np
from scipy.special import ndtri

import gen


def test_quantile_table_matches_library_inverse_cdf():
    k = np.arange(0, 65536, 97)
    q = np.array([gen.quantile(int(i)) for i in k])
    ref = ndtri((k + 0.5) / 65536.0)
    assert np.abs(q - ref).max() < 1e-9
    # exact symmetry
    assert all(gen.quantile(i) == -gen.quantile(65535 - i) for i in (0, 1, 1000, 32767))


def test_counter_based_slices_agree():
    full = gen.normal(5, 6, (1000,), sigma=0.02, dtype="bf16")
    part = gen.normal(5, 6, (100,), sigma=0.02, dtype="bf16", offset=450)
    assert np.array_equal(full[450:550], part)
    assert np.array_equal(full, gen.normal(5, 6, (1000,), sigma=0.02, dtype="bf16"))
    assert not np.array_equal(full, gen.normal(5, 7, (1000,), sigma=0.02, dtype="bf16"))
    assert not np.array_equal(full, gen.normal(4, 6, (1000,), sigma=0.02, dtype="bf16"))


def test_normal_moments():
    a = gen.normal(1, 2, (1 << 20,), sigma=0.02, dtype="f32").astype(np.float64)
    assert abs(a.mean()) < 1e-4
    assert abs(a.std() - 0.02) < 2e-4
    b = gen.bf16_bits_to_f32(gen.normal(1, 3, (1 << 20,), sigma=1.0, dtype="bf16")).astype(np.float64)
    assert abs(b.std() - 1.0) < 5e-3
    kurt = np.mean(b ** 4) / np.mean(b ** 2) ** 2
    assert abs(kurt - 3.0) < 0.05


def test_ints_and_permutation():
    t = gen.ints(9, 1, 0, 256, 100000)
    assert t.min() >= 0 and t.max() < 256
    counts = np.bincount(t, minlength=256)
    assert counts.min() > 300
    p = gen.permutation(9, 2, 4096)
    assert np.array_equal(np.sort(p), np.arange(4096))


def test_workload_recipes():
    wl = gen.WORKLOADS["8b_paged"]
    sm = gen.slot_map(wl)
    assert sm.shape == (8, 512)
    assert np.array_equal(np.sort(sm.ravel()), np.arange(4096))
    pos = gen.row_positions(wl)
    assert pos.shape == (8,) and pos.min() >= 0 and pos.max() < wl.cap
    assert list(gen.row_positions(gen.WORKLOADS["1b_long"])) == [100, 8000, 20000, 32767]
    # roofline byte counts quoted for the 8B-shape step
    wl3 = gen.WORKLOADS["8b"]
    assert abs(wl3.kv_swept_bytes() - 1.074e9) < 1e6
    assert abs(wl3.weight_bytes() - 15.01e9) < 1e7
    kv = gen.kv_prefill(gen.WORKLOADS["tiny"], 1, 0, 0, 10)
    kv2 = gen.kv_prefill(gen.WORKLOADS["tiny"], 1, 0, 0, 4, start=6)
    assert np.array_equal(kv[6:], kv2)
