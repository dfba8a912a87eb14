"""The five workload configurations, table-driven: every parameter of each
configuration as the workload list states it, and a GPU parity test that runs
each one at its full size.  An empty or incomplete table fails."""
from __future__ import annotations

import os
import re

import pytest

import gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name: (layers, d_model, q heads, kv heads, head_dim, SwiGLU hidden, vocab, weight / KV dtype,
#        KV capacity, rows, KV layout, page size, page pool, RoPE theta, fixed positions)
TABLE = {
    "tiny": (2, 64, 4, 4, 16, 128, 256, "f32", 64, 1, "contiguous", None, None, 1e4, ()),
    "1b": (16, 2048, 32, 8, 64, 8192, 32000, "bf16", 4096, 1, "contiguous", None, None, 5e5, ()),
    "8b": (32, 4096, 32, 8, 128, 14336, 128256, "bf16", 8192, 1, "contiguous", None, None, 5e5,
           (1, 1024, 4096, 8191)),
    "8b_paged": (32, 4096, 32, 8, 128, 14336, 128256, "bf16", 8192, 8, "paged", 16, 4096, 5e5, ()),
    "1b_long": (16, 2048, 32, 8, 64, 8192, 32000, "bf16", 32768, 4, "contiguous", None, None, 5e5,
                (100, 8000, 20000, 32767)),
}

# the GPU test that runs each configuration at its full size
FULL_SIZE_TESTS = {
    "tiny": ("test_parity_gpu.py", "test_tiny_prompt_then_greedy"),
    "1b": ("test_parity_gpu.py", "test_1b_prompt_then_greedy"),
    "8b": ("test_parity_gpu.py", "test_8b_decode_at_prefilled_positions"),
    "8b_paged": ("test_rows_tc_gpu.py", "test_8b_paged_rows8_prefilled"),
    "1b_long": ("test_parity_gpu.py", "test_1b_long_cap_rows4"),
}


def test_table_is_complete():
    assert len(TABLE) == 5 and set(TABLE) == set(FULL_SIZE_TESTS)
    assert set(TABLE) <= set(gen.WORKLOADS)


@pytest.mark.parametrize("name", sorted(TABLE))
def test_workload_matches_its_configuration(name):
    L, d, hq, hkv, hd, F, V, dt, cap, rows, layout, page, pool, theta, positions = TABLE[name]
    wl = gen.WORKLOADS[name]
    assert (wl.n_layers, wl.d_model, wl.n_heads, wl.n_kv_heads, wl.head_dim) == (L, d, hq, hkv, hd)
    assert (wl.ffn_hidden, wl.vocab, wl.wdtype, wl.kvdtype) == (F, V, dt, dt)
    assert (wl.cap, wl.rows, wl.layout) == (cap, rows, layout)
    if layout == "paged":
        assert (wl.page_size, wl.num_pages) == (page, pool)
        assert wl.num_pages * wl.page_size >= wl.rows * wl.cap
    assert wl.rms_eps == 1e-5 and wl.rope_theta == theta
    assert tuple(wl.positions) == positions
    assert wl.gain_sigma == 0.0      # gains 1; only the tiny_gain variant draws them


@pytest.mark.parametrize("name", sorted(FULL_SIZE_TESTS))
def test_each_configuration_has_a_full_size_gpu_parity_test(name):
    fname, test = FULL_SIZE_TESTS[name]
    src = open(os.path.join(ROOT, "tests", fname)).read()
    # the test with its decorators (a parametrize list may name the workload)
    m = re.search(rf"((?:^@[^\n]*\n)*)^def {test}\(.*?(?=^@|^def |\Z)", src, flags=re.S | re.M)
    assert m, f"{fname}::{test} is missing"
    body = m.group(0)
    # the test takes the named workload whole (no replace() that shrinks it)
    assert re.search(rf"WORKLOADS\[\"{name}\"\]", body) or re.search(rf"\"{name}\"", body), body[:300]
    assert ".replace(" not in body, f"{test} shrinks the {name} workload"
    # it is a GPU test: its file marks every test gpu
    assert "pytestmark = pytest.mark.gpu" in src
