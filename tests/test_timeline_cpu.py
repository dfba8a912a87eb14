"""Host arithmetic of bench.py's phase timeline: per-phase durations, rates and
spreads from the in-kernel %globaltimer stamps, on stamps written by hand."""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_phase_bytes_of_the_8b_shape():
    import bench
    import gen
    wl = gen.WORKLOADS["8b"]
    nb = bench.phase_bytes(wl)
    assert nb["qkv"] == (4096 + 2 * 1024) * 4096 * 2
    assert nb["attn"] == 2 * 8192 * 1024 * 2
    assert nb["gu"] == 2 * 14336 * 4096 * 2
    assert nb["head"] == 128256 * 4096 * 2
    # one step's algorithmic bytes = every phase once per layer + embedding row + gains
    per_layer = sum(nb[k] for k in bench.PHASES)
    gains = (2 * wl.n_layers + 1) * wl.d_model * 2
    assert wl.step_bytes() == wl.n_layers * per_layer + nb["head"] + wl.d_model * 2 + gains


def test_summary_of_hand_written_stamps():
    import bench
    import gen
    wl = gen.WORKLOADS["8b"].replace(name="8b_one_layer", n_layers=1)
    # phases: embed, qkv, attn, o, gu, down, head; stamps in ns:
    # [earliest start, latest past wait, earliest end, latest end]
    us = np.array([[0, 0, 1, 2],
                   [1, 3, 10, 12],       # qkv ends 10 us after embed's last end
                   [11, 13, 20, 21],     # attn: 9 us, spread 1, wait latency 1
                   [20, 22, 29, 30],
                   [29, 31, 60, 65],     # gu: 35 us, spread 5
                   [60, 66, 80, 85],
                   [80, 86, 230, 235]], dtype=np.float64)
    stamps = (us * 1e3 + 5e9).astype(np.uint64)    # absolute ns, arbitrary origin
    s = bench.summarize_timeline(stamps, wl)
    nb = bench.phase_bytes(wl)
    assert s["qkv"]["us_mean"] == 10.0 and s["qkv"]["wait_latency_us"] == 1.0
    assert s["attn"]["us_mean"] == 9.0 and s["attn"]["end_spread_us"] == 1.0
    assert s["gu"]["us_mean"] == 35.0 and s["gu"]["end_spread_us"] == 5.0
    assert s["head"]["us_mean"] == 150.0 and s["head"]["phases"] == 1
    assert abs(s["gu"]["gbs"] - nb["gu"] / 35e-6 / 1e9) < 0.1
    assert s["span_us"] == 235.0
    assert sum(s[k]["us_total"] for k in bench.PHASES + ("head",)) == 235.0 - 2.0
