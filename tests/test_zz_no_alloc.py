"""The allocation-free attention entry point (dec_attention_static).

Callers that cannot allocate device memory where they run attention (inside a
stream capture, on a fixed memory budget, or where cudaMalloc's implicit device
synchronisation is not acceptable) use dec_attention_static, which keeps its
split scratch in a fixed array inside the library.  It must give the same
results as dec_attention, which uses the handle's workspace, call after call:
the array keeps the previous call's contents, so a second call in a row checks
that nothing stale leaks into the result.  This file is collected last.
"""
import numpy as np
import pytest

import gen
from _harness import assert_close, make_decoder

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name, rows", [("1b", 2), ("8b", 1)])
def test_static_scratch_attention_matches_workspace_attention(name, rows):
    import torch
    from graph_replay_gb300 import _binding as B
    from gen.device import place_kv

    wl = gen.WORKLOADS[name].replace(name=f"{name}_noalloc", n_layers=2, vocab=1024, cap=4096, rows=rows)
    dec, _ = make_decoder(wl)
    positions = [3000, 1234][:rows]
    for r in range(rows):
        for which in (0, 1):
            place_kv(dec.kv(1, which), gen.kv_prefill(wl, 1, which, r, positions[r]), r)
    qkv = torch.from_numpy(gen.normal(wl.seed, 91, (rows, wl.q_dim + 2 * wl.kv_dim), sigma=1.0,
                                      dtype="f32")).cuda()
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda:0")
    ref = torch.empty(rows, wl.q_dim, dtype=torch.float32, device="cuda:0")
    dec.attention(1, qkv, pos, ref)   # existing entry point: scratch in the workspace
    ref_h = ref.cpu().numpy()
    for call in range(2):
        out = torch.full((rows, wl.q_dim), float("nan"), dtype=torch.float32, device="cuda:0")
        dec._after_torch()
        rc = B.dec_attention_static(dec.h, 1, qkv.data_ptr(), pos.data_ptr(), out.data_ptr())
        assert rc == B.DEC_OK, B.last_error(dec.h)
        got = out.cpu().numpy()
        for r in range(rows):
            assert_close(got[r], ref_h[r], wl, f"static-scratch attention, call {call}, row {r}")
    dec.close()
