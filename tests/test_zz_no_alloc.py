"""The allocation-free attention entry point (dec_attention_static).

Some callers cannot allocate device memory where they run attention: a serving
process that reserved its whole device-memory budget up front, or a loop whose
latency cannot absorb cudaMalloc / cudaFree (which may synchronise the whole
device).  dec_attention_static keeps its split scratch in a fixed array inside
the library instead.  It must give the same results as dec_attention, which
uses the handle's workspace, call after call: the array keeps the previous
call's contents, so a second call in a row checks that nothing stale leaks into
the result.  After its first call on a device (which resolves the array's
address and may load the library's module), it must not change the device's
free memory.  A shape whose scratch exceeds the array is refused and leaves the
handle usable.  This file is collected last.
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
    outs = [torch.full((rows, wl.q_dim), float("nan"), dtype=torch.float32, device="cuda:0") for _ in range(3)]
    torch.cuda.synchronize()
    free_after_first = None
    for call in range(3):
        dec._after_torch()
        rc = B.dec_attention_static(dec.h, 1, qkv.data_ptr(), pos.data_ptr(), outs[call].data_ptr())
        assert rc == B.DEC_OK, B.last_error(dec.h)
        torch.cuda.synchronize()
        free_now = torch.cuda.mem_get_info()[0]
        if call == 0:
            free_after_first = free_now
        else:
            assert free_now == free_after_first, "dec_attention_static changed the device's free memory"
        got = outs[call].cpu().numpy()
        for r in range(rows):
            assert_close(got[r], ref_h[r], wl, f"static-scratch attention, call {call}, row {r}")
    dec.close()


def test_static_scratch_refuses_a_shape_beyond_the_array():
    """8 rows x 192 kv heads need 1536 split-completion counters, more than the
    array's 1024: refused with DEC_E_UNSUPPORTED before any device work; the
    handle then runs dec_attention as before."""
    import torch
    from graph_replay_gb300 import _binding as B

    wl = gen.WORKLOADS["1b"].replace(name="noalloc_wide", n_layers=1, d_model=1024, n_heads=192, n_kv_heads=192,
                                     head_dim=64, ffn_hidden=1024, vocab=256, cap=64, rows=8)
    dec, _ = make_decoder(wl)
    qkv = torch.from_numpy(gen.normal(wl.seed, 92, (wl.rows, wl.q_dim + 2 * wl.kv_dim), sigma=1.0,
                                      dtype="f32")).cuda()
    pos = torch.arange(wl.rows, dtype=torch.int32, device="cuda:0")
    out = torch.zeros(wl.rows, wl.q_dim, dtype=torch.float32, device="cuda:0")
    dec._after_torch()
    rc = B.dec_attention_static(dec.h, 0, qkv.data_ptr(), pos.data_ptr(), out.data_ptr())
    assert rc == B.DEC_E_UNSUPPORTED
    assert "fixed" in B.last_error(dec.h)
    assert dec.stats()["state"] == 0
    assert torch.count_nonzero(out).item() == 0        # nothing was written
    dec.attention(0, qkv, pos, out)                    # the handle still works
    assert torch.isfinite(out).all().item()
    dec.close()
