"""Failure handling on the GPU without faulting it ("Execution", section
"Failure handling"): host range checks, device-side checks that set the error
word (injected through the device slot record, which skips the host checks),
the needs-reset state, and the bounded wait that poisons the handle."""
import ctypes

import numpy as np
import pytest

import gen
import oracle
from _harness import assert_close, make_decoder

pytestmark = pytest.mark.gpu


def _slots(dec, tokens, pos, wmap=None):
    import torch
    wmap = [0] * dec.rows if wmap is None else wmap
    return torch.tensor(list(tokens) + list(pos) + list(wmap), dtype=torch.int32, device="cuda:0")


def test_host_range_checks_refuse_before_launch():
    from graph_replay_gb300 import _binding as B
    wl = gen.WORKLOADS["tiny"]
    dec, mw = make_decoder(wl)
    for toks, pos in (([wl.vocab], [0]), ([-1], [0]), ([0], [wl.cap]), ([0], [-1])):
        with pytest.raises(B.DecError) as ei:
            dec.step(toks, pos)
        assert ei.value.status == B.DEC_E_RANGE
    assert dec.stats()["replays"] == 0
    res = dec.step([3], [0])          # the handle is still ready
    ref = oracle.Oracle(mw, cap=wl.cap).step(0, 3, 0)
    assert_close(res.logits[0], ref, wl)
    dec.close()


@pytest.mark.parametrize("bad, bit", [("token", 0x1), ("pos", 0x2)])
def test_device_check_sets_error_word_and_needs_reset(bad, bit):
    from graph_replay_gb300 import _binding as B
    wl = gen.WORKLOADS["tiny"]
    dec, mw = make_decoder(wl)
    dec.step([7], [0])
    tok, pos = ([wl.vocab + 3], [1]) if bad == "token" else ([7], [wl.cap + 5])
    dec.launch(_slots(dec, tok, pos))
    with pytest.raises(B.DecError) as ei:
        dec.wait()
    assert ei.value.status == B.DEC_E_DEVICE_FAULT
    st = dec.stats()
    assert st["last_fault"] & bit and st["state"] == 1
    with pytest.raises(B.DecError) as ei:
        dec.step([1], [1])
    assert ei.value.status == B.DEC_E_NEEDS_RESET
    dec.reset_state()
    assert dec.stats()["state"] == 0
    orc = oracle.Oracle(mw, cap=wl.cap)
    for p, t in enumerate([5, 9, 11]):
        assert_close(dec.step([t], [p]).logits[0], orc.step(0, t, p), wl)
    dec.close()


def test_device_check_write_map_paged():
    from graph_replay_gb300 import _binding as B
    wl = gen.WORKLOADS["tiny"].replace(name="tiny_pg", layout="paged", page_size=16, num_pages=8)
    dec, mw = make_decoder(wl)
    dec.step([4], [0])
    dec.launch(_slots(dec, [4], [1], [wl.num_pages * 16 + 1]))
    with pytest.raises(B.DecError) as ei:
        dec.wait()
    assert ei.value.status == B.DEC_E_DEVICE_FAULT
    assert dec.stats()["last_fault"] & B.DEC_FAULT_WRITE_MAP
    with pytest.raises(B.DecError) as ei:
        dec.set_slot_map(np.full((1, wl.cap // 16), wl.num_pages, dtype=np.int32))
    assert ei.value.status == B.DEC_E_RANGE
    dec.reset_state()
    dec.step([4], [0])
    dec.close()


def test_wait_timeout_poisons_handle():
    from graph_replay_gb300 import _binding as B
    wl = gen.WORKLOADS["tiny"]
    dec, mw = make_decoder(wl)
    dec.step([1], [0])
    B.dec_set_timeout(dec.h, 20)
    B.dec_debug_busy(dec.h, 300000)        # a kernel that ends by itself after ~0.3 s
    with pytest.raises(B.DecError) as ei:
        dec.wait()
    assert ei.value.status == B.DEC_E_TIMEOUT
    assert dec.stats()["state"] == 2
    for call in (lambda: dec.step([1], [1]), dec.reset_state, lambda: dec.launch(None)):
        with pytest.raises(B.DecError) as ei:
            call()
        assert ei.value.status == B.DEC_E_POISONED
    import torch
    torch.cuda.synchronize()               # the busy kernel has ended; nothing is left in flight
    dec.close()


def test_unbound_and_misshaped_weights_refused():
    from graph_replay_gb300 import _binding as B
    from graph_replay_gb300 import make_config
    from gen.device import upload_weights
    wl = gen.WORKLOADS["tiny"]
    mw = gen.make_weights(wl)
    w = upload_weights(mw, "cuda:0")
    cfg = make_config(wl.n_layers, wl.d_model, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.ffn_hidden, wl.vocab,
                      "f32", "f32", wl.rms_eps, wl.rope_theta)
    h = B.dec_init(cfg)
    t = w["embed"]
    bad = B.dec_weight(B.DEC_W_EMBED, -1, B.DEC_DTYPE_F32, 0, wl.vocab + 1, wl.d_model, t.data_ptr())
    with pytest.raises(B.DecError) as ei:
        B.dec_load_weights(h, [bad])
    assert ei.value.status == B.DEC_E_INVALID and "shape" in str(ei.value)
    ok = B.dec_weight(B.DEC_W_EMBED, -1, B.DEC_DTYPE_F32, 0, wl.vocab, wl.d_model, t.data_ptr())
    B.dec_load_weights(h, [ok])
    with pytest.raises(B.DecError) as ei:
        B.dec_capture(h, wl.cap, 1, B.DEC_KV_CONTIGUOUS)
    assert ei.value.status == B.DEC_E_INVALID and "unbound" in str(ei.value)
    B.dec_destroy(h)
