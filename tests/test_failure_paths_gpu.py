"""The failure branches of the hot path, driven on the GPU without faulting it
("Execution", sections "Failure handling" and "Verification"):

* the non-finite flag of the head ("The Driver": the host reads back the
  chosen id and a non-finite flag) seen at 1 -- a NaN planted in one token's
  embedding row poisons that row only; an Inf in the LM head poisons every row;
* the device SlotMap check (DEC_FAULT_SLOT_MAP) -- an out-of-range page id
  written straight into the device slot map, past dec_set_slot_map's host check;
* the bounded in-kernel waits of the persistent step giving up (DEC_FAULT_WAIT)
  -- a grid-wide dependency that cannot complete, and a ring stage whose copy
  is never issued; the kernel exits, the step is a typed fault, reset recovers.

Every fault here is a value the kernels' own checks turn into an error bit, or
a wait that ends by its own bound: no test traps, hangs or faults the GPU."""
import dataclasses

import numpy as np
import pytest

import gen
import oracle
from _harness import assert_close, make_decoder

pytestmark = pytest.mark.gpu

ONE_B_2L = gen.WORKLOADS["1b"].replace(name="1b_fail", n_layers=2, cap=256)


def _oracle_flag(logits) -> int:
    return int(not np.isfinite(np.asarray(logits)).all())


@pytest.mark.parametrize("strategy, rows", [("graph", 2), ("persistent", 1), ("persistent", 2)])
def test_nonfinite_flag_follows_the_row(strategy, rows):
    import torch
    wl = ONE_B_2L.replace(rows=rows)
    dec, mw = make_decoder(wl, strategy=strategy)
    bad, good = 17, 4242
    # a NaN in one embedding element of token `bad` (the library reads the weights in place)
    dec._weights["embed"][bad, 5] = float("nan")
    torch.cuda.synchronize()
    mw_bad = dataclasses.replace(mw, embed=mw.embed.copy())
    mw_bad.embed[bad, 5] = 0x7FC0           # the same NaN, bf16 bits, for the oracle
    orc_good = oracle.Oracle(mw, cap=wl.cap)
    orc_bad = oracle.Oracle(mw_bad, cap=wl.cap)
    if rows == 2:
        res = dec.step([bad, good], [0, 0])
        ref_bad = orc_bad.step(0, bad, 0)
        ref_good = orc_good.step(0, good, 0)
        assert _oracle_flag(ref_bad) == 1 and _oracle_flag(ref_good) == 0
        assert list(res.nonfinite) == [1, 0]
        assert_close(res.logits[1], ref_good, wl, "clean row beside a non-finite row")
    else:
        res = dec.step([good], [0])
        assert list(res.nonfinite) == [0]
        assert_close(res.logits[0], orc_good.step(0, good, 0), wl, "clean step")
        res = dec.step([bad], [1])
        assert list(res.nonfinite) == [1]
        assert not np.isfinite(res.logits[0]).all()
    st = dec.stats()
    assert st["state"] == 0                 # a non-finite logit is a result, not a fault
    dec.close()


@pytest.mark.parametrize("strategy, rows", [("graph", 2), ("persistent", 1), ("persistent", 4)])
def test_nonfinite_flag_from_the_head(strategy, rows):
    import torch
    wl = ONE_B_2L.replace(rows=rows)
    dec, mw = make_decoder(wl, strategy=strategy)
    toks = [int(t) for t in gen.prompt_tokens(wl, n=rows)]
    res = dec.step(toks, [3] * rows)
    assert list(res.nonfinite) == [0] * rows
    dec.reset_state()
    dec._weights["lm_head"][777, 11] = float("inf")   # logit 777 is +-Inf (or NaN) for every row
    torch.cuda.synchronize()
    res = dec.step(toks, [3] * rows)
    assert list(res.nonfinite) == [1] * rows
    assert not np.isfinite(res.logits[:, 777]).any()
    dec.close()


def _slot_map_case(strategy, rows):
    wl = ONE_B_2L.replace(name=f"1b_fail_pg{rows}", rows=rows, layout="paged", page_size=16, num_pages=64)
    return wl, make_decoder(wl, strategy=strategy)


@pytest.mark.parametrize("name, strategy, rows", [("tiny", "graph", 1), ("1b", "graph", 2), ("1b", "persistent", 1)])
def test_device_slot_map_check(name, strategy, rows):
    """An out-of-range page id reaches the device slot map without the host
    check; the attention kernels' own check flags it instead of forming an
    address from it, the step is a typed fault, and reset recovers."""
    import torch
    from graph_replay_gb300 import _binding as B
    if name == "tiny":
        wl = gen.WORKLOADS["tiny"].replace(name="tiny_pg_sm", layout="paged", page_size=16, num_pages=8)
        dec, mw = make_decoder(wl)
    else:
        wl, (dec, mw) = _slot_map_case(strategy, rows)
    ppr = wl.cap // wl.page_size
    toks = [int(t) for t in gen.prompt_tokens(wl, n=rows)]
    first = dec.step(toks, [0] * rows).logits.copy()
    dec.reset_state()
    # the last page of row 0: read by every step's sweep of [0, cap), not written at pos 0
    view = torch.as_tensor(_dev_int32(B.dec_slot_map_ptr(dec.h), rows * ppr), device="cuda:0")
    view[ppr - 1] = wl.num_pages + 5
    torch.cuda.synchronize()
    with pytest.raises(B.DecError) as ei:
        dec.step(toks, [0] * rows)
    assert ei.value.status == B.DEC_E_DEVICE_FAULT
    st = dec.stats()
    assert st["last_fault"] & B.DEC_FAULT_SLOT_MAP and st["state"] == 1
    with pytest.raises(B.DecError) as ei:
        dec.step(toks, [0] * rows)
    assert ei.value.status == B.DEC_E_NEEDS_RESET
    # recovery: a valid map through the host call, then reset
    dec.set_slot_map(np.arange(rows * ppr, dtype=np.int32).reshape(rows, ppr))
    dec.reset_state()
    again = dec.step(toks, [0] * rows).logits
    assert np.array_equal(first, again)
    ref = oracle.Oracle(mw, cap=wl.cap).step(0, toks[0], 0)
    assert_close(again[0], ref, wl, "after slot-map recovery")
    dec.close()


class _dev_int32:
    """A device int32 buffer seen through __cuda_array_interface__ (no copy)."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": (n,), "typestr": "<i4",
                                         "strides": None, "version": 2}


@pytest.mark.parametrize("hook", ["hold_phase", "drop_stage"])
def test_persistent_wait_gives_up_and_recovers(hook):
    """A wait of the whole-step kernel that cannot complete gives up after its
    poll bound: the step returns DEC_E_DEVICE_FAULT with DEC_FAULT_WAIT, the
    kernel has exited (the next call does not hang), reset recovers, and the
    next step equals the one before the fault bit for bit."""
    import torch
    from graph_replay_gb300 import _binding as B
    wl = ONE_B_2L
    dec, mw = make_decoder(wl, strategy="persistent")
    toks = [int(t) for t in gen.prompt_tokens(wl, n=3)]
    before = [dec.step([t], [p]).logits[0].copy() for p, t in enumerate(toks)]
    dec.reset_state()
    if hook == "hold_phase":
        # the O-proj of layer 1 waits for attention's count to exceed the grid size
        B.dec_debug_wait(dec.h, grid_polls=1 << 12, hold_phase=1 + 5 * 1 + 1)
    else:
        # CTA 0 never issues its third stage; its consumers give up on it
        B.dec_debug_wait(dec.h, ring_polls=1 << 16, drop_stage=2)
    with pytest.raises(B.DecError) as ei:
        dec.step([toks[0]], [0])
    assert ei.value.status == B.DEC_E_DEVICE_FAULT
    st = dec.stats()
    assert st["last_fault"] & B.DEC_FAULT_WAIT and st["state"] == 1
    torch.cuda.synchronize()                  # nothing of the failed step is still running
    B.dec_debug_wait(dec.h)                   # default bounds, no hooks
    dec.reset_state()
    after = [dec.step([t], [p]).logits[0].copy() for p, t in enumerate(toks)]
    for a, b in zip(before, after):
        assert np.array_equal(a, b)
    orc = oracle.Oracle(mw, cap=wl.cap)
    for p, t in enumerate(toks):
        assert_close(after[p], orc.step(0, t, p), wl, f"after the give-up, pos {p}")
    dec.close()


def test_wait_hooks_need_the_persistent_strategy():
    from graph_replay_gb300 import _binding as B
    dec, _ = make_decoder(ONE_B_2L.replace(rows=2))
    with pytest.raises(B.DecError) as ei:
        B.dec_debug_wait(dec.h, 1, 1, 0, 0)
    assert ei.value.status == B.DEC_E_STATE
    dec.close()
