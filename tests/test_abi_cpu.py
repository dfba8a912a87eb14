"""The C ABI on a machine without a GPU: the library builds, loads and exports
every entry point include/graphdec.h declares; configuration checks refuse bad
configurations before any device call; pure host arithmetic."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "graphdec.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char \*|const char\*)\s*(dec_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from graph_replay_gb300 import build, _binding
    build.build()
    return _binding.load_library()


def test_header_declares_the_contract():
    names = _declared()
    for required in ("dec_init", "dec_load_weights", "dec_capture", "dec_step", "dec_reset_state",
                     "dec_destroy", "dec_set_slot_map"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from graph_replay_gb300 import _binding
    names = _declared()
    assert sorted(_binding.SYMBOLS) == names
    for n in names:
        assert getattr(lib, n) is not None


def _cfg(**kw):
    from graph_replay_gb300 import make_config
    base = dict(n_layers=2, d_model=64, n_heads=4, n_kv_heads=4, head_dim=16, ffn_hidden=128, vocab=256,
                weight_dtype="f32", kv_dtype="f32", rms_eps=1e-5, rope_theta=1e4)
    base.update(kw)
    return make_config(**base)


@pytest.mark.parametrize("kw, code, word", [
    (dict(n_layers=0), 1, "n_layers"),
    (dict(n_kv_heads=3), 1, "divide"),
    (dict(head_dim=15), 1, "even"),
    (dict(vocab=0), 1, "vocab"),
    (dict(rope_theta=0.0), 1, "rope_theta"),
    (dict(weight_dtype=7), 1, "weight_dtype"),
    (dict(head_dim=48, n_heads=4, d_model=192), 2, "head_dim"),
    (dict(n_heads=12, n_kv_heads=4, d_model=192), 2, "n_heads / n_kv_heads"),
    (dict(weight_dtype="bf16", d_model=68), 2, "d_model"),
])
def test_init_refuses_bad_configs_without_a_device(lib, kw, code, word):
    from graph_replay_gb300 import _binding as B
    cfg = _cfg(**kw)
    h = ctypes.c_void_p()
    rc = lib.dec_init(ctypes.byref(cfg), ctypes.byref(h))
    assert rc == code
    assert h.value is None
    assert word in lib.dec_last_error(None).decode()
    assert B.status_str(rc) in ("DEC_E_INVALID", "DEC_E_UNSUPPORTED")


def test_workspace_size_arithmetic(lib):
    from graph_replay_gb300 import _binding as B
    import gen
    wl = gen.WORKLOADS["8b"]
    cfg = _cfg(n_layers=wl.n_layers, d_model=wl.d_model, n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads,
               head_dim=wl.head_dim, ffn_hidden=wl.ffn_hidden, vocab=wl.vocab, weight_dtype="bf16", kv_dtype="bf16")
    n = B.dec_workspace_size(cfg, wl.cap, 1, B.DEC_KV_CONTIGUOUS)
    kv = wl.kv_swept_bytes()
    assert kv <= n <= kv + 64 * 2 ** 20
    wl4 = gen.WORKLOADS["8b_paged"]
    n4 = B.dec_workspace_size(cfg, wl4.cap, 8, B.DEC_KV_PAGED, 16, 4096)
    pool = 2 * wl4.n_layers * 4096 * 16 * wl4.kv_dim * 2
    assert pool <= n4 <= pool + 64 * 2 ** 20
    with pytest.raises(B.DecError):
        B.dec_workspace_size(cfg, 100, 1, B.DEC_KV_PAGED, 16, 4096)   # cap not a multiple of the page


def test_status_strings(lib):
    from graph_replay_gb300 import _binding as B
    assert B.status_str(B.DEC_OK) == "DEC_OK"
    assert B.status_str(B.DEC_E_TIMEOUT) == "DEC_E_TIMEOUT"
    assert B.status_str(12345) == "DEC_E_UNKNOWN"


def test_no_cpu_fallback_without_library(tmp_path):
    from graph_replay_gb300 import _binding as B
    with pytest.raises(ImportError):
        B.load_library(str(tmp_path / "missing.so"))


def test_every_handle_call_refuses_a_null_handle(lib):
    # no device is touched: the handle check comes first in every entry point
    import ctypes as C
    from graph_replay_gb300 import _binding as B
    skip = {"dec_init", "dec_workspace_size", "dec_last_error", "dec_status_str"}
    checked = 0
    for name, _, argtypes in B._SIG:
        if name in skip:
            continue
        args = []
        for t in argtypes:
            if t in (C.c_int32, C.c_int64, C.c_size_t, C.c_int, C.c_uint32):
                args.append(1)
            else:
                args.append(None)
        assert getattr(lib, name)(*args) == B.DEC_E_INVALID, name
        checked += 1
    assert checked == len(B.SYMBOLS) - len(skip)


def test_header_is_plain_c():
    # the boundary is a C ABI: the header compiles as C99 (no C++ or torch types)
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler on this machine")
    r = subprocess.run([cc, "-fsyntax-only", "-x", "c", "-std=c99", "-Wall", "-Wextra", "-Werror", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
