"""Python face of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` leg are the only callers.  Nothing in the
``graph_replay_gb300`` package imports it, and it imports nothing from there.

``ORACLE_LIB_UNDER_TEST`` (environment): load that compiled copy of
``oracle.c`` instead of building this one.  Only the mutation test sets it, to
check that the pins reject deliberately broken copies of the oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
_DT = {"f32": F32, "bf16": BF16}
LAYER_ROLES = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc -O2, OpenMP, IEEE fp64, no contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
                           "-fPIC", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrcModel(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn_hidden", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("wdtype", ctypes.c_int), ("kvdtype", ctypes.c_int),
                ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layer", ctypes.POINTER(ctypes.c_void_p))]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(os.environ.get("ORACLE_LIB_UNDER_TEST") or build())
            P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            I64 = ctypes.c_int64
            lib.orc_bf16_value.restype = D
            lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_round.restype = ctypes.c_uint16
            lib.orc_bf16_round.argtypes = [D]
            lib.orc_rmsnorm.restype = None
            lib.orc_rmsnorm.argtypes = [P, I, P, I, D, P]
            lib.orc_matvec.restype = None
            lib.orc_matvec.argtypes = [P, I, I, I, P, P]
            lib.orc_rope.restype = None
            lib.orc_rope.argtypes = [P, I, I, D]
            lib.orc_silu.restype = D
            lib.orc_silu.argtypes = [D]
            lib.orc_softmax.restype = None
            lib.orc_softmax.argtypes = [P, I, P]
            lib.orc_attend.restype = None
            lib.orc_attend.argtypes = [P, P, P, I, I64, I, I, P]
            lib.orc_argmax.restype = I
            lib.orc_argmax.argtypes = [P, I]
            lib.orc_step.restype = I
            lib.orc_step.argtypes = [ctypes.POINTER(OrcModel), P, P, I, I, I, P, P]
            lib.orc_set_threads.restype = None
            lib.orc_set_threads.argtypes = [I]
            lib.orc_threads.restype = I
            lib.orc_threads.argtypes = []
            lib.orc_full_causal.restype = I
            lib.orc_full_causal.argtypes = [ctypes.POINTER(OrcModel), P, I, P, P, P]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _dt_of(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError(a.dtype)


# ---------- the pieces, one call each ----------

def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(bits)


def bf16_round(v: float) -> int:
    return _load().orc_bf16_round(float(v))


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x = _f64(x)
    g = np.ascontiguousarray(g)
    out = np.empty_like(x)
    _load().orc_rmsnorm(x.ctypes.data, x.size, g.ctypes.data, _dt_of(g), eps, out.ctypes.data)
    return out


def matvec(W, h) -> np.ndarray:
    W = np.ascontiguousarray(W)
    h = _f64(h)
    rows, cols = W.shape
    out = np.empty(rows, dtype=np.float64)
    _load().orc_matvec(W.ctypes.data, _dt_of(W), rows, cols, h.ctypes.data, out.ctypes.data)
    return out


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = _f64(v).copy()
    _load().orc_rope(v.ctypes.data, v.size, pos, theta)
    return v


def silu(z: float) -> float:
    return _load().orc_silu(float(z))


def softmax(s) -> np.ndarray:
    s = _f64(s)
    a = np.empty_like(s)
    _load().orc_softmax(s.ctypes.data, s.size, a.ctypes.data)
    return a


def attend(q, K, V) -> np.ndarray:
    """One head over positions [0, len(K)): K, V arrays [npos, hd] (uint16 bf16, float32 or float64)."""
    q = _f64(q)
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    assert K.dtype == V.dtype and K.shape == V.shape
    npos, hd = K.shape
    o = np.empty(hd, dtype=np.float64)
    _load().orc_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, _dt_of(K), hd, npos, hd,
                       o.ctypes.data)
    return o


def argmax(v) -> int:
    v = _f64(v)
    return _load().orc_argmax(v.ctypes.data, v.size)


def set_threads(n: int) -> int:
    """Thread count of the oracle's parallel loops (for timing; results do not
    depend on it).  Returns the count now in effect."""
    lib = _load()
    lib.orc_set_threads(int(n))
    return lib.orc_threads()


def top2_margin(logits) -> float:
    """Largest logit minus the second largest (0 when the maximum is shared)."""
    v = np.sort(np.asarray(logits, dtype=np.float64))
    return float(v[-1] - v[-2])


class Oracle:
    """The oracle decoder over one set of host weights (gen.ModelWeights).

    Each sequence (row) owns a KV store: per layer, K and V arrays
    [cap, n_kv_heads, head_dim] in logical position order and in the KV dtype
    (uint16 bf16 bits or float32).  Rows are independent sequences."""

    def __init__(self, mw, cap: int, rows: int = 1, alloc_kv: bool = True):
        wl = mw.wl
        self.mw, self.wl, self.cap, self.rows = mw, wl, cap, rows
        self._keep: List[np.ndarray] = []
        ptrs = []
        for lw in mw.layers:
            for r in LAYER_ROLES:
                a = np.ascontiguousarray(lw[r])
                self._keep.append(a)
                ptrs.append(a.ctypes.data)
        self._layer_ptrs = (ctypes.c_void_p * len(ptrs))(*ptrs)
        for a in (mw.embed, mw.final_norm, mw.lm_head):
            assert a.flags["C_CONTIGUOUS"]
        self.model = OrcModel(wl.n_layers, wl.d_model, wl.n_heads, wl.n_kv_heads, wl.head_dim,
                              wl.ffn_hidden, wl.vocab, wl.rms_eps, wl.rope_theta, _DT[wl.wdtype],
                              _DT[wl.kvdtype], mw.embed.ctypes.data, mw.final_norm.ctypes.data,
                              mw.lm_head.ctypes.data,
                              ctypes.cast(self._layer_ptrs, ctypes.POINTER(ctypes.c_void_p)))
        kvt = np.uint16 if wl.kvdtype == "bf16" else np.float32
        self.kvt = kvt
        self.K: List[List[np.ndarray]] = []
        self.V: List[List[np.ndarray]] = []
        if alloc_kv:
            for _ in range(rows):
                self.K.append([np.zeros((cap, wl.n_kv_heads, wl.head_dim), dtype=kvt)
                               for _ in range(wl.n_layers)])
                self.V.append([np.zeros((cap, wl.n_kv_heads, wl.head_dim), dtype=kvt)
                               for _ in range(wl.n_layers)])

    def step(self, row: int, token: int, pos: int, hidden: bool = False):
        """One decode step of sequence `row`: writes K/V at pos, returns fp64 logits [vocab]."""
        wl = self.wl
        kp = (ctypes.c_void_p * wl.n_layers)(*[a.ctypes.data for a in self.K[row]])
        vp = (ctypes.c_void_p * wl.n_layers)(*[a.ctypes.data for a in self.V[row]])
        logits = np.empty(wl.vocab, dtype=np.float64)
        hid = np.empty(wl.d_model, dtype=np.float64) if hidden else None
        rc = _load().orc_step(ctypes.byref(self.model), ctypes.cast(kp, ctypes.c_void_p),
                              ctypes.cast(vp, ctypes.c_void_p), self.cap, int(token), int(pos),
                              logits.ctypes.data, hid.ctypes.data if hidden else None)
        if rc != 0:
            raise ValueError(f"oracle step refused (token={token}, pos={pos}, cap={self.cap})")
        return (logits, hid) if hidden else logits

    def full_causal(self, tokens):
        """Direct causal pass over a whole prompt: (logits [n, vocab], K, V per layer [n, Hkv, hd])."""
        wl = self.wl
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tokens.size
        Ks = [np.zeros((n, wl.n_kv_heads, wl.head_dim), dtype=self.kvt) for _ in range(wl.n_layers)]
        Vs = [np.zeros((n, wl.n_kv_heads, wl.head_dim), dtype=self.kvt) for _ in range(wl.n_layers)]
        kp = (ctypes.c_void_p * wl.n_layers)(*[a.ctypes.data for a in Ks])
        vp = (ctypes.c_void_p * wl.n_layers)(*[a.ctypes.data for a in Vs])
        logits = np.empty((n, wl.vocab), dtype=np.float64)
        rc = _load().orc_full_causal(ctypes.byref(self.model), tokens.ctypes.data, n, logits.ctypes.data,
                                     ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp, ctypes.c_void_p))
        if rc != 0:
            raise ValueError("oracle full causal pass refused")
        return logits, Ks, Vs


# ---- sampling suffix ("Models, Registry and the Driver", section "The Driver":
# Head::Sample -- temperature, top-k, top-p, min-p, top-n logprobs).  Plain fp64
# restatement of the definition; the uniform comes from splitmix64 (Steele, Lea
# and Flood's SplitMix64 with Vigna's finalizer), written here from its
# published definition. ----

_M64 = (1 << 64) - 1


def splitmix64_at(seed: int, counter: int) -> int:
    """Output `counter` (0-based) of splitmix64 started at `seed`."""
    z = (seed + (counter + 1) * 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def uniform(seed: int, row: int, pos: int) -> float:
    """The sampling uniform of (row, position): top 53 bits of output (row << 32 | pos)."""
    return (splitmix64_at(seed & _M64, (row << 32) | pos) >> 11) * 2.0 ** -53


def sample(logits, temperature: float, top_k: int, top_p: float = 1.0, min_p: float = 0.0, u: float = 0.0):
    """One pick.  Returns (token, order, S, last): `order` the candidate ids by
    (logit desc, index asc), S the inclusive sums of their weights
    exp((l - l_max) / temperature), `last` the index in `order` of the last kept
    candidate.  temperature == 0 is the greedy pick."""
    l = np.asarray(logits, dtype=np.float64)
    order = np.lexsort((np.arange(l.size), -l))            # logit desc, then index asc
    if temperature <= 0.0:
        return int(order[0]), order[:1], np.ones(1), 0
    k = int(min(max(top_k, 1), l.size))
    order = order[:k]
    q = np.exp((l[order] - l[order[0]]) / temperature)
    S = np.cumsum(q)
    last_p = int(np.argmax(S >= min(top_p, 1.0) * S[-1]))   # shortest prefix reaching top_p of the mass
    last_m = int(np.count_nonzero(q >= min_p)) - 1          # q is non-increasing along `order`
    last = max(0, min(last_p, last_m))
    target = u * S[last]
    j = int(np.argmax(S[: last + 1] > target))
    return int(order[j]), order, S, last


def top_logprobs(logits, n: int):
    """The n tokens of largest logit (ties: lower index) and their log softmax values."""
    l = np.asarray(logits, dtype=np.float64)
    order = np.lexsort((np.arange(l.size), -l))[:n]
    m = l.max()
    lse = m + np.log(np.sum(np.exp(l - m)))
    return order, l[order] - lse
