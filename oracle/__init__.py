"""CPU oracle of the SnapStream fixed-size KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
two share no code: this wrapper loads ``liboracle.so`` compiled from
``snap_oracle.c`` (plain C99, IEEE double on bf16 inputs).

Method (SnapStream episode companion page, "Fixed-Size Cache Layout" and
"Ring Buffer vs. Naive Slicing"): one static cache per sequence,
``[L_sink sinks | K selected | L_recent ring]``, built once at prefill by
SnapKV-style window scoring + max-pool + top-K, then decode writes each new
token into ring slot ``L_sink + K + (pos mod L_recent)``.

Parity status: every function here is pinned by tests/test_oracle_pins.py
except the reading of the softmax denominator (the full causal row), which no
page fixes: "parity unpinned" for that reading.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile snap_oracle.c into oracle/_build/liboracle.so with gcc."""
    src = os.path.join(_HERE, "snap_oracle.c")
    hdr = os.path.join(_HERE, "snap_oracle.h")
    newest = max(os.path.getmtime(src), os.path.getmtime(hdr))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    # -ffp-contract=off keeps every double operation individually rounded.
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Config(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("d_qk", ctypes.c_int), ("d_v", ctypes.c_int),
                ("L_sink", ctypes.c_int), ("K", ctypes.c_int), ("L_recent", ctypes.c_int),
                ("W", ctypes.c_int), ("P", ctypes.c_int), ("sm_scale", ctypes.c_double)]


class _Meta(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int64), ("T", ctypes.c_int64), ("n_sink", ctypes.c_int64),
                ("R0", ctypes.c_int64), ("n_mid", ctypes.c_int64)]


def build_mutant(k: int, out_dir: str) -> str:
    """Builds the oracle with deliberate mistake number k (tests of the pins only)."""
    src = os.path.join(_HERE, "snap_oracle.c")
    path = os.path.join(out_dir, f"liboracle_mutant{k}.so")
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           f"-DORACLE_MUTANT={k}", "-o", path, src, "-lm"])
    return path


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # SNAP_ORACLE_LIB points the pins at a deliberately broken build (mutation tests)
            lib = ctypes.CDLL(os.environ.get("SNAP_ORACLE_LIB") or build())
            P = ctypes.POINTER
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.snap_oracle_check_config.argtypes = [P(_Config)]
            lib.snap_oracle_plan.argtypes = [P(_Config), i64, P(_Meta)]
            lib.snap_oracle_window_scores.argtypes = [P(_Config), i64, vp, i64, i64, vp, vp, vp]
            lib.snap_oracle_maxpool.argtypes = [vp, i64, ctypes.c_int, vp]
            lib.snap_oracle_maxpool.restype = None
            lib.snap_oracle_select.argtypes = [vp, i64, i64, i64, vp]
            lib.snap_oracle_select.restype = i64
            lib.snap_oracle_compress.argtypes = [P(_Config), i64, vp, vp, i64, i64, vp, vp, vp,
                                                 vp, vp, P(_Meta)]
            lib.snap_oracle_compress_scored.argtypes = [P(_Config), i64, vp, vp, i64, i64, vp, vp, vp,
                                                        vp, vp, P(_Meta)]
            lib.snap_oracle_ring_slot.argtypes = [P(_Config), i64]
            lib.snap_oracle_ring_slot.restype = i64
            lib.snap_oracle_slot_valid.argtypes = [P(_Config), P(_Meta), i64]
            lib.snap_oracle_slot_position.argtypes = [P(_Config), P(_Meta), vp, i64]
            lib.snap_oracle_slot_position.restype = i64
            lib.snap_oracle_append.argtypes = [P(_Config), vp, vp, P(_Meta), vp, vp]
            lib.snap_oracle_decode_attn.argtypes = [P(_Config), vp, vp, P(_Meta), vp, vp]
            lib.snap_oracle_prefill_attn.argtypes = [P(_Config), i64, vp, vp, vp, i64, i64, vp, vp]
            _lib = lib
    return _lib


@dataclass
class Config:
    """Oracle-side configuration (same meaning as the library's, kept separate)."""
    layout: int
    n_q_heads: int
    n_kv_heads: int
    d_qk: int
    d_v: int
    L_sink: int
    K: int
    L_recent: int
    W: int
    P: int
    sm_scale: float

    @property
    def G(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def C(self) -> int:
        return self.L_sink + self.K + self.L_recent

    def _c(self) -> _Config:
        return _Config(self.layout, self.n_q_heads, self.n_kv_heads, self.d_qk, self.d_v,
                       self.L_sink, self.K, self.L_recent, self.W, self.P, float(self.sm_scale))


@dataclass
class Meta:
    S: int
    T: int
    n_sink: int
    R0: int
    n_mid: int

    def _c(self) -> _Meta:
        return _Meta(self.S, self.T, self.n_sink, self.R0, self.n_mid)

    @staticmethod
    def _from(m: _Meta) -> "Meta":
        return Meta(m.S, m.T, m.n_sink, m.R0, m.n_mid)


def _bits(a) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit patterns."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        t = a.detach().to("cpu").contiguous()
        assert t.dtype == torch.bfloat16, t.dtype
        return t.view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def check_config(cfg: Config) -> bool:
    return _load().snap_oracle_check_config(ctypes.byref(cfg._c())) == 0


def plan(cfg: Config, S: int) -> Meta:
    m = _Meta()
    rc = _load().snap_oracle_plan(ctypes.byref(cfg._c()), S, ctypes.byref(m))
    if rc != 0:
        raise ValueError(f"oracle plan rejected config/S (rc={rc})")
    return Meta._from(m)


def window_scores(cfg: Config, K, Q):
    """K: [S][H_kv][d_qk] bf16, Q: [W][H_q][d_qk] bf16 -> (lse [H_kv][W][G], col [H_kv][S])."""
    kb, qb = _bits(K), _bits(Q)
    S = kb.shape[0]
    lse = np.zeros((cfg.n_kv_heads, cfg.W, cfg.G), np.float64)
    col = np.zeros((cfg.n_kv_heads, S), np.float64)
    rc = _load().snap_oracle_window_scores(ctypes.byref(cfg._c()), S, _ptr(kb),
                                           cfg.n_kv_heads * cfg.d_qk, cfg.d_qk, _ptr(qb),
                                           _ptr(lse), _ptr(col))
    if rc != 0:
        raise ValueError(f"oracle window_scores rc={rc}")
    return lse, col


def window_columns(cfg: Config, K, Q, threads: int = 1, group: int = 0) -> np.ndarray:
    """The column scores of window_scores(cfg, K, Q) ([H_kv][S]), computed as sums over
    groups of `group` query heads (default: one group per KV head) with one
    window_scores call per (KV head, group), run on `threads` threads (the C oracle
    releases the GIL).  The scores are sums over observation rows, so the grouping
    changes only the order of the double-precision additions."""
    from concurrent.futures import ThreadPoolExecutor
    import torch
    G = cfg.G
    group = G if group <= 0 else group
    assert G % group == 0, (G, group)
    Kt = K if hasattr(K, "detach") else torch.from_numpy(np.ascontiguousarray(K)).view(torch.bfloat16)
    Qt = Q if hasattr(Q, "detach") else torch.from_numpy(np.ascontiguousarray(Q)).view(torch.bfloat16)
    S = Kt.shape[0]
    sub = Config(cfg.layout, group, 1, cfg.d_qk, cfg.d_v, cfg.L_sink, cfg.K, cfg.L_recent, cfg.W, cfg.P,
                 cfg.sm_scale)
    jobs = [(h, g0) for h in range(cfg.n_kv_heads) for g0 in range(0, G, group)]

    def run(job):
        h, g0 = job
        q0 = h * G + g0
        return window_scores(sub, Kt[:, h:h + 1].contiguous(), Qt[:, q0:q0 + group].contiguous())[1][0]

    col = np.zeros((cfg.n_kv_heads, S), np.float64)
    with ThreadPoolExecutor(max(1, threads)) as ex:
        for (h, _), c in zip(jobs, ex.map(run, jobs)):
            col[h] += c
    return col


def maxpool(x, P: int) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    y = np.zeros_like(x)
    _load().snap_oracle_maxpool(_ptr(x), x.shape[0], P, _ptr(y))
    return y


def select(score, lo: int, hi: int, K: int) -> np.ndarray:
    score = np.ascontiguousarray(score, np.float64)
    out = np.full(max(K, 1), -1, np.int32)
    n = _load().snap_oracle_select(_ptr(score), lo, hi, K, _ptr(out))
    return out[:n].copy()


@dataclass
class Cache:
    """Oracle cache of one sequence: k [H_kv][C][d_qk] / v [H_kv][C][d_v] uint16 bits."""
    cfg: Config
    k: np.ndarray
    v: np.ndarray | None
    sel: np.ndarray   # [H_kv][K] int32, -1 past n_mid
    meta: Meta
    pool: np.ndarray | None = None  # [H_kv][S-W] when scoring ran

    def valid(self, s: int) -> bool:
        return bool(_load().snap_oracle_slot_valid(ctypes.byref(self.cfg._c()),
                                                   ctypes.byref(self.meta._c()), s))

    def slot_positions(self) -> np.ndarray:
        """[H_kv][C] absolute position held by each slot, -1 where invalid."""
        lib = _load()
        c, m = self.cfg._c(), self.meta._c()
        out = np.full((self.cfg.n_kv_heads, self.cfg.C), -1, np.int64)
        for h in range(self.cfg.n_kv_heads):
            sel_h = np.ascontiguousarray(self.sel[h])
            for s in range(self.cfg.C):
                out[h, s] = lib.snap_oracle_slot_position(ctypes.byref(c), ctypes.byref(m),
                                                          _ptr(sel_h), s)
        return out


def compress(cfg: Config, K, V, Q, want_pool: bool = False, col=None) -> Cache:
    """K/V: [S][H_kv][d] bf16 (V None for MLA); Q: [W][H_q][d_qk] bf16.  With `col`
    ([H_kv][S] column scores, e.g. from window_columns) the scoring step is taken from
    it instead of being recomputed from Q (Q may then be None)."""
    kb = _bits(K)
    qb = _bits(Q) if Q is not None else None
    vb = _bits(V) if V is not None else None
    S = kb.shape[0]
    C, H = cfg.C, cfg.n_kv_heads
    ck = np.zeros((H, C, cfg.d_qk), np.uint16)
    cv = np.zeros((H, C, cfg.d_v), np.uint16) if cfg.layout == 0 else None
    sel = np.full((H, max(cfg.K, 1)), -1, np.int32)
    pool = np.zeros((H, max(S - cfg.W, 1)), np.float64) if want_pool else None
    m = _Meta()
    if col is not None:
        colb = np.ascontiguousarray(col, np.float64)
        assert colb.shape == (H, S), colb.shape
        rc = _load().snap_oracle_compress_scored(
            ctypes.byref(cfg._c()), S, _ptr(kb), _ptr(vb) if vb is not None else None,
            H * cfg.d_qk, cfg.d_qk, _ptr(colb), _ptr(ck), _ptr(cv) if cv is not None else None,
            _ptr(sel), _ptr(pool) if pool is not None else None, ctypes.byref(m))
    else:
        rc = _load().snap_oracle_compress(
            ctypes.byref(cfg._c()), S, _ptr(kb), _ptr(vb) if vb is not None else None,
            H * cfg.d_qk, cfg.d_qk, _ptr(qb), _ptr(ck), _ptr(cv) if cv is not None else None,
            _ptr(sel), _ptr(pool) if pool is not None else None, ctypes.byref(m))
    if rc != 0:
        raise ValueError(f"oracle compress rc={rc}")
    return Cache(cfg, ck, cv, sel[:, :cfg.K], Meta._from(m), pool)


def append(cache: Cache, k_new, v_new=None) -> None:
    kb = _bits(k_new)
    vb = _bits(v_new) if v_new is not None else None
    m = cache.meta._c()
    rc = _load().snap_oracle_append(ctypes.byref(cache.cfg._c()), _ptr(cache.k),
                                    _ptr(cache.v) if cache.v is not None else None,
                                    ctypes.byref(m), _ptr(kb), _ptr(vb) if vb is not None else None)
    if rc != 0:
        raise ValueError(f"oracle append rc={rc}")
    cache.meta = Meta._from(m)


def decode_attn(cache: Cache, q) -> np.ndarray:
    """q: [H_q][d_qk] bf16 -> out [H_q][d_v] float64."""
    qb = _bits(q)
    out = np.zeros((cache.cfg.n_q_heads, cache.cfg.d_v), np.float64)
    ck = np.ascontiguousarray(cache.k)
    cv = np.ascontiguousarray(cache.v) if cache.v is not None else None
    rc = _load().snap_oracle_decode_attn(ctypes.byref(cache.cfg._c()), _ptr(ck),
                                         _ptr(cv) if cv is not None else None,
                                         ctypes.byref(cache.meta._c()), _ptr(qb), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle decode_attn rc={rc}")
    return out


def prefill_attn(cfg: Config, Q, K, V):
    """Causal prefill attention: Q [S][H_q][d], K/V [S][H_kv][d] bf16 ->
    (out [S][H_q][d_v] float64, lse [S][H_q] float64, natural log)."""
    qb, kb, vb = _bits(Q), _bits(K), _bits(V)
    S = qb.shape[0]
    out = np.zeros((S, cfg.n_q_heads, cfg.d_v), np.float64)
    lse = np.zeros((S, cfg.n_q_heads), np.float64)
    rc = _load().snap_oracle_prefill_attn(ctypes.byref(cfg._c()), S, _ptr(qb), _ptr(kb), _ptr(vb),
                                          cfg.n_kv_heads * cfg.d_qk, cfg.d_qk, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle prefill_attn rc={rc}")
    return out, lse
