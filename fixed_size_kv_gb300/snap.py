"""Thin ctypes binding of libsnap (include/snap.h): argument marshalling only.

Every step of the method runs in the CUDA library; this module turns torch
tensors into device pointers and streams into handles, and raises on a non-OK
status.  PyTorch provides device memory and streams, nothing else.  There is no
fallback: if libsnap.so is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SNAP_OK = 0
SNAP_ERR_INVALID_ARG = 1
SNAP_ERR_SHAPE = 2
SNAP_ERR_UNSUPPORTED = 3
SNAP_ERR_CUDA = 4
SNAP_ERR_TIMEOUT = 5
SNAP_ERR_DEVICE_CHECK = 6

LAYOUT_GQA = 0
LAYOUT_MLA = 1

STAGE_ROWS = 1
STAGE_COLUMNS = 2
STAGE_SELECT = 4
STAGE_WRITE = 8
STAGE_ALL = 15


class SnapError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class snap_config(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("d_qk", ctypes.c_int), ("d_v", ctypes.c_int), ("L_sink", ctypes.c_int),
                ("K", ctypes.c_int), ("L_recent", ctypes.c_int), ("W", ctypes.c_int),
                ("P", ctypes.c_int), ("sm_scale", ctypes.c_float)]


class snap_cache_view(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("sel", ctypes.c_void_p), ("status", ctypes.c_void_p), ("C", ctypes.c_int64),
                ("max_batch", ctypes.c_int)]


# every symbol include/snap.h declares, with its ctypes signature
_P, _VP, _I, _I64, _SZ = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "snap_status_string": (ctypes.c_char_p, [_I]),
    "snap_abi_version": (_I, []),
    "snap_config_check": (_I, [_P(snap_config)]),
    "snap_cache_bytes": (_I, [_P(snap_config), _I, _P(_SZ)]),
    "snap_cache_create": (_I, [_P(snap_config), _I, _VP, _SZ, _VP, _P(_VP)]),
    "snap_cache_destroy": (None, [_VP]),
    "snap_cache_view_get": (_I, [_VP, _P(snap_cache_view)]),
    "snap_compress_ws_bytes": (_I, [_P(snap_config), _I64, _P(_SZ)]),
    "snap_compress": (_I, [_VP, _I, _VP, _VP, _I64, _I64, _I64, _VP, _VP, _SZ, _VP]),
    "snap_compress_lse": (_I, [_VP, _I, _VP, _VP, _I64, _I64, _I64, _VP, _VP, _VP, _SZ, _VP]),
    "snap_compress_stages": (_I, [_VP, _I, _VP, _VP, _I64, _I64, _I64, _VP, _VP, _VP, _SZ, _I, _VP]),
    "snap_window_logits": (_I, [_VP, _VP, _I64, _I64, _I64, _VP, _VP, _VP]),
    "snap_decode_append": (_I, [_VP, _VP, _I, _VP, _VP, _VP]),
    "snap_prefill_attn": (_I, [_VP, _VP, _I64, _VP, _VP, _I64, _I64, _VP, _VP, _VP]),
    "snap_decode_attn_ws_bytes": (_I, [_P(snap_config), _I, _P(_SZ)]),
    "snap_decode_attn_plan": (_I, [_VP, _I, _P(_I), _P(_I), _P(_I)]),
    "snap_selftest_bounded_wait": (_I, [_VP, _VP]),
    "snap_decode_attn": (_I, [_VP, _VP, _I, _VP, _VP, _VP, _SZ, _VP]),
    "snap_decode_step": (_I, [_VP, _VP, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "snap_check_device": (_I, [_VP, _VP]),
    "snap_decode_attn_noalloc": (_I, [_VP, _VP, _I, _VP, _VP, _VP]),
}

_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Loads libsnap.so; raises if it is absent (no fallback path exists)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libsnap.so not built ({path}); run "
                                       "`python -m fixed_size_kv_gb300.build`")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(s: int) -> str:
    try:
        return load().snap_status_string(int(s)).decode()
    except Exception:
        return f"status {s}"


def _check(status: int, where: str) -> None:
    if status != SNAP_OK:
        raise SnapError(status, where)


def make_config(layout, n_q_heads, n_kv_heads, d_qk, d_v, L_sink, K, L_recent, W, P,
                sm_scale) -> snap_config:
    return snap_config(layout, n_q_heads, n_kv_heads, d_qk, d_v, L_sink, K, L_recent, W, P,
                       float(sm_scale))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p | None:
    if t is None:
        return None
    assert t.is_cuda, "libsnap takes device tensors"
    return ctypes.c_void_p(t.data_ptr())


def config_check(cfg: snap_config) -> int:
    return load().snap_config_check(ctypes.byref(cfg))


def cache_bytes(cfg: snap_config, max_batch: int) -> int:
    n = ctypes.c_size_t()
    _check(load().snap_cache_bytes(ctypes.byref(cfg), max_batch, ctypes.byref(n)), "snap_cache_bytes")
    return n.value


def compress_ws_bytes(cfg: snap_config, S_max: int) -> int:
    n = ctypes.c_size_t()
    _check(load().snap_compress_ws_bytes(ctypes.byref(cfg), S_max, ctypes.byref(n)),
           "snap_compress_ws_bytes")
    return n.value


def decode_attn_ws_bytes(cfg: snap_config, max_n: int) -> int:
    n = ctypes.c_size_t()
    _check(load().snap_decode_attn_ws_bytes(ctypes.byref(cfg), max_n, ctypes.byref(n)),
           "snap_decode_attn_ws_bytes")
    return n.value


class SnapCache:
    """A cache bound to a torch-allocated device buffer, plus its workspaces.

    Methods call the C entry points of the same name (snap_compress,
    snap_decode_append, snap_decode_attn, snap_check_device).
    """

    def __init__(self, cfg: snap_config, max_batch: int, max_prompt: int = 1, max_n: int | None = None,
                 device="cuda", stream=None):
        self.cfg = cfg
        self.max_batch = max_batch
        self.device = torch.device(device)
        lib = load()
        nbytes = cache_bytes(cfg, max_batch)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        _check(lib.snap_cache_create(ctypes.byref(cfg), max_batch, _ptr(self.buf), nbytes,
                                     _stream(stream), ctypes.byref(h)), "snap_cache_create")
        self.handle = h
        self.ws_compress = torch.empty(compress_ws_bytes(cfg, max(max_prompt, 1)), dtype=torch.uint8,
                                       device=self.device)
        self.ws_decode = torch.empty(decode_attn_ws_bytes(cfg, max_n or max_batch), dtype=torch.uint8,
                                     device=self.device)
        v = snap_cache_view()
        _check(lib.snap_cache_view_get(h, ctypes.byref(v)), "snap_cache_view_get")
        self.view = v
        self.C = v.C

    def close(self):
        if getattr(self, "handle", None):
            load().snap_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def ensure_compress_ws(self, S: int):
        need = compress_ws_bytes(self.cfg, S)
        if self.ws_compress.numel() < need:
            self.ws_compress = torch.empty(need, dtype=torch.uint8, device=self.device)

    # ---------------------------------------------------------------- entry points
    def compress(self, slot: int, K: torch.Tensor, V: torch.Tensor | None, Q_obs: torch.Tensor,
                 stream=None) -> None:
        """K/V: [S][H_kv][d] bf16 (any strides with unit inner stride); Q_obs [W][H_q][d_qk]."""
        S = K.shape[0]
        self.ensure_compress_ws(S)
        assert K.dtype == torch.bfloat16 and K.stride(2) == 1
        if V is not None:
            assert V.stride() == K.stride() and V.dtype == torch.bfloat16
        Q_obs = Q_obs.contiguous()
        _check(load().snap_compress(self.handle, slot, _ptr(K), _ptr(V), S, K.stride(0), K.stride(1),
                                    _ptr(Q_obs), _ptr(self.ws_compress), self.ws_compress.numel(),
                                    _stream(stream)), "snap_compress")

    def compress_lse(self, slot: int, K: torch.Tensor, V: torch.Tensor | None, Q_obs: torch.Tensor,
                     lse_obs: torch.Tensor, stream=None) -> None:
        """snap_compress_lse: lse_obs fp32 [W][H_q], natural-log LSE of the window rows."""
        S = K.shape[0]
        self.ensure_compress_ws(S)
        assert lse_obs.dtype == torch.float32 and lse_obs.is_contiguous()
        Q_obs = Q_obs.contiguous()
        _check(load().snap_compress_lse(self.handle, slot, _ptr(K), _ptr(V), S, K.stride(0), K.stride(1),
                                        _ptr(Q_obs), _ptr(lse_obs), _ptr(self.ws_compress),
                                        self.ws_compress.numel(), _stream(stream)), "snap_compress_lse")

    def compress_stages(self, slot: int, K: torch.Tensor, V: torch.Tensor | None, Q_obs: torch.Tensor,
                        stages: int, lse_obs: torch.Tensor | None = None, stream=None) -> None:
        """snap_compress_stages: only the stages in `stages` (STAGE_* bits), in order."""
        S = K.shape[0]
        self.ensure_compress_ws(S)
        if lse_obs is not None:
            assert lse_obs.dtype == torch.float32 and lse_obs.is_contiguous()
        Q_obs = Q_obs.contiguous()
        _check(load().snap_compress_stages(self.handle, slot, _ptr(K), _ptr(V), S, K.stride(0), K.stride(1),
                                           _ptr(Q_obs), _ptr(lse_obs), _ptr(self.ws_compress),
                                           self.ws_compress.numel(), int(stages), _stream(stream)),
               "snap_compress_stages")

    def window_logits(self, K: torch.Tensor, Q_obs: torch.Tensor, stream=None) -> torch.Tensor:
        """Base-2 logits of the observation rows against every prompt key:
        fp32 [H_kv][G*W][S] (the compression's score GEMM, for inspection)."""
        S = K.shape[0]
        G = self.cfg.n_q_heads // self.cfg.n_kv_heads
        out = torch.empty((self.cfg.n_kv_heads, G * self.cfg.W, S), dtype=torch.float32, device=self.device)
        Q_obs = Q_obs.contiguous()
        _check(load().snap_window_logits(self.handle, _ptr(K), S, K.stride(0), K.stride(1), _ptr(Q_obs),
                                         _ptr(out), _stream(stream)), "snap_window_logits")
        return out

    def prefill_attn(self, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                     lse_obs: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """snap_prefill_attn: causal attention of one prompt (Q [S][H_q][128] contiguous,
        K/V [S][H_kv][128] with unit inner stride); writes O (bf16, same shape as Q) and,
        if given, lse_obs fp32 [W][H_q] for the last W rows.  Returns O."""
        S = Q.shape[0]
        Q = Q.contiguous()
        assert K.stride(2) == 1 and V.stride() == K.stride()
        if O is None:
            O = torch.empty_like(Q)
        assert O.is_contiguous() and O.dtype == torch.bfloat16
        if lse_obs is not None:
            assert lse_obs.dtype == torch.float32 and lse_obs.is_contiguous()
        _check(load().snap_prefill_attn(self.handle, _ptr(Q), S, _ptr(K), _ptr(V), K.stride(0), K.stride(1),
                                        _ptr(O), _ptr(lse_obs), _stream(stream)), "snap_prefill_attn")
        return O

    def decode_append(self, slots: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor | None,
                      stream=None) -> None:
        assert slots.dtype == torch.int32 and slots.is_contiguous()
        _check(load().snap_decode_append(self.handle, _ptr(slots), slots.numel(), _ptr(k_new.contiguous()),
                                         _ptr(v_new.contiguous() if v_new is not None else None),
                                         _stream(stream)), "snap_decode_append")

    def decode_attn(self, slots: torch.Tensor, q: torch.Tensor, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
        assert slots.dtype == torch.int32 and slots.is_contiguous()
        n = slots.numel()
        if out is None:
            out = torch.empty((n, self.cfg.n_q_heads, self.cfg.d_v), dtype=torch.float32,
                              device=self.device)
        assert out.dtype == torch.float32 and out.is_contiguous()
        _check(load().snap_decode_attn(self.handle, _ptr(slots), n, _ptr(q.contiguous()), _ptr(out),
                                       _ptr(self.ws_decode), self.ws_decode.numel(), _stream(stream)),
               "snap_decode_attn")
        return out

    def decode_step(self, slots: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor | None,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """snap_decode_step: append k_new/v_new, then attend with q (one call)."""
        assert slots.dtype == torch.int32 and slots.is_contiguous()
        n = slots.numel()
        if out is None:
            out = torch.empty((n, self.cfg.n_q_heads, self.cfg.d_v), dtype=torch.float32, device=self.device)
        _check(load().snap_decode_step(self.handle, _ptr(slots), n, _ptr(q.contiguous()), _ptr(k_new.contiguous()),
                                       _ptr(v_new.contiguous() if v_new is not None else None), _ptr(out),
                                       _ptr(self.ws_decode), self.ws_decode.numel(), _stream(stream)),
               "snap_decode_step")
        return out

    def decode_attn_noalloc(self, slots: torch.Tensor, q: torch.Tensor, out: torch.Tensor,
                            stream=None) -> int:
        """snap_decode_attn_noalloc: the same attention with the split partials in the
        library's fixed scratch array (no workspace).  Returns the status code."""
        assert slots.dtype == torch.int32 and slots.is_contiguous()
        assert out.dtype == torch.float32 and out.is_contiguous()
        return load().snap_decode_attn_noalloc(self.handle, _ptr(slots), slots.numel(), _ptr(q.contiguous()),
                                               _ptr(out), _stream(stream))

    def decode_attn_plan(self, n: int):
        """snap_decode_attn_plan: (splits, tiles_per_split, ctas_per_wave) for n sequences."""
        sp, tp, wv = _I(), _I(), _I()
        _check(load().snap_decode_attn_plan(self.handle, n, ctypes.byref(sp), ctypes.byref(tp), ctypes.byref(wv)),
               "snap_decode_attn_plan")
        return sp.value, tp.value, wv.value

    def selftest_bounded_wait(self, stream=None) -> None:
        """snap_selftest_bounded_wait: one kernel whose only wait expires (about 2 s); the
        next check_device() returns SNAP_ERR_TIMEOUT."""
        _check(load().snap_selftest_bounded_wait(self.handle, _stream(stream)), "snap_selftest_bounded_wait")

    def check_device(self, stream=None) -> int:
        return load().snap_check_device(self.handle, _stream(stream))

    # ------------------------------------------------------------------- inspection
    def _region(self, addr: int, numel: int, dtype) -> torch.Tensor:
        off = addr - self.buf.data_ptr()
        nbytes = numel * torch.tensor([], dtype=dtype).element_size()
        return self.buf[off:off + nbytes].view(dtype)

    def k_cache(self) -> torch.Tensor:
        c = self.cfg
        return self._region(self.view.k, self.max_batch * c.n_kv_heads * self.C * c.d_qk,
                            torch.bfloat16).view(self.max_batch, c.n_kv_heads, self.C, c.d_qk)

    def v_cache(self) -> torch.Tensor | None:
        if not self.view.v:
            return None
        c = self.cfg
        return self._region(self.view.v, self.max_batch * c.n_kv_heads * self.C * c.d_v,
                            torch.bfloat16).view(self.max_batch, c.n_kv_heads, self.C, c.d_v)

    def meta(self) -> torch.Tensor:
        """int32 [max_batch][8]: S, T, R0, n_sink, n_mid, pad."""
        return self._region(self.view.meta, self.max_batch * 8, torch.int32).view(self.max_batch, 8)

    def selected(self) -> torch.Tensor:
        c = self.cfg
        return self._region(self.view.sel, self.max_batch * c.n_kv_heads * c.K,
                            torch.int32).view(self.max_batch, c.n_kv_heads, c.K)
