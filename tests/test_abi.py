"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/snap.h declares; host-only calls behave as documented (no GPU needed)."""
import ctypes
import math
import os
import re

import pytest

from fixed_size_kv_gb300 import build, inputs, snap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "snap.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(snap_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (brings the CUDA runtime libraries into the process)
    build.build()
    return snap.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    assert set(names) == set(snap.SIGNATURES), set(names) ^ set(snap.SIGNATURES)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert snap.status_string(s)
    assert snap.status_string(0) == "ok"


def _cfg(name):
    return snap.make_config(**inputs.WORKLOADS[name].config_kwargs())


def test_config_check(lib):
    for name in inputs.WORKLOADS:
        assert snap.config_check(_cfg(name)) == snap.SNAP_OK, name
    good = inputs.WORKLOADS["gqa_2k_tiny"]
    bad = [dict(P=4), dict(W=300), dict(L_recent=0), dict(n_q_heads=30), dict(sm_scale=0.0),
           dict(K=-1)]
    for kw in bad:
        assert snap.config_check(snap.make_config(**good.replace(**kw).config_kwargs())) == snap.SNAP_ERR_SHAPE, kw
    unsupported = [dict(d_qk=64, d_v=64), dict(n_q_heads=80, n_kv_heads=8)]
    for kw in unsupported:
        assert snap.config_check(snap.make_config(**good.replace(**kw).config_kwargs())) == snap.SNAP_ERR_UNSUPPORTED


def test_cache_bytes_four_times_smaller(lib):
    """The cache of a 128k prompt is 4x smaller than a full cache of it: exactly for
    the K/V rows, and within 0.5% for the whole buffer (which also holds the
    per-sequence meta and the selected-position list)."""
    for name in ("gqa_128k_b16", "mla_128k_b8"):
        wl = inputs.WORKLOADS[name]
        full_wl = wl.replace(L_sink=0, K=0, L_recent=131072)
        fixed = snap.cache_bytes(_cfg(name), 1)
        full = snap.cache_bytes(snap.make_config(**full_wl.config_kwargs()), 1)
        row = wl.n_kv_heads * (wl.d_qk + (wl.d_v if wl.layout == 0 else 0)) * 2
        assert (full_wl.C * row) / (wl.C * row) == 4.0
        assert fixed >= wl.C * row and full >= full_wl.C * row
        assert math.isclose(full / fixed, 4.0, rel_tol=5e-3)
