"""Comparison helpers shared by the GPU parity tests (the CUDA library vs the oracle).

Tolerances follow the problem statement that accompanies the SnapStream pages:
selected positions and ring contents bit-exact, except that a selected position
may differ from the oracle's only where the oracle's pooled scores of the two
candidates differ by less than 1e-6 relative; attention outputs within 2e-2
max-abs and 5e-3 mean-abs (bf16 inputs and outputs, fp32 accumulation).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap

MAX_ABS = 2e-2
MEAN_ABS = 5e-3
SEL_REL = 1e-6


def oracle_cfg(wl: inputs.Workload) -> oracle.Config:
    return oracle.Config(**wl.config_kwargs())


def snap_cfg(wl: inputs.Workload) -> snap.snap_config:
    return snap.make_config(**wl.config_kwargs())


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_selection(gpu_sel, ora_sel, ora_pool: np.ndarray, where: str = "") -> int:
    """GPU and oracle selections (ascending positions) agree up to ties within
    SEL_REL of the oracle's K-th pooled score.  ora_pool is indexed by position.
    Returns the number of tolerated swaps."""
    g = np.asarray(gpu_sel, dtype=np.int64)
    o = np.asarray(ora_sel, dtype=np.int64)
    assert len(g) == len(o), (where, len(g), len(o))
    assert (np.diff(g) > 0).all(), f"{where}: GPU selection not strictly ascending"
    gs, os_ = set(g.tolist()), set(o.tolist())
    diff = gs ^ os_
    if not diff:
        return 0
    tau = float(min(ora_pool[list(os_)]))
    for j in diff:
        assert abs(float(ora_pool[j]) - tau) <= SEL_REL * abs(tau), \
            f"{where}: position {j} (oracle score {ora_pool[j]!r}) vs K-th {tau!r}"
    return len(diff) // 2


def check_outputs(gpu_out: torch.Tensor, ora_out: np.ndarray, where: str = "") -> tuple[float, float]:
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    d = np.abs(g - ora_out)
    mx, mean = float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{where}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean


def gpu_meta(cache: snap.SnapCache, slot: int) -> dict:
    m = cache.meta()[slot].cpu().tolist()
    return dict(S=m[0], T=m[1], R0=m[2], n_sink=m[3], n_mid=m[4])


def check_cache_rows(cache: snap.SnapCache, slot: int, ocache: oracle.Cache, K_all: torch.Tensor,
                     V_all: torch.Tensor | None, where: str = "") -> None:
    """Every valid slot of the GPU cache holds, bit-exactly, the row of the position the
    oracle's layout assigns to it; middle slots hold the rows of the GPU's own selection;
    slots that hold nothing are zero.  K_all/V_all: [T][H_kv][d] all tokens so far."""
    cfg = ocache.cfg
    m = gpu_meta(cache, slot)
    om = ocache.meta
    assert (m["S"], m["T"], m["R0"], m["n_sink"], m["n_mid"]) == (om.S, om.T, om.R0, om.n_sink, om.n_mid), \
        (where, m, om)
    gk = bits(cache.k_cache()[slot])
    gv = bits(cache.v_cache()[slot]) if V_all is not None else None
    kb = bits(K_all)
    vb = bits(V_all) if V_all is not None else None
    pos = ocache.slot_positions()
    gsel = cache.selected()[slot].cpu().numpy() if cfg.K > 0 else None
    for h in range(cfg.n_kv_heads):
        for s in range(cfg.C):
            p = int(pos[h, s])
            if cfg.L_sink <= s < cfg.L_sink + cfg.K and p >= 0:
                p = int(gsel[h, s - cfg.L_sink])
            if p < 0:
                if s < cfg.L_sink + cfg.K:  # never-written sink / middle slots are zero
                    assert not gk[h, s].any(), (where, h, s)
                continue
            if not np.array_equal(gk[h, s], kb[p, h]):
                raise AssertionError(f"{where}: K row mismatch head {h} slot {s} position {p}")
            if vb is not None and not np.array_equal(gv[h, s], vb[p, h]):
                raise AssertionError(f"{where}: V row mismatch head {h} slot {s} position {p}")


def one_head_workload(wl: inputs.Workload) -> inputs.Workload:
    """The problem of one KV head alone: that head and its G query heads (every step of
    the method is independent across KV heads)."""
    return wl.replace(n_q_heads=wl.G, n_kv_heads=1)


def oracle_head_cache(wl: inputs.Workload, K: torch.Tensor, V: torch.Tensor | None, Q: torch.Tensor, h: int,
                      threads: int = 1, group: int = 0) -> oracle.Cache:
    """The oracle's cache of KV head h of one sequence, built from the prompt alone:
    K/V [S][H_kv][d] and Q [W][H_q][d] (CPU bf16).  Scoring runs on `threads` threads over
    groups of `group` query heads (oracle.window_columns).  pool holds the pooled scores."""
    G = wl.G
    one = one_head_workload(wl)
    ocfg = oracle_cfg(one)
    K1 = K[:, h:h + 1].contiguous()
    V1 = V[:, h:h + 1].contiguous() if V is not None else None
    Q1 = Q[:, h * G:(h + 1) * G].contiguous()
    m = oracle.plan(ocfg, K1.shape[0])
    scored = wl.K > 0 and m.R0 - m.n_sink > wl.K
    col = oracle.window_columns(ocfg, K1, Q1, threads=threads, group=group) if scored else None
    return oracle.compress(ocfg, K1, V1, Q1, want_pool=True, col=col)


def oracle_workers() -> int:
    import os
    return max(1, os.cpu_count() or 1)
