"""Failure detection on the GPU without a fault.

Every pipeline kernel bounds its waits (mbarrier polls timed by the device's global
timer).  When a wait expires, the kernel records SNAP_ERR_TIMEOUT in the cache's status
word and exits, and the host reads it with snap_check_device().  Here a self-test
kernel makes one wait run out (an mbarrier nothing arrives on): the status must say so,
and the same context must then run a decode step that still matches the oracle.  No
trap, assert, bad address or endless loop is involved.
"""
import math
import time

import pytest
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap
from parity import check_outputs, oracle_cfg, snap_cfg

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_the_context_stays_usable():
    wl = inputs.Workload("fail", 0, 32, 8, 128, 128, 4, 60, 64, 16, 7, 1, 0, 0, 0, 1 / math.sqrt(128))
    cache = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=300)
    pre = inputs.gen_prefill(wl, 300, seed=5)
    cache.compress(0, pre.K.cuda(), pre.V.cuda(), pre.Q.cuda())
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK

    t0 = time.perf_counter()
    cache.selftest_bounded_wait()
    status = cache.check_device()
    waited = time.perf_counter() - t0
    assert status == snap.SNAP_ERR_TIMEOUT
    assert 0.5 < waited < 60.0, waited            # the wait gave up after its bound
    assert cache.check_device() == snap.SNAP_OK    # cleared by the read

    # the same context keeps working
    ocache = oracle.compress(oracle_cfg(wl), pre.K, pre.V, pre.Q)
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = inputs.gen_decode(wl, 1, step=0, seed=5)
    out = cache.decode_step(slots, tok.q.cuda(), tok.k.cuda(), tok.v.cuda())
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    oracle.append(ocache, tok.k[0], tok.v[0])
    check_outputs(out[0], oracle.decode_attn(ocache, tok.q[0]), "after the expired wait")
