"""The compression's score GEMM (tcgen05 tensor cores fed by TMA) against a plain
fp32 matrix product, through the snap_window_logits inspection entry point.

The logits are the dense contraction the SnapKV scoring step is built on: for KV
head h, observation row r = w*G + g (query head h*G + g at prompt position S-W+w)
against prompt key j, log2(e) * sm_scale * q.k.
"""
import math

import pytest
import torch

from fixed_size_kv_gb300 import inputs, snap
from parity import snap_cfg

pytestmark = pytest.mark.gpu


def reference_logits(wl, K, Q):
    G, W = wl.G, wl.W
    Qr = Q.float().view(W, wl.n_kv_heads, G, wl.d_qk).permute(1, 0, 2, 3).reshape(wl.n_kv_heads, W * G, wl.d_qk)
    Kh = K.float().permute(1, 2, 0)                     # [H_kv][d][S]
    return torch.bmm(Qr, Kh) * (wl.sm_scale * math.log2(math.e))


@pytest.mark.parametrize("shape", [
    dict(Hq=32, Hkv=8, d=128, W=64, S=1000),      # R = 256, ragged S
    dict(Hq=32, Hkv=8, d=128, W=32, S=2048),      # R = 128
    dict(Hq=16, Hkv=2, d=128, W=16, S=777),       # G = 8, R = 128
    dict(Hq=32, Hkv=8, d=128, W=3, S=300),        # R = 12 (one partial row tile)
    dict(Hq=128, Hkv=1, d=576, W=2, S=600, mla=True),  # MLA latent rows, R = 256
    dict(Hq=128, Hkv=1, d=576, W=3, S=450, mla=True),  # R = 384: three row tiles
])
def test_window_logits_match_matmul(shape):
    mla = shape.get("mla", False)
    wl = inputs.Workload("g", 1 if mla else 0, shape["Hq"], shape["Hkv"], shape["d"], 512 if mla else shape["d"],
                         4, 16, max(64, shape["W"]), shape["W"], 5, 1, 0, 0, 0, 1 / math.sqrt(128))
    pre = inputs.gen_prefill(wl, shape["S"], seed=shape["S"], device="cuda")
    cache = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=shape["S"])
    got = cache.window_logits(pre.K, pre.Q)
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    ref = reference_logits(wl, pre.K, pre.Q)
    # causal limit is not applied to logits; every entry must match the product
    err = (got - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= 2e-5 * max(1.0, scale) * math.sqrt(shape["d"] / 128), (err, scale)
