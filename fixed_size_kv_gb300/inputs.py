"""Seeded synthetic workloads and input generators.

Shared by the tests (for both the CUDA library and the CPU oracle) and by the
benchmark.  This module holds no arithmetic of the method: it only draws
tensors and describes the workload shapes.

Workload shapes follow the SnapStream pages: Llama-3.1-8B (GQA, 32 query / 8 KV
heads of width 128) and DeepSeek-R1 (MLA: 128 query heads over one latent of
width 512 plus a 64-wide rope key), 128k context, the DeepSeek recent window of
31,744 tokens (episode companion page, "Reasoning Benchmarks Never Trigger
Decode Eviction (Table III)") and a 4x smaller cache at 128k ("4.0x lower KV
memory").  The pages publish no data: every tensor here is iid N(0,1) rounded
to bf16, and 1% of each KV head's prefix keys are "heavy hitters", shifted by
gamma * sqrt(d) along the mean direction of that head's window queries.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAVY_FRACTION = 0.01
HEAVY_GAMMA = 3.0


@dataclass(frozen=True)
class Workload:
    name: str
    layout: int            # 0 GQA, 1 MLA
    n_q_heads: int
    n_kv_heads: int
    d_qk: int
    d_v: int
    L_sink: int
    K: int
    L_recent: int
    W: int
    P: int
    batch: int
    prompt_min: int
    prompt_max: int
    decode_steps: int
    sm_scale: float
    arrival_every: int = 0   # >0: continuous batch with arrivals every this many steps
    notes: str = ""

    @property
    def G(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def C(self) -> int:
        return self.L_sink + self.K + self.L_recent

    def config_kwargs(self) -> dict:
        return dict(layout=self.layout, n_q_heads=self.n_q_heads, n_kv_heads=self.n_kv_heads,
                    d_qk=self.d_qk, d_v=self.d_v, L_sink=self.L_sink, K=self.K,
                    L_recent=self.L_recent, W=self.W, P=self.P, sm_scale=self.sm_scale)

    def replace(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


GQA_SCALE = 1.0 / math.sqrt(128.0)
# MLA: q.k runs over the 128-wide no-rope part plus the 64-wide rope part per head
# before absorption (DeepSeek-V2), so the scale is 1/sqrt(192).
MLA_SCALE = 1.0 / math.sqrt(192.0)

WORKLOADS = {
    "gqa_2k_tiny": Workload("gqa_2k_tiny", 0, 32, 8, 128, 128, 4, 252, 256, 32, 7,
                            batch=1, prompt_min=2048, prompt_max=2048, decode_steps=64,
                            sm_scale=GQA_SCALE,
                            notes="Llama-3.1-8B GQA single layer, one 2048-token prompt, cache 512"),
    "gqa_16k32k_b8": Workload("gqa_16k32k_b8", 0, 32, 8, 128, 128, 4, 2044, 2048, 64, 7,
                              batch=8, prompt_min=16384, prompt_max=32768, decode_steps=256,
                              sm_scale=GQA_SCALE,
                              notes="continuous batch of 8, prompts U[16k,32k], cache 4096"),
    "gqa_128k_b16": Workload("gqa_128k_b16", 0, 32, 8, 128, 128, 4, 16380, 16384, 64, 7,
                             batch=16, prompt_min=131072, prompt_max=131072, decode_steps=512,
                             sm_scale=GQA_SCALE,
                             notes="batch 16 at 128k context, cache 32768 (4x smaller)"),
    "mla_128k_b8": Workload("mla_128k_b8", 1, 128, 1, 576, 512, 64, 960, 31744, 64, 7,
                            batch=8, prompt_min=131072, prompt_max=131072, decode_steps=512,
                            sm_scale=MLA_SCALE,
                            notes="DeepSeek-R1 MLA latent, batch 8 at 128k, cache 32768"),
    "gqa_mixed_b64": Workload("gqa_mixed_b64", 0, 32, 8, 128, 128, 4, 4092, 4096, 64, 7,
                              batch=64, prompt_min=4096, prompt_max=131072, decode_steps=2048,
                              sm_scale=GQA_SCALE, arrival_every=32,
                              notes="64-slot continuous batch, prompts U[4k,128k], cache 8192"),
}


def _gen(seed: int, *tags: int, device="cpu") -> torch.Generator:
    """A generator whose seed mixes the workload seed with integer tags."""
    s = seed & 0xFFFFFFFF
    for t in tags:
        s = (s * 1000003 + (t & 0xFFFFFFFF) + 0x9E3779B9) & 0xFFFFFFFFFFFF
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def prompt_lengths(wl: Workload, seed: int, n: int | None = None, tag: int = 0) -> list[int]:
    """Seeded prompt lengths, uniform integers in [prompt_min, prompt_max]."""
    n = wl.batch if n is None else n
    if wl.prompt_min == wl.prompt_max:
        return [wl.prompt_min] * n
    g = _gen(seed, 17, tag)
    return torch.randint(wl.prompt_min, wl.prompt_max + 1, (n,), generator=g).tolist()


def output_lengths(seed: int, n: int, tag: int = 0, lo: int = 32, hi: int = 1024) -> list[int]:
    """Seeded decode lengths of continuous-batch requests, uniform in [lo, hi]."""
    g = _gen(seed, 23, tag)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


@dataclass
class Prefill:
    K: torch.Tensor            # bf16 [S][H_kv][d_qk]
    V: torch.Tensor | None     # bf16 [S][H_kv][d_v] (GQA) or None (MLA)
    Q: torch.Tensor            # bf16 [W][H_q][d_qk]  observation-window queries
    heavy: torch.Tensor        # int64 [H_kv][n_heavy] planted positions
    extra: dict = field(default_factory=dict)


def gen_prefill(wl: Workload, S: int, seed: int, seq: int = 0, device="cpu",
                heavy_fraction: float = HEAVY_FRACTION, gamma: float = HEAVY_GAMMA) -> Prefill:
    """Prefill K/V of one sequence plus its observation-window queries."""
    g = _gen(seed, 101, seq, device=device)
    Hq, Hkv, dk, dv, W = wl.n_q_heads, wl.n_kv_heads, wl.d_qk, wl.d_v, wl.W
    Q = _randn((W, Hq, dk), g, device).to(torch.bfloat16)
    K = _randn((S, Hkv, dk), g, device)
    V = _randn((S, Hkv, dv), g, device).to(torch.bfloat16) if wl.layout == 0 else None
    n_prefix = max(S - W, 0)
    n_heavy = int(math.floor(heavy_fraction * n_prefix))
    heavy = torch.zeros((Hkv, n_heavy), dtype=torch.int64, device=device)
    if n_heavy > 0 and gamma != 0.0:
        Qf = Q.float().view(W, Hkv, wl.G, dk)
        for h in range(Hkv):
            qbar = Qf[:, h].reshape(-1, dk).mean(dim=0)
            u = qbar / qbar.norm().clamp_min(1e-12) * math.sqrt(dk)
            pos = torch.randperm(n_prefix, generator=g, device=device)[:n_heavy]
            heavy[h] = pos
            K[pos, h, :] += gamma * u
    return Prefill(K=K.to(torch.bfloat16), V=V, Q=Q, heavy=heavy)


def gen_prompt_queries(wl: Workload, pre: Prefill, seed: int, seq: int = 0, device="cpu") -> torch.Tensor:
    """Queries of every prompt position, bf16 [S][H_q][d_qk], for the prefill attention:
    fresh N(0,1) rows for positions 0 .. S-W-1 and the prefill's observation-window
    queries (pre.Q) for the last W positions."""
    S = pre.K.shape[0]
    g = _gen(seed, 307, seq, device=device)
    Q = _randn((S, wl.n_q_heads, wl.d_qk), g, device).to(torch.bfloat16)
    W = min(wl.W, S)
    Q[S - W:] = pre.Q[wl.W - W:].to(device)
    return Q


@dataclass
class DecodeToken:
    q: torch.Tensor            # bf16 [n][H_q][d_qk]
    k: torch.Tensor            # bf16 [n][H_kv][d_qk]
    v: torch.Tensor | None     # bf16 [n][H_kv][d_v] (GQA) or None


def gen_decode(wl: Workload, n: int, step: int, seed: int, device="cpu") -> DecodeToken:
    """Fresh N(0,1) query / key / value of one decode step for n sequences."""
    g = _gen(seed, 211, step, device=device)
    q = _randn((n, wl.n_q_heads, wl.d_qk), g, device).to(torch.bfloat16)
    k = _randn((n, wl.n_kv_heads, wl.d_qk), g, device).to(torch.bfloat16)
    v = (_randn((n, wl.n_kv_heads, wl.d_v), g, device).to(torch.bfloat16)
         if wl.layout == 0 else None)
    return DecodeToken(q=q, k=k, v=v)
