"""Seeded synthetic inputs for the DSpark per-step path.

This module only draws random numbers with the shapes, sizes and value
distributions of the workloads the DSpark pages describe.  It holds no step of
the method (no softmax, no sampling rule, no scheduler arithmetic): both the
CUDA library and the fp64 oracle consume what it returns, and neither imports
the other.

Workload model (from the DSpark pages' experiment settings: Qwen3 / DeepSeek
vocabularies, gamma = 4..16, hundreds to thousands of concurrent requests):

* target logits  z[r, j, v] ~ N(0, 3^2) - 1.1 * ln(v + 1)   (Zipf(1.1) log-prior
  over token ids), one independent row per verify position j = 0..gamma;
* draft base logits  U[r, k-1, v] = z[r, k-1, v] + s_r * (1 + 0.2 k) * N(0, 1)
  for draft positions k = 1..gamma (s_r = 1 except the DeepSeek-vocab workload,
  where s_r ~ U[0.5, 3] per request);
* W1, W2 ~ N(0, 0.02^2); confidence weight w ~ N(0, 0.05^2); h ~ N(0, 1);
* anchors uniform over the vocabulary; request ids 0..B-1;
* engine cost tables SPS as stated per workload.

The public benchmark suites the pages evaluate on are not used: these seeded
inputs stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

SCHED_OFF = 0
SCHED_GREEDY = 1
SCHED_ASYNC_TOPK = 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    H: int
    r: int
    dtype: str  # "f32" or "bf16"
    temp: str  # "1.0", "0.7", "0", "mixed" (even req_id greedy, odd 1.0)
    sched: int
    sps: str  # "tiny" (1000/(1+b/64)) or "exp2048" (60*(1-exp(-2048/b)))
    sts: Optional[tuple] = None  # (lo, hi) uniform per-position STS temperatures
    noise_scale: Optional[tuple] = None  # (lo, hi) per-request draft noise scale
    seed: int = 0


WORKLOADS = {
    # tiny oracle case
    "tiny": Workload("tiny", 4, 4, 1024, 64, 16, "f32", "mixed", SCHED_GREEDY, "tiny", seed=0),
    # Qwen3-4B-shaped step, scheduler off
    "qwen3_4b": Workload("qwen3_4b", 64, 7, 151936, 2560, 256, "bf16", "1.0", SCHED_OFF, "exp2048", seed=1),
    # Qwen3-8B-shaped step with scheduling and STS temperatures
    "qwen3_8b_sched": Workload("qwen3_8b_sched", 256, 15, 151936, 4096, 256, "bf16", "0.7",
                               SCHED_GREEDY, "exp2048", sts=(0.8, 1.5), seed=2),
    # high-concurrency DeepSeek-vocab step, half greedy
    "deepseek_vocab": Workload("deepseek_vocab", 1024, 7, 129280, 7168, 256, "bf16", "mixed",
                               SCHED_GREEDY, "exp2048", noise_scale=(0.5, 3.0), seed=3),
}


def sweep_point(B: int, gamma: int) -> Workload:
    """One point of the batch/gamma sweep (V=151936, r=256, bf16, T=1, scheduler on)."""
    return Workload(f"sweep_B{B}_g{gamma}", B, gamma, 151936, 4096, 256, "bf16", "1.0",
                    SCHED_GREEDY, "exp2048", seed=4)


# the bench's headline point: the sweep's B=256, gamma=7 point
HEADLINE = sweep_point(256, 7)


def get_workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep_B"):
        b, g = name[len("sweep_B"):].split("_g")
        return sweep_point(int(b), int(g))
    raise KeyError(name)


def sps_table(kind: str, B: int, gamma: int) -> np.ndarray:
    """Engine steps/s indexed by total verify tokens n (entries 0..B*(1+gamma)); entry 0 unused."""
    n = np.arange(B * (1 + gamma) + 1, dtype=np.float64)
    n[0] = 1.0
    if kind == "tiny":
        t = 1000.0 / (1.0 + n / 64.0)
    elif kind == "exp2048":
        t = 60.0 * (1.0 - np.exp(-2048.0 / n))
    else:
        raise ValueError(kind)
    t[0] = 0.0
    return t


def temperatures(kind: str, req_id: np.ndarray) -> np.ndarray:
    if kind == "mixed":
        return np.where(req_id % 2 == 0, 0.0, 1.0).astype(np.float32)
    return np.full(req_id.shape, float(kind), dtype=np.float32)


def _torch_dtype(d: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[d]


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None, temp: Optional[str] = None,
                sampling_seed: Optional[int] = None, with_target=True) -> dict:
    """Draw one step's inputs for workload `wl` on `device` (torch tensors).

    Returns a dict with U [B,g,V], W1 [V,r], W2 [r,V], h [B,g,H], w [H+r] (all in
    the workload dtype), anchor [B] i32, temp [B] f32, req_id [B] u32-as-i64,
    seed (python int), target [B,g+1,V] (workload dtype), sts [g] f32,
    sps [B(1+g)+1] f64 (numpy), sched mode.
    """
    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * seed + 12345)
    B, G, V, H, r = wl.B, wl.gamma, wl.V, wl.H, wl.r
    dt = _torch_dtype(wl.dtype)
    f32 = torch.float32
    logprior = -1.1 * torch.log(torch.arange(V, device=device, dtype=f32) + 1.0)
    out = {}
    tgt = torch.randn((B, G + 1, V), generator=g, device=device, dtype=f32)
    tgt.mul_(3.0).add_(logprior)
    if wl.noise_scale is not None:
        lo, hi = wl.noise_scale
        s_r = lo + (hi - lo) * torch.rand((B,), generator=g, device=device, dtype=f32)
    else:
        s_r = torch.ones((B,), device=device, dtype=f32)
    U = torch.empty((B, G, V), device=device, dtype=dt)
    for k in range(1, G + 1):
        noise = torch.randn((B, V), generator=g, device=device, dtype=f32)
        noise.mul_((s_r * (1.0 + 0.2 * k))[:, None]).add_(tgt[:, k - 1])
        U[:, k - 1].copy_(noise)
        del noise
    out["U"] = U
    if with_target:
        out["target"] = tgt.to(dt)
    del tgt
    out["W1"] = (0.02 * torch.randn((V, r), generator=g, device=device, dtype=f32)).to(dt)
    out["W2"] = (0.02 * torch.randn((r, V), generator=g, device=device, dtype=f32)).to(dt)
    out["h"] = torch.randn((B, G, H), generator=g, device=device, dtype=f32).to(dt)
    out["w"] = (0.05 * torch.randn((H + r,), generator=g, device=device, dtype=f32)).to(dt)
    out["anchor"] = torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    req = np.arange(B, dtype=np.int64)
    out["req_id"] = torch.from_numpy(req.astype(np.int32)).to(device)
    out["temp"] = torch.from_numpy(temperatures(temp or wl.temp, req)).to(device)
    if wl.sts is not None:
        lo, hi = wl.sts
        sts = lo + (hi - lo) * torch.rand((G,), generator=g, device=device, dtype=f32)
    else:
        sts = torch.ones((G,), device=device, dtype=f32)
    out["sts"] = sts
    out["sps"] = sps_table(wl.sps, B, G)
    out["sched"] = wl.sched
    out["seed"] = int(0x5EED_0000_0000 + 7919 * seed) if sampling_seed is None else int(sampling_seed)
    return out


def random_conf_logits(B: int, gamma: int, seed: int, scale: float = 2.5, shift: float = 0.5) -> np.ndarray:
    """fp32 confidence logits ~ N(shift, scale^2) for scheduler-only cases."""
    rng = np.random.default_rng(seed)
    return (shift + scale * rng.standard_normal((B, gamma))).astype(np.float32)


def random_tokens(B: int, gamma: int, V: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, V, size=(B, gamma), dtype=np.int64).astype(np.int32)


# ---------------------------------------------------------------------------
# held-out blocks for fitting the STS temperatures
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class StsWorkload:
    name: str
    N: int          # held-out draft blocks
    gamma: int
    n_grid: int     # candidate temperatures, geometric between grid_lo and grid_hi
    n_bins: int
    grid_lo: float = 0.25
    grid_hi: float = 4.0
    seed: int = 0


STS_WORKLOADS = {
    # small case the oracle finishes in seconds
    "sts_small": StsWorkload("sts_small", 3000, 5, 24, 15, seed=11),
    # held-out set of a production-sized calibration run
    "sts_N131072_g7_G128_M15": StsWorkload("sts_N131072_g7_G128_M15", 131072, 7, 128, 15, seed=12),
}


def sts_grid(n_grid: int, lo: float = 0.25, hi: float = 4.0) -> np.ndarray:
    """fp32 candidate temperatures, geometric from lo to hi (one value: lo)."""
    if n_grid == 1:
        return np.array([lo], np.float32)
    return np.geomspace(lo, hi, n_grid).astype(np.float32)


def sts_heldout(N: int, gamma: int, seed: int, kappa=None, mu0: float = 2.2, mu_step: float = 0.25,
                spread: float = 1.5, noise: float = 0.0):
    """Held-out draft blocks with a known calibration.

    Data model: the chance that draft position k is accepted, given that the
    positions before it were, is q = 1 / (1 + exp(-u)) with u ~ N(mu0 -
    mu_step (k-1), spread^2); a block's accept length is the number of leading
    accepted positions drawn that way.  The confidence head reports the
    over-confident logit z = kappa_k u (+ noise N(0, noise^2)), so that the
    temperature kappa_k calibrates position k exactly when noise = 0.
    Returns (conf_logit [N, gamma] float32, accept_len [N] int32, kappa [gamma])."""
    rng = np.random.default_rng(seed)
    if kappa is None:  # raw ECE of 4-8 % falling to about 1 % after fitting, as the pages report
        kappa = 1.3 + 0.05 * np.arange(gamma)
    kappa = np.asarray(kappa, dtype=np.float64)
    mu = mu0 - mu_step * np.arange(gamma)
    u = mu[None, :] + spread * rng.standard_normal((N, gamma))
    q = 1.0 / (1.0 + np.exp(-u))
    acc = rng.random((N, gamma)) < q
    accept_len = np.cumprod(acc, axis=1).sum(axis=1).astype(np.int32)
    z = kappa[None, :] * u + noise * rng.standard_normal((N, gamma))
    return z.astype(np.float32), accept_len, kappa


def sts_inputs(wl: StsWorkload, noise: float = 0.6):
    """conf_logit, accept_len and grid of a held-out workload (the head is noisy:
    its discrimination is imperfect, as the pages' ROC-AUC of 0.81-0.90 says)."""
    z, L, kappa = sts_heldout(wl.N, wl.gamma, wl.seed, noise=noise)
    return dict(conf_logit=z, accept_len=L, grid=sts_grid(wl.n_grid, wl.grid_lo, wl.grid_hi),
                n_bins=wl.n_bins, kappa=kappa)


def rnn_weights(r: int, H: int, dtype: str, seed: int, device="cpu", gain: float = 1.5) -> torch.Tensor:
    """W_rnn [3r, 2r + H] (rows W_g, W_c, W_o) of the RNN head, N(0, gain^2 / (2r + H)):
    pre-activations of order gain for unit-scale inputs."""
    g = torch.Generator(device="cpu").manual_seed(7700 + seed)
    K = 2 * r + H
    w = gain / math.sqrt(K) * torch.randn((3 * r, K), generator=g, dtype=torch.float32)
    return w.to(_torch_dtype(dtype)).to(device)
