"""Seeded synthetic inputs for the five tovl workloads.

This module holds random-number recipes only: no gather, scatter, plan,
counter or contraction arithmetic.  Both the CUDA path's tests/benchmark and
the CPU oracle consume the tensors it returns, so the two sides always see the
same bytes.

Recipes (the pages fix only shapes and the popularity law; the rest is the
plain reading):
  * activations and weights: N(0, 1) scaled by 1/sqrt(K), rounded to bf16
    by torch's round-to-nearest-even conversion;
  * uniform top-k routing: k distinct experts per token, uniformly at random;
  * Zipf(s) top-k routing: expert e has popularity (e+1)^-s; k distinct
    experts per token by Gumbel-top-k, which is sequential weighted sampling
    without replacement;
  * permuted copy: a uniform random permutation of the rows and random bytes.
Routings and permutations come from numpy's PCG64; tensors from torch's
generator on the requested device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


# ---------------------------------------------------------------- configs
@dataclass(frozen=True)
class GatherCfg:
    name: str
    shards: int
    rows_per_shard: int
    K: int
    N: int
    rounds: int
    seed: int = 0

    @property
    def M(self) -> int:
        return self.shards * self.rows_per_shard

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


@dataclass(frozen=True)
class DispatchCfg:
    name: str
    T: int
    H: int
    k: int
    E: int
    N: int
    routing: str          # "uniform" or "zipf"
    zipf_s: float = 0.0
    rounds: int = 10
    seed: int = 0


@dataclass(frozen=True)
class CopyCfg:
    name: str
    n_rows: int
    row_bytes: int
    rounds: int
    seed: int = 0
    row_sizes: tuple = field(default=(256, 512, 1024, 2048, 4096, 8192, 16384))


TINY = GatherCfg("tiny gated all-gather+GEMM: 2 shards x 128 rows, K=512, N=256",
                 shards=2, rows_per_shard=128, K=512, N=256, rounds=3)
TP = GatherCfg("all-gather+GEMM (TP shape): 4 shards x 768 rows, M=3072, K=4096, N=4096",
               shards=4, rows_per_shard=768, K=4096, N=4096, rounds=20)
DISPATCH = DispatchCfg("dispatch+grouped GEMM: T=4096, H=4096, top-2 uniform over 8 experts, N=2048",
                       T=4096, H=4096, k=2, E=8, N=2048, routing="uniform", rounds=10)
SKEWED = DispatchCfg("skewed dispatch: T=8192, H=7168, top-4 Zipf(1.2) over 32 experts, N=2048",
                     T=8192, H=7168, k=4, E=32, N=2048, routing="zipf", zipf_s=1.2, rounds=10)
COPY = CopyCfg("gated copy sweep: 2^20 rows permuted, 64-row chunks", n_rows=1 << 20,
               row_bytes=8192, rounds=1000)


def round_seed(seed: int, r: int) -> int:
    """Per-round seed: inputs change every round so a stale read of the
    previous round cannot pass a parity check."""
    return seed * 1000 + r


# ---------------------------------------------------------------- tensors
def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def bf16_normal(shape, scale: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) * scale rounded to bf16 (contiguous)."""
    g = _gen(device, seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(scale)
    return t.to(torch.bfloat16)


def random_bytes(n_rows: int, row_bytes: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed)
    return torch.randint(0, 256, (n_rows, row_bytes), generator=g, device=device, dtype=torch.uint8)


def gather_inputs(cfg: GatherCfg, seed: int, device="cpu"):
    """Shards [S][R][K] and weight W [K][N], both bf16 ~ N(0,1)/sqrt(K)."""
    s = 1.0 / math.sqrt(cfg.K)
    X = bf16_normal((cfg.shards, cfg.rows_per_shard, cfg.K), s, seed, device)
    W = bf16_normal((cfg.K, cfg.N), s, seed + 7919, device)
    return X, W


def dispatch_inputs(cfg: DispatchCfg, seed: int, device="cpu"):
    """Tokens x [T][H], routing topk [T][k] (int32), expert weights [E][H][N]."""
    s = 1.0 / math.sqrt(cfg.H)
    x = bf16_normal((cfg.T, cfg.H), s, seed, device)
    W = bf16_normal((cfg.E, cfg.H, cfg.N), s, seed + 7919, device)
    topk = routing(cfg, seed)
    return x, topk, W


# ---------------------------------------------------------------- routing
def uniform_topk(T: int, k: int, E: int, seed: int) -> np.ndarray:
    """k distinct experts per token, uniformly at random (int32 [T][k])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def zipf_topk(T: int, k: int, E: int, s: float, seed: int) -> np.ndarray:
    """k distinct experts per token, popularity (e+1)^-s, Gumbel-top-k."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    g = rng.gumbel(size=(T, E))
    return np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :k].astype(np.int32)


def routing(cfg: DispatchCfg, seed: int) -> np.ndarray:
    if cfg.routing == "uniform":
        return uniform_topk(cfg.T, cfg.k, cfg.E, seed)
    if cfg.routing == "zipf":
        return zipf_topk(cfg.T, cfg.k, cfg.E, cfg.zipf_s, seed)
    raise ValueError(cfg.routing)


def gate_weights(T: int, k: int, seed: int) -> np.ndarray:
    """Router gate weights of the k chosen experts: softmax of N(0,1) logits
    over each token's k choices (fp32 [T][k], rows sum to 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = rng.standard_normal((T, k))
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def repeated_topk(T: int, k: int, E: int, seed: int) -> np.ndarray:
    """k experts per token drawn uniformly WITH replacement (int32 [T][k]):
    k may exceed E and a token may name one expert several times."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, E, size=(T, k), dtype=np.int32)


def all_to_one_topk(T: int, E: int, e: int = 0) -> np.ndarray:
    """Degenerate routing: every token to expert e (k = 1)."""
    return np.full((T, 1), e, np.int32)


def permutation(n: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.permutation(n).astype(np.int32)


# ---------------------------------------------------------------- helpers
def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
