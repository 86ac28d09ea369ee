"""Seeded synthetic workloads for the EP dispatch / combine path.

This module only draws inputs: routings (top-k expert ids, top-k weights)
and bf16 payloads.  It holds none of the method's arithmetic and imports
neither the CUDA binding nor the CPU oracle, so both sides can be fed the
same bytes.

Routing integers are drawn on the host with numpy (``default_rng`` seeded per
(workload seed, field)).  Large bf16 payloads are drawn with torch's seeded
generator on the requested device (on a GPU for the full-size workloads,
where a host draw of several GB would take minutes); either way the tensor a
test hands to the oracle is the very tensor the kernels read.

The five named workloads follow the DeepSeek-V3-like shapes the EP pages use
(hidden 7168, 256 experts, top-8) plus one small case:

  ``normal_small``   R=8,  T=256,  H=1024, E=32,  K=4, uniform routing
  ``normal_v3``      R=8,  T=4096, H=7168, E=256, K=8, N(0,1) logits + Gumbel
                     noise per (token, expert), weights = softmax of the
                     chosen logits, expert_alignment 128
  ``fp8_zipf``       R=16, T=4096, H=7168, E=256, K=8, Zipf(1.2) expert
                     popularity over a seeded permutation, 5% of slots
                     masked, 1% outlier channels scaled x50
  ``ll_v3``          R=32, T=128 (max 128), H=7168, E=256, K=8 uniform
  ``combine_heavy``  R=16, T=4096, H=7168, E=256, K=8 uniform, two
                     N(0, 0.1) bias tensors, ten fresh expert outputs
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    R: int          # virtual ranks
    T: int          # tokens per rank
    H: int          # hidden size
    E: int          # experts
    K: int          # top-k
    routing: str    # uniform | gumbel | zipf
    C: int = 12     # channels (num_sms / 2 with the pages' test setting of 24 SMs)
    A: int = 1      # expert_alignment
    max_tokens: int = 0   # low-latency num_max_dispatch_tokens_per_rank (0 = T)
    mask_p: float = 0.0   # probability that a top-k slot is masked (-1)
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    n_combines: int = 1
    bias_std: float = 0.0
    seed: int = 0

    @property
    def EL(self) -> int:
        return self.E // self.R

    def scaled(self, T: int | None = None, H: int | None = None, R: int | None = None,
               E: int | None = None) -> "Shape":
        """Same recipe at another size (parity tests at sizes the oracle finishes in seconds)."""
        R2 = R or self.R
        E2 = E or self.E
        T2 = T if T is not None else self.T
        mt = self.max_tokens and max(T2, 1)
        return dataclasses.replace(self, T=T2, H=H or self.H, R=R2, E=E2, max_tokens=mt,
                                   name=f"{self.name}@R{R2}T{T2}H{H or self.H}E{E2}")


WORKLOADS = {
    "normal_small": Shape("normal_small", R=8, T=256, H=1024, E=32, K=4, routing="uniform", seed=1001),
    "normal_v3": Shape("normal_v3", R=8, T=4096, H=7168, E=256, K=8, routing="gumbel", A=128, seed=1002),
    "fp8_zipf": Shape("fp8_zipf", R=16, T=4096, H=7168, E=256, K=8, routing="zipf", mask_p=0.05,
                      outlier_frac=0.01, outlier_scale=50.0, seed=1003),
    "ll_v3": Shape("ll_v3", R=32, T=128, H=7168, E=256, K=8, routing="uniform", max_tokens=128, seed=1004),
    "combine_heavy": Shape("combine_heavy", R=16, T=4096, H=7168, E=256, K=8, routing="uniform",
                           n_combines=10, bias_std=0.1, seed=1005),
}


def _seed(seed: int, field: str) -> int:
    h = hashlib.sha256(f"{seed}/{field}".encode()).digest()
    return int.from_bytes(h[:8], "little") & 0x7FFF_FFFF_FFFF_FFFF


def rng(seed: int, field: str) -> np.random.Generator:
    return np.random.default_rng(_seed(seed, field))


def _topk_by_score(score: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K largest scores per row, slots ordered by descending score
    (ties to the lower expert id)."""
    part = np.argpartition(-score, K - 1, axis=1)[:, :K]
    vals = np.take_along_axis(score, part, axis=1)
    order = np.lexsort((part, -vals), axis=1)
    return np.take_along_axis(part, order, axis=1)


def routing(shape: Shape):
    """Top-k expert ids [R][T][K] int64 (-1 = masked slot) and weights [R][T][K] float32."""
    R, T, E, K = shape.R, shape.T, shape.E, shape.K
    n = R * T
    g = rng(shape.seed, "routing")
    if n == 0:
        return np.zeros((R, T, K), np.int64), np.zeros((R, T, K), np.float32)
    if shape.routing == "uniform":
        idx = _topk_by_score(g.random((n, E)), K)
        logits = rng(shape.seed, "weights").standard_normal((n, K)).astype(np.float32)
    elif shape.routing == "gumbel":
        logits_all = g.standard_normal((n, E)).astype(np.float32)
        score = logits_all + g.gumbel(size=(n, E)).astype(np.float32)
        idx = _topk_by_score(score, K)
        logits = np.take_along_axis(logits_all, idx, axis=1)
    elif shape.routing == "zipf":
        perm = rng(shape.seed, "zipf_perm").permutation(E)
        p = (np.arange(E, dtype=np.float64) + 1.0) ** -1.2
        logp = np.empty(E)
        logp[perm] = np.log(p / p.sum())
        score = logp[None, :] + g.gumbel(size=(n, E))
        idx = _topk_by_score(score, K)
        logits = rng(shape.seed, "weights").standard_normal((n, K)).astype(np.float32)
    else:
        raise ValueError(shape.routing)
    ex = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    idx = idx.astype(np.int64)
    if shape.mask_p > 0:
        m = rng(shape.seed, "mask").random((n, K)) < shape.mask_p
        idx[m] = -1
    return idx.reshape(R, T, K), w.reshape(R, T, K)


def normal_bf16(shape_tuple, seed: int, field: str, device="cpu", std: float = 1.0,
                outlier_channels=None, outlier_scale: float = 1.0) -> torch.Tensor:
    """N(0, std^2) values rounded to bf16 (torch's seeded generator on `device`)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(_seed(seed, field))
    v = torch.randn(shape_tuple, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    if outlier_channels is not None and len(outlier_channels):
        ch = torch.as_tensor(outlier_channels, device=device, dtype=torch.long)
        v[..., ch] *= outlier_scale
    return v.to(torch.bfloat16)


def outlier_channels(shape: Shape) -> np.ndarray:
    n = int(round(shape.outlier_frac * shape.H))
    if n == 0:
        return np.zeros(0, np.int64)
    return np.sort(rng(shape.seed, "outliers").choice(shape.H, size=n, replace=False)).astype(np.int64)


def tokens_x(shape: Shape, device="cpu") -> torch.Tensor:
    """Source token rows x [R][T][H] bf16."""
    return normal_bf16((shape.R, shape.T, shape.H), shape.seed, "x", device,
                       outlier_channels=outlier_channels(shape), outlier_scale=shape.outlier_scale)


def biases(shape: Shape, device="cpu"):
    """bias_0, bias_1 [R][T][H] bf16 ~ N(0, bias_std^2), or (None, None)."""
    if shape.bias_std <= 0:
        return None, None
    return (normal_bf16((shape.R, shape.T, shape.H), shape.seed, "bias0", device, std=shape.bias_std),
            normal_bf16((shape.R, shape.T, shape.H), shape.seed, "bias1", device, std=shape.bias_std))


def expert_outputs(shape: Shape, rows: int, i: int = 0, device="cpu") -> torch.Tensor:
    """Fresh expert outputs for combine number i: [rows][H] bf16 ~ N(0, 1)."""
    return normal_bf16((rows, shape.H), shape.seed + 7919 * (i + 1), "y", device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_tokens(shape: Shape, n: int, field: str = "sample") -> np.ndarray:
    """n distinct flat token ids s*T+t (sorted), always including the first and last."""
    total = shape.R * shape.T
    if total == 0:
        return np.zeros(0, np.int64)
    if n >= total:
        return np.arange(total, dtype=np.int64)
    pick = rng(shape.seed, field).choice(total, size=n, replace=False)
    pick = np.union1d(pick, [0, total - 1])
    return pick.astype(np.int64)
