"""Seeded synthetic inputs for the k-means assignment step.

This module only draws numbers: it holds none of the method's arithmetic (no
norms, no scores, no argmin), so the CUDA path and the oracle can both be fed
from it without sharing any code that computes an answer.

Every generator draws fp32 values from a seeded ``torch.Generator`` on the CPU
and rounds them to bf16 with ``Tensor.to(torch.bfloat16)`` (round to nearest
even).  Both sides of a parity test consume the same bf16 bits.

The five workloads follow the shapes of the pages' benchmark (flashlib PR #22
"Optimize Blackwell k-means assignment reduction", Performance table: N from
65,536 to 1,048,576, D 64/128/256, K 512 to 16,384) and the value mixes this
library is specified against.  The pages give no value distributions for
their production shapes, so these synthetic sets stand in for them.
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    N: int
    D: int
    K: int
    seed: int
    kind: str
    precomputed_norms: bool
    integer: bool
    text: str


WORKLOADS = {
    "tiny_blobs": Workload(
        "tiny_blobs", 4096, 64, 128, 0, "blobs", False, False,
        "N=4,096, D=64, K=128: X from 128 isotropic Gaussian blobs (centers "
        "N(0,1), sigma 0.1); C = blob centers + N(0,0.01) noise; norms computed "
        "inside the step"),
    "sampled_centroids": Workload(
        "sampled_centroids", 65536, 128, 4096, 1, "sampled", True, False,
        "N=65,536, D=128, K=4,096: X from 4,096 Gaussian clusters (centers "
        "N(0,1), sigma 0.3, uniform labels); C = K rows of X drawn without "
        "replacement; fp32 norms precomputed"),
    "iid_normal": Workload(
        "iid_normal", 262144, 256, 16384, 2, "iid", False, False,
        "N=262,144, D=256, K=16,384: X and C iid N(0,1) (dense near-ties)"),
    "lognormal_clusters": Workload(
        "lognormal_clusters", 1048576, 128, 4096, 3, "lognormal", False, False,
        "N=1,048,576, D=128, K=4,096: 4,096 clusters (centers N(0,1)), sizes "
        "from LogNormal(0,1) weights, per-cluster scale U(0.1,1.0); C = centers "
        "+ N(0,0.05)"),
    "adversarial_ties": Workload(
        "adversarial_ties", 65536, 64, 16384, 4, "adversarial", False, True,
        "N=65,536, D=64, K=16,384: integers in [-4,4]; C[j] == C[j+K/2]; the "
        "first 128 unique centroids all equal (256 equal rows); 10% of X rows "
        "copy a centroid; 1% of X rows hold one NaN, +inf, -inf or -0.0"),
}

# Workloads in the order they are listed in the specification (1-based ids).
ORDER = ["tiny_blobs", "sampled_centroids", "iid_normal", "lognormal_clusters",
         "adversarial_ties"]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float32).to(torch.bfloat16).contiguous()


def blobs(N: int, K: int, D: int, seed: int):
    g = _gen(seed)
    centers = torch.randn(K, D, generator=g)
    labels = torch.randint(0, K, (N,), generator=g)
    X = centers[labels] + 0.1 * torch.randn(N, D, generator=g)
    C = centers + 0.01 * torch.randn(K, D, generator=g)
    return _bf16(X), _bf16(C)


def sampled(N: int, K: int, D: int, seed: int):
    if K > N:
        raise ValueError("sampled centroids need K <= N")
    g = _gen(seed)
    nclust = K
    centers = torch.randn(nclust, D, generator=g)
    labels = torch.randint(0, nclust, (N,), generator=g)
    X = _bf16(centers[labels] + 0.3 * torch.randn(N, D, generator=g))
    pick = torch.randperm(N, generator=g)[:K]
    C = X[pick].clone().contiguous()
    return X, C


def iid(N: int, K: int, D: int, seed: int):
    g = _gen(seed)
    X = torch.randn(N, D, generator=g)
    C = torch.randn(K, D, generator=g)
    return _bf16(X), _bf16(C)


def lognormal(N: int, K: int, D: int, seed: int):
    g = _gen(seed)
    centers = torch.randn(K, D, generator=g)
    weights = torch.exp(torch.randn(K, generator=g))          # LogNormal(0, 1)
    scale = 0.1 + 0.9 * torch.rand(K, generator=g)            # U(0.1, 1.0)
    labels = torch.multinomial(weights, N, replacement=True, generator=g)
    X = centers[labels] + scale[labels].unsqueeze(1) * torch.randn(N, D, generator=g)
    C = centers + 0.05 * torch.randn(K, D, generator=g)
    return _bf16(X), _bf16(C)


SPECIALS = (float("nan"), float("inf"), float("-inf"), -0.0)


def adversarial(N: int, K: int, D: int, seed: int, equal_rows: int = 128,
                copy_frac: float = 0.10, special_frac: float = 0.01):
    """Integer-valued tie/special-value workload.

    K must be even: centroid j and j + K/2 are identical, so every centroid
    has a twin in another part of the centroid range.  The first
    ``min(equal_rows, K/2)`` unique centroids are all equal.
    """
    if K % 2:
        raise ValueError("adversarial workload needs an even K")
    g = _gen(seed)
    half = K // 2
    U = torch.randint(-4, 5, (half, D), generator=g).to(torch.float32)
    ne = min(equal_rows, half)
    U[:ne] = U[0].clone()
    C = torch.cat([U, U], dim=0)
    X = torch.randint(-4, 5, (N, D), generator=g).to(torch.float32)
    ncopy = int(round(copy_frac * N))
    if ncopy:
        rows = torch.randperm(N, generator=g)[:ncopy]
        src = torch.randint(0, K, (ncopy,), generator=g)
        X[rows] = C[src]
    nspec = int(round(special_frac * N))
    if nspec:
        rows = torch.randperm(N, generator=g)[:nspec]
        dims = torch.randint(0, D, (nspec,), generator=g)
        kinds = torch.randint(0, len(SPECIALS), (nspec,), generator=g)
        for r, d, k in zip(rows.tolist(), dims.tolist(), kinds.tolist()):
            X[r, d] = SPECIALS[k]
    return _bf16(X), _bf16(C)


def integers(N: int, K: int, D: int, seed: int, lo: int = -4, hi: int = 4):
    """Integer-valued X and C in [lo, hi] (plenty of exact ties)."""
    g = _gen(seed)
    X = torch.randint(lo, hi + 1, (N, D), generator=g).to(torch.float32)
    C = torch.randint(lo, hi + 1, (K, D), generator=g).to(torch.float32)
    return _bf16(X), _bf16(C)


_KINDS = {"blobs": blobs, "sampled": sampled, "iid": iid, "lognormal": lognormal,
          "adversarial": adversarial}


def make(key: str, N: int | None = None, K: int | None = None, D: int | None = None,
         variant: int = 0):
    """Inputs of workload ``key`` (optionally at other sizes).

    ``variant`` selects one of the rotating input sets: seed + 1000 * variant.
    Variant 0 is the parity set.  Returns (X, C) as bf16 CPU tensors.
    """
    w = WORKLOADS[key]
    N = w.N if N is None else int(N)
    K = w.K if K is None else int(K)
    D = w.D if D is None else int(D)
    return _KINDS[w.kind](N, K, D, w.seed + 1000 * int(variant))


def bits(t: torch.Tensor):
    """bf16 CPU tensor -> numpy uint16 view of the same bits."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
