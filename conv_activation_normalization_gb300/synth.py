"""Seeded synthetic inputs for the four operator chains.

This module draws random numbers and nothing else: it holds none of the
operators' arithmetic, so both the CUDA path's tests and the fp64 oracle can
take their inputs from it.

Generator: numpy ``PCG64`` seeded per workload, arrays drawn as float32 in the
order listed in each recipe, so the same seed gives the same bits on x86 and
Arm.  Shapes and distributions follow the problem statements of the source
pages (POPCORNBENCH level-2 problems p37, p64, p5 and p60), which stand in for
that suite's own input generators; the suite's files are not used.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 20260000


def _rng(seed):
    return np.random.Generator(np.random.PCG64(int(seed)))


def _normal(rng, shape, std=1.0):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _uniform(rng, shape, lo, hi):
    a = rng.random(size=shape, dtype=np.float32)
    a *= np.float32(hi - lo)
    a += np.float32(lo)
    return a


def _draw_x(rng, shape, dist):
    if dist == "normal":
        return _normal(rng, shape)
    if dist == "uniform01":
        return _uniform(rng, shape, 0.0, 1.0)
    raise ValueError(dist)


def _draw_w(rng, shape, dist, bound):
    if dist == "default":
        return _uniform(rng, shape, -bound, bound)
    if dist == "normal":
        return _normal(rng, shape)
    if dist == "uniform01":
        return _uniform(rng, shape, 0.0, 1.0)
    raise ValueError(dist)


# --------------------------------------------------------------- recipes
@dataclasses.dataclass(frozen=True)
class LinearGNShape:
    """Linear(K->N) -> Swish -> +bias[N] -> GroupNorm(groups, N) on x[M, K]."""
    M: int = 32768
    K: int = 1024
    N: int = 4096
    groups: int = 64
    eps: float = 1e-5


def linear_gn_inputs(shape: LinearGNShape, seed: int, x_dist: str = "normal", w_dist: str = "default"):
    """x ~ N(0,1); W, b_lin ~ U(+-1/sqrt(K)); bias ~ N(0,1);
    gamma ~ U(0.5, 1.5); beta ~ N(0, 0.1).  Drawn in that order.

    Stress variants: ``x_dist="uniform01"`` draws x ~ U[0,1) (the torch.rand
    inputs that page Kimi-K2.6__l2_p37 reasons about in turn 1);
    ``w_dist="normal"`` draws W ~ N(0,1) (that page's other assumption in the
    same turn), ``w_dist="uniform01"`` W ~ U[0,1) (page Kimi-K2.6__l2_p64's
    all-uniform case, turn 1).  b_lin keeps its default distribution."""
    r = _rng(seed)
    bound = 1.0 / math.sqrt(shape.K)
    x = _draw_x(r, (shape.M, shape.K), x_dist)
    W = _draw_w(r, (shape.N, shape.K), w_dist, bound)
    b_lin = _uniform(r, (shape.N,), -bound, bound)
    bias = _normal(r, (shape.N,))
    gamma = _uniform(r, (shape.N,), 0.5, 1.5)
    beta = _normal(r, (shape.N,), 0.1)
    return dict(x=x, W=W, b_lin=b_lin, bias=bias, gamma=gamma, beta=beta)


@dataclasses.dataclass(frozen=True)
class LinearLSEShape:
    """Linear(K->N) -> logsumexp(dim 1) -> LeakyReLU x2 -> GELU x2 on x[M, K]."""
    M: int = 1024
    K: int = 8192
    N: int = 8192
    negative_slope: float = 0.01


def linear_lse_inputs(shape: LinearLSEShape, seed: int, bias_shift: float = 0.0, dist: str = "default"):
    """x ~ N(0,1); W, b ~ U(+-1/sqrt(K)), drawn in that order.  ``bias_shift``
    adds a constant to b (used to reach the negative LeakyReLU branch).

    ``dist="uniform01"`` draws x, W and b ~ U[0,1) instead: the all-uniform
    case page Kimi-K2.6__l2_p64 reasons about in turn 1, where every logit is
    a sum of K products of mean 1/4, so logsumexp lands in the thousands."""
    r = _rng(seed)
    bound = 1.0 / math.sqrt(shape.K)
    if dist == "default":
        x = _normal(r, (shape.M, shape.K))
        W = _uniform(r, (shape.N, shape.K), -bound, bound)
        b = _uniform(r, (shape.N,), -bound, bound)
    elif dist == "uniform01":
        x = _uniform(r, (shape.M, shape.K), 0.0, 1.0)
        W = _uniform(r, (shape.N, shape.K), 0.0, 1.0)
        b = _uniform(r, (shape.N,), 0.0, 1.0)
    else:
        raise ValueError(dist)
    if bias_shift:
        b += np.float32(bias_shift)
    return dict(x=x, W=W, b=b)


@dataclasses.dataclass(frozen=True)
class DConv1dShape:
    """LayerNorm([C, L]) -> GELU -> Conv1d(C->C, k, dilation, padding) -> +x."""
    B: int = 32
    C: int = 256
    L: int = 4096
    ksize: int = 3
    dilation: int = 4
    padding: int = 4
    eps: float = 1e-5


def dconv1d_inputs(shape: DConv1dShape, seed: int, affine: str = "default"):
    """x ~ N(0,1); conv W[C, C, k], b[C] ~ U(+-1/sqrt(C k)), drawn in that
    order.  LayerNorm affine: ``"default"`` gives PyTorch's initial gamma = 1,
    beta = 0; ``"perturbed"`` then draws gamma ~ U(0.5, 1.5) and
    beta ~ N(0, 0.1) of shape [C, L] so the affine path is exercised."""
    r = _rng(seed)
    fan = shape.C * shape.ksize
    bound = 1.0 / math.sqrt(fan)
    x = _normal(r, (shape.B, shape.C, shape.L))
    conv_w = _uniform(r, (shape.C, shape.C, shape.ksize), -bound, bound)
    conv_b = _uniform(r, (shape.C,), -bound, bound)
    if affine == "default":
        ln_gamma = np.ones((shape.C, shape.L), np.float32)
        ln_beta = np.zeros((shape.C, shape.L), np.float32)
    elif affine == "perturbed":
        ln_gamma = _uniform(r, (shape.C, shape.L), 0.5, 1.5)
        ln_beta = _normal(r, (shape.C, shape.L), 0.1)
    else:
        raise ValueError(affine)
    return dict(x=x, ln_gamma=ln_gamma, ln_beta=ln_beta, conv_w=conv_w, conv_b=conv_b)


@dataclasses.dataclass(frozen=True)
class ConvT3dShape:
    """ConvTranspose3d(Cin->Cout, k, stride, pad) -> Swish -> GroupNorm -> HardSwish."""
    N: int = 128
    Cin: int = 3
    Cout: int = 16
    D: int = 16
    H: int = 32
    W: int = 32
    k: int = 3
    stride: int = 2
    pad: int = 1
    groups: int = 4
    eps: float = 1e-5


def convt3d_inputs(shape: ConvT3dShape, seed: int, x_dist: str = "normal"):
    """x ~ N(0,1) (or U[0,1) with ``x_dist="uniform01"``); w[Cin, Cout, k, k, k],
    b[Cout] ~ U(+-1/sqrt(fan)) with fan = Cout k^3 (PyTorch's fan-in for the
    ConvTranspose weight layout); gamma ~ U(0.5, 1.5); beta ~ N(0, 0.1).
    Drawn in that order."""
    r = _rng(seed)
    fan = shape.Cout * shape.k ** 3
    bound = 1.0 / math.sqrt(fan)
    xs = (shape.N, shape.Cin, shape.D, shape.H, shape.W)
    if x_dist == "normal":
        x = _normal(r, xs)
    elif x_dist == "uniform01":
        x = _uniform(r, xs, 0.0, 1.0)
    else:
        raise ValueError(x_dist)
    w = _uniform(r, (shape.Cin, shape.Cout, shape.k, shape.k, shape.k), -bound, bound)
    b = _uniform(r, (shape.Cout,), -bound, bound)
    gamma = _uniform(r, (shape.Cout,), 0.5, 1.5)
    beta = _normal(r, (shape.Cout,), 0.1)
    return dict(x=x, w=w, b=b, gamma=gamma, beta=beta)


# ------------------------------------------------------- the five workloads
WORKLOADS = {
    # name: (recipe shape, seed)
    "linear_gn_m256": (LinearGNShape(M=256), SEED_BASE + 1),
    "linear_gn_m32768": (LinearGNShape(M=32768), SEED_BASE + 2),
    "linear_lse_m1024": (LinearLSEShape(), SEED_BASE + 3),
    "ln_dconv1d_b32": (DConv1dShape(), SEED_BASE + 4),
    "convt3d_n128": (ConvT3dShape(), SEED_BASE + 5),
}
