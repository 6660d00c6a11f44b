"""Seeded synthetic inputs for the compensated FP4 linear layer.

This module only draws random numbers: it holds none of the quantization or
GEMM arithmetic, and both the CUDA path and the CPU oracle consume what it
returns.  The ResServe paper times its linear kernels on "shared synthetic
BF16 inputs and weights" without naming a distribution (App. C.1, "Kernel
Timing"), and its precision cohorts use captured model activations that are
not available here; the distributions below stand in for both.  Each recipe
is an activation matrix X [M][K] and a weight W [N][K] (nn.Linear layout),
drawn in fp32 with numpy's PCG64 and rounded to bf16 (round to nearest even).

Recipes (name -> shapes and distributions):

* ``gauss_outlier_k2048``: M=1, K=N=2048.  X ~ N(0,1) with 8 channels chosen
  uniformly without replacement scaled by 20; W ~ N(0, 0.02^2).
* ``attn_proj_k4096``: M in {1,2,4,8}, K=N=4096.  X = Student-t(nu=4) per
  element times one LogNormal(0,1) factor per channel (column); W ~ N(0,0.02^2).
* ``mlp_gate_up`` / ``mlp_down``: M=8; gate/up K=4096, N=28672 (fused);
  down K=14336, N=4096.  X = Student-t(nu=3) with 8 channels scaled by 20;
  W ~ N(0, 0.015^2).  The two GEMMs draw independent X (the activation
  function between them is not part of the linear layer).
* ``mx_k5120_n27648``: M in {1,4,8,16,32,64,128}, K=5120, N=27648.
  X ~ N(0,1) with 1% of channels (51) scaled by 30; W ~ N(0, 0.02^2).
* ``prefill_k8192``: M=4096, K=N=8192.  X as ``attn_proj_k4096``;
  W ~ N(0, 0.01^2).
* ``attn_decode`` (``make_attention``): decode-attention query, keys and
  values; see that function.
* ``proj_shapes``: the 22 projection shapes (N, K) of the paper's per-shape
  M-Ext latency figures (ResServe Fig. 18 NVFP4, Fig. 19 MXFP4; QKV, output,
  gate/up and down projections of several models at TP1 / TP8), listed in
  ``PROJECTION_SHAPES``, M in {1, 8, 64, 512}.  X as ``attn_proj_k4096``;
  W ~ N(0, 0.02^2); N and K given per call.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Recipe:
    name: str
    K: int
    N: int
    x_kind: str          # "gauss_outlier" | "t_lognormal" | "t_outlier"
    x_params: tuple
    w_sigma: float
    seed: int


RECIPES = {
    "gauss_outlier_k2048": Recipe("gauss_outlier_k2048", 2048, 2048,
                                  "gauss_outlier", (8, 20.0), 0.02, 0),
    "attn_proj_k4096": Recipe("attn_proj_k4096", 4096, 4096,
                              "t_lognormal", (4.0,), 0.02, 0),
    "mlp_gate_up": Recipe("mlp_gate_up", 4096, 28672, "t_outlier", (3.0, 8, 20.0), 0.015, 0),
    "mlp_down": Recipe("mlp_down", 14336, 4096, "t_outlier", (3.0, 8, 20.0), 0.015, 2),
    "mx_k5120_n27648": Recipe("mx_k5120_n27648", 5120, 27648,
                              "gauss_outlier", (51, 30.0), 0.02, 0),
    "prefill_k8192": Recipe("prefill_k8192", 8192, 8192, "t_lognormal", (4.0,), 0.01, 0),
    "proj_shapes": Recipe("proj_shapes", 4096, 4096, "t_lognormal", (4.0,), 0.02, 5),
}

# (N, K) of the 22 projection shapes timed per shape in ResServe Fig. 18 / 19,
# in increasing N * K.
PROJECTION_SHAPES = tuple(sorted([
    (6144, 2560), (2560, 4096), (19456, 2560), (2560, 9728),
    (6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288),
    (10240, 5120), (5120, 8192), (51200, 5120), (5120, 25600),
    (14336, 5120), (34816, 5120), (5120, 17408), (16384, 5120),
    (5120, 6144), (4608, 8192), (8192, 2048), (8192, 1024),
    (2304, 8192), (2560, 8192),
], key=lambda nk: (nk[0] * nk[1], nk)))


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, tag]))


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """fp32 numpy array -> bf16 torch CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit pattern of a bf16 CPU tensor (the oracle's input form)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def activations(kind: str, params: tuple, M: int, K: int, rng: np.random.Generator,
                channel_rng: np.random.Generator) -> np.ndarray:
    """fp32 X [M][K].  Channel-level draws (outlier channels, per-channel
    scales) come from ``channel_rng`` so that they do not depend on M."""
    if kind == "gauss_outlier":
        n_out, factor = params
        x = rng.standard_normal((M, K), dtype=np.float32)
        ch = channel_rng.choice(K, size=int(n_out), replace=False)
        x[:, ch] *= np.float32(factor)
        return x
    if kind == "t_lognormal":
        (df,) = params
        x = rng.standard_t(df, size=(M, K)).astype(np.float32)
        scale = channel_rng.lognormal(0.0, 1.0, size=K).astype(np.float32)
        return x * scale[None, :]
    if kind == "t_outlier":
        df, n_out, factor = params
        x = rng.standard_t(df, size=(M, K)).astype(np.float32)
        ch = channel_rng.choice(K, size=int(n_out), replace=False)
        x[:, ch] *= np.float32(factor)
        return x
    raise ValueError(f"unknown activation kind {kind!r}")


def make_x(recipe: str | Recipe, M: int, K: int | None = None, seed: int | None = None
           ) -> torch.Tensor:
    """bf16 X [M][K] for a recipe (K defaults to the recipe's)."""
    r = RECIPES[recipe] if isinstance(recipe, str) else recipe
    K = r.K if K is None else K
    s = r.seed if seed is None else seed
    x = activations(r.x_kind, r.x_params, M, K, _rng(s, 1), _rng(s, 2))
    return to_bf16(x)


def make_w(recipe: str | Recipe, N: int | None = None, K: int | None = None,
           seed: int | None = None) -> torch.Tensor:
    """bf16 W [N][K] ~ N(0, sigma^2) for a recipe."""
    r = RECIPES[recipe] if isinstance(recipe, str) else recipe
    N = r.N if N is None else N
    K = r.K if K is None else K
    s = r.seed if seed is None else seed
    w = _rng(s, 3).standard_normal((N, K), dtype=np.float32) * np.float32(r.w_sigma)
    return to_bf16(w)


def make_attention(B: int, Hq: int, Hkv: int, D: int, L: int, seed: int = 0):
    """bf16 decode-attention inputs (``attn_decode`` recipe): query
    [B][Hq][D] = Student-t(nu=4) times one LogNormal(0, 0.5) factor per head
    dimension; keys [B][L][Hkv][D] = N(0,1) times one LogNormal(0, 1) factor
    per (KV head, dimension), so a few dimensions carry outliers as cached
    keys do; values [B][L][Hkv][D] = N(0,1).  The paper evaluates head sizes
    128 and 256 with 4, 6 or 8 query heads per KV head and 8K to 500K cached
    tokens (decode-attention evaluation, Fig. 10)."""
    rng, ch = _rng(seed, 11), _rng(seed, 12)
    q = rng.standard_t(4.0, size=(B, Hq, D)).astype(np.float32)
    q *= ch.lognormal(0.0, 0.5, size=D).astype(np.float32)[None, None, :]
    k = rng.standard_normal((B, L, Hkv, D), dtype=np.float32)
    k *= ch.lognormal(0.0, 1.0, size=(Hkv, D)).astype(np.float32)[None, None, :, :]
    v = rng.standard_normal((B, L, Hkv, D), dtype=np.float32)
    return to_bf16(q), to_bf16(k), to_bf16(v)


def random_bf16(shape, seed: int, scale: float = 1.0) -> torch.Tensor:
    """Plain N(0, scale^2) bf16 tensor for edge-case tests."""
    return to_bf16(_rng(seed, 7).standard_normal(shape, dtype=np.float32) * np.float32(scale))
