"""Seeded synthetic inputs shaped like the pages' BitNet embedding models.

This module holds shapes and random draws only -- none of the projection's
arithmetic -- so that the CUDA path and the CPU oracle can be fed identical
inputs.  Shapes follow the model table of "BitNet Embeddings GGUF Conversion
Implementation", section 1 ("Background"): the Qwen3-shaped 0.6B model
(hidden 1024, attention width 16 x 128 = 2048, FFN 3072, 28 layers) and the
Gemma3-shaped 270M model (hidden 640, attention width 4 x 256 = 1024, FFN 2048,
18 layers), with the per-projection norm widths of its per-layer tensor table.

Distributions (no trained weights exist here):
  x        ~ N(0, 1), optionally with 1% of the feature columns scaled x20;
  norm_w   = 1 + 0.1 * N(0, 1);
  latent W ~ 0.02 * N(0, 1), quantised by each side (library or oracle) itself.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

EPS = 1e-6  # rms_norm_eps of both models (model table, section 1)


@dataclass(frozen=True)
class Projection:
    name: str
    K: int  # input features (the norm weight's length)
    N: int  # output features


# (name, K, N): q/k/v/gate/up read the hidden state, o the attention output,
# down the FFN activation (per-layer tensor table, section 1, and the
# load_tensors shapes of section 4.5).
QWEN3_0P6B_LAYER = (
    Projection("q", 1024, 2048),
    Projection("k", 1024, 1024),
    Projection("v", 1024, 1024),
    Projection("o", 2048, 1024),
    Projection("gate", 1024, 3072),
    Projection("up", 1024, 3072),
    Projection("down", 3072, 1024),
)
QWEN3_0P6B_LAYERS = 28

GEMMA3_270M_LAYER = (
    Projection("q", 640, 1024),
    Projection("k", 640, 256),
    Projection("v", 640, 256),
    Projection("o", 1024, 640),
    Projection("gate", 640, 2048),
    Projection("up", 640, 2048),
    Projection("down", 2048, 640),
)
GEMMA3_270M_LAYERS = 18

SWEEP_KN = (1024, 4096, 8192, 16384)
SWEEP_M = (1, 16, 128, 2048, 16384)

# tensor ids inside one projection's seed
T_X, T_G, T_W, T_OUTLIER = 0, 1, 2, 3


def seed_for(config: int, layer: int, proj: int, tensor: int) -> int:
    """One 32-bit seed per (workload, layer, projection, tensor)."""
    return int(np.random.SeedSequence([config, layer, proj, tensor]).generate_state(1)[0])


def gen_x(M: int, K: int, seed: int, outlier_frac: float = 0.0, outlier_gain: float = 20.0,
          outlier_seed: int | None = None) -> np.ndarray:
    """Activations x[M, K] ~ N(0, 1) in fp32; with outlier_frac > 0, that fraction
    of feature columns (at least one, chosen without replacement) is scaled by
    outlier_gain for every token."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outlier_frac > 0.0:
        n_out = max(1, int(round(outlier_frac * K)))
        orng = np.random.default_rng(seed if outlier_seed is None else outlier_seed)
        cols = orng.choice(K, size=n_out, replace=False)
        x[:, cols] *= np.float32(outlier_gain)
    return x


def gen_norm_w(K: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)


def gen_latent_w(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (std * rng.standard_normal((N, K), dtype=np.float32)).astype(np.float32)


def gen_projection(config: int, layer: int, proj: int, M: int, K: int, N: int,
                   outlier_frac: float = 0.0):
    """(x[M,K], norm_w[K], latent W[N,K]) for one projection, all fp32 numpy."""
    x = gen_x(M, K, seed_for(config, layer, proj, T_X), outlier_frac,
              outlier_seed=seed_for(config, layer, proj, T_OUTLIER))
    g = gen_norm_w(K, seed_for(config, layer, proj, T_G))
    w = gen_latent_w(N, K, seed_for(config, layer, proj, T_W))
    return x, g, w


def gen_device(shape, seed: int, device, kind: str = "normal", std: float = 1.0, mean: float = 0.0):
    """Large draws made directly on a CUDA device with torch's Philox generator
    (used where a numpy draw on the host would dominate set-up time); the oracle
    receives copies of the same tensors."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    if kind != "normal":
        raise ValueError(kind)
    t.normal_(mean=mean, std=std, generator=gen)
    return t


def gen_device_outlier_cols(K: int, seed: int, frac: float = 0.01) -> np.ndarray:
    n_out = max(1, int(round(frac * K)))
    return np.random.default_rng(seed).choice(K, size=n_out, replace=False)
