"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module holds shapes and random draws only: no step of the denoising
method is computed here.  Both sides receive identical numbers from it and
nothing else.

Shapes follow the five model configurations this library is measured on
(a tiny DiT plus Wan2.1-1.3B / Wan2.2-TI2V-5B / Wan2.1-14B shaped models),
plus a "mid" configuration used only by parity tests: full head width
(dh = 128), a ragged chunk length (T = 200 is not a multiple of 128) and two
streams, small enough for the fp64 oracle to finish in seconds.

Draw order (fixed, documented so any consumer can regenerate a tensor):
  * model weights from ``numpy.random.default_rng(weight_seed)`` (PCG64):
    global tensors first, then block 0..B-1, each in ``tensor_specs`` order;
    every weight matrix is N(0, 0.02) drawn in float32 and rounded to the
    nearest bfloat16 (ties to even), because the served model is a bf16
    model; every bias is exactly zero and consumes no draws;
  * stream i uses ``default_rng(1000 + i)``: first its conditioning vector
    cond ~ N(0, 1)[d] (float32), then one noise chunk N(0, 1)[T*C] (float32)
    per chunk, in chunk order.
"""
from __future__ import annotations

import numpy as np

# Fixed hyper-parameters of every configuration (timestep-embedding width,
# LayerNorm epsilon, RoPE base).
T_EMBED = 256
LN_EPS = 1e-6
ROPE_THETA = 1e4

CONFIGS = {
    # Tiny DiT: the configuration the oracle runs end to end in full.
    "tiny": dict(B=2, S=2, d=128, H=4, dh=32, F=512, C=16, T=64, W=3,
                 n_streams=1, n_chunks=6),
    # Parity-only: dh = 128 like the large models, T ragged against 128-row
    # tiles, two streams batched into one wave.
    "mid": dict(B=2, S=4, d=256, H=2, dh=128, F=768, C=32, T=200, W=2,
                n_streams=2, n_chunks=7),
    "wan21_1p3b": dict(B=30, S=4, d=1536, H=12, dh=128, F=8960, C=64, T=1560,
                       W=4, n_streams=1, n_chunks=64),
    "wan22_5b": dict(B=30, S=4, d=3072, H=24, dh=128, F=14336, C=192, T=880,
                     W=4, n_streams=1, n_chunks=64),
    "wan21_1p3b_x8": dict(B=30, S=4, d=1536, H=12, dh=128, F=8960, C=64,
                          T=1560, W=4, n_streams=8, n_chunks=32),
    "wan21_14b": dict(B=40, S=4, d=5120, H=40, dh=128, F=13824, C=64, T=1560,
                      W=4, n_streams=2, n_chunks=32),
}

WEIGHT_STD = 0.02


def config(name: str, **overrides) -> dict:
    """Return a copy of a named configuration with optional overrides."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    cfg.setdefault("t_embed", T_EMBED)
    cfg.setdefault("ln_eps", LN_EPS)
    cfg.setdefault("rope_theta", ROPE_THETA)
    assert cfg["H"] * cfg["dh"] == cfg["d"]
    return cfg


def global_specs(cfg: dict):
    """(name, shape) of the model-level tensors, in draw order.

    Linear weights are [out, in] row-major; every ``*_w`` has a ``*_b``.
    """
    d, C, E = cfg["d"], cfg["C"], cfg["t_embed"]
    return [
        ("in_w", (d, C)), ("in_b", (d,)),
        ("t1_w", (d, E)), ("t1_b", (d,)),
        ("t2_w", (d, d)), ("t2_b", (d,)),
        ("fmod_w", (2 * d, d)), ("fmod_b", (2 * d,)),
        ("out_w", (C, d)), ("out_b", (C,)),
    ]


def block_specs(cfg: dict):
    """(name, shape) of one transformer block's tensors, in draw order."""
    d, F = cfg["d"], cfg["F"]
    return [
        ("qkv_w", (3 * d, d)), ("qkv_b", (3 * d,)),
        ("o_w", (d, d)), ("o_b", (d,)),
        ("up_w", (F, d)), ("up_b", (F,)),
        ("down_w", (d, F)), ("down_b", (d,)),
        ("mod_w", (6 * d, d)), ("mod_b", (6 * d,)),
    ]


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array -> float32 array holding the nearest bfloat16 values.

    Round-to-nearest-even on the bit pattern; used only to make the synthetic
    weights exactly representable in bf16.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _draw(rng: np.random.Generator, name: str, shape) -> np.ndarray:
    if name.endswith("_b"):
        return np.zeros(shape, dtype=np.float32)
    w = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(WEIGHT_STD)
    return round_to_bf16(w)


def iter_weights(cfg: dict, seed: int = 0):
    """Yield (block, name, float32 array) in draw order; block = -1 for globals.

    Streaming keeps host memory at one tensor for the large configurations.
    """
    rng = np.random.default_rng(seed)
    for name, shape in global_specs(cfg):
        yield -1, name, _draw(rng, name, shape)
    for b in range(cfg["B"]):
        for name, shape in block_specs(cfg):
            yield b, name, _draw(rng, name, shape)


def make_weights(cfg: dict, seed: int = 0) -> dict:
    """All weights as {"global": {name: arr}, "blocks": [{name: arr}, ...]}."""
    out = {"global": {}, "blocks": [dict() for _ in range(cfg["B"])]}
    for b, name, arr in iter_weights(cfg, seed):
        if b < 0:
            out["global"][name] = arr
        else:
            out["blocks"][b][name] = arr
    return out


class StreamInputs:
    """Conditioning vector and per-chunk noise of one stream (seed 1000 + i)."""

    def __init__(self, cfg: dict, index: int):
        self.cfg = cfg
        self._rng = np.random.default_rng(1000 + index)
        self.cond = self._rng.standard_normal(size=cfg["d"], dtype=np.float32)
        self._noise = []

    def noise(self, c: int) -> np.ndarray:
        """Noise of chunk c, float32 [T, C]; chunks are drawn in order."""
        T, C = self.cfg["T"], self.cfg["C"]
        while len(self._noise) <= c:
            self._noise.append(
                self._rng.standard_normal(size=T * C, dtype=np.float32).reshape(T, C))
        return self._noise[c]


def make_streams(cfg: dict, n_streams: int | None = None):
    n = cfg["n_streams"] if n_streams is None else n_streams
    return [StreamInputs(cfg, i) for i in range(n)]


def iter_device_weights(cfg: dict, seed: int = 0, device: str = "cuda"):
    """Yield (block, name, torch tensor) drawn on the GPU with torch's seeded
    Philox generator: matrices N(0, 0.02) as bf16, biases zero f32.

    Same shapes, order and distribution as ``iter_weights`` but a different
    generator (the values differ); used where only the timing matters, to
    avoid drawing billions of numbers on the host.
    """
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    specs = [(-1, n, s) for n, s in global_specs(cfg)]
    for b in range(cfg["B"]):
        specs += [(b, n, s) for n, s in block_specs(cfg)]
    for b, name, shape in specs:
        if name.endswith("_b"):
            yield b, name, torch.zeros(shape, dtype=torch.float32, device=device)
        else:
            w = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
            yield b, name, (w * WEIGHT_STD).to(torch.bfloat16)
