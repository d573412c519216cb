"""CPU oracle of the autoregressive-denoising DiT block math (numpy).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
baseline of the benchmark may import this package.  It shares no code with
the CUDA library and never calls it.

Every function is the plain definition, written in the order the method
states it, with a library matmul as the only building block.  It runs in
float64 by default; ``dtype=np.float32`` gives the (slower to converge, faster
to run) fp32 variant used for the CPU timing baseline.  RoPE angles are
always formed in float64.

Sources.  The pages (the PhysisServe announcements) fix the *serving*
semantics: a chunk starts from pure noise and is denoised over S steps; at
every step and every transformer block it reads the still-noisy KV that the
preceding chunk left at that same step and block (AREX article
"vLLM 与 Physis-AI 联合介绍 PhysisServe 推理系统", §难题; BAAI announcement
"智源悟界·PhysisServe", §新一代物理 AI 的基础设施, Fig. 1).  The pages give no
block internals.  The block is the tiny-DiT definition this library serves:
adaLN-modulated LayerNorm without affine (eps 1e-6), QKV with 1-D RoPE
(theta 1e4, global position c*T+i), attention over own + W previous chunks'
same-(block, step) KV, gated residuals, GELU MLP, a final adaLN + linear
head and an Euler update x += (t_{s+1} - t_s) v with t_s = 1 - s/S.
Readings where the definition is open are marked ``reading <n>``:
  <1> the sinusoid argument is t_s itself (no x1000 scale);
  <2> sinusoid = [cos(t f_j), sin(t f_j)], f_j = exp(-ln(1e4) j / (E/2));
  <3> stream conditioning enters by addition: e_s = temb(t_s) + cond;
  <4> mod[s][b] = W_mod,b SiLU(e_s) + b_mod,b split as
      [shift1, scale1, gate1, shift2, scale2, gate2];
  <5> the final head is adaLN (fmod = W_fmod SiLU(e_s) + b, split
      [shift_f, scale_f]) followed by a linear layer;
  <6> x_0 is the submitted noise, already patchified [T, C];
  <7> head h uses columns [h*dh, (h+1)*dh) of q, k and v;
  <8> RoPE rotates interleaved pairs (2j, 2j+1) by pos * theta^(-2j/dh);
  <9> no mask: a chunk is bidirectional and its whole window is visible;
  <10> softmax scale 1/sqrt(dh);
  <11> GELU is the tanh approximation;
  <18> a chunk submitted with its own conditioning vector (an action /
       observation embedding) uses it in place of the stream's at every
       step of that chunk: e_s = temb(t_s) + cond_chunk (``runner.submit``).
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Elementary pieces
# ---------------------------------------------------------------------------

def timestep_embedding(t: float, dim: int, theta: float = 1e4) -> np.ndarray:
    """Sinusoidal embedding of a scalar time, readings <1>, <2> (float64)."""
    half = dim // 2
    freqs = np.exp(-math.log(theta) * np.arange(half, dtype=np.float64) / half)
    arg = float(t) * freqs
    return np.concatenate([np.cos(arg), np.sin(arg)])


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh form, reading <11>."""
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x * x * x)))


def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """nn.Linear convention: w is [out, in]."""
    return x @ w.T + b


def layer_norm(h: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis, biased variance, no affine."""
    mu = h.mean(axis=-1, keepdims=True)
    var = ((h - mu) ** 2).mean(axis=-1, keepdims=True)
    return (h - mu) / np.sqrt(var + eps)


def modulate(x: np.ndarray, shift: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """adaLN modulation x * (1 + scale) + shift."""
    return x * (1.0 + scale) + shift


def rope(x: np.ndarray, pos: np.ndarray, n_heads: int, dh: int, theta: float) -> np.ndarray:
    """1-D rotary embedding of every head of x [T, n_heads*dh], reading <8>.

    Pair (2j, 2j+1) of each head is rotated by pos * theta^(-2j/dh); the
    angle is formed in float64 whatever the dtype of x.
    """
    T = x.shape[0]
    j = np.arange(dh // 2, dtype=np.float64)
    inv = theta ** (-2.0 * j / dh)
    ang = pos.astype(np.float64)[:, None] * inv[None, :]
    cos = np.cos(ang).astype(x.dtype)[:, None, :]
    sin = np.sin(ang).astype(x.dtype)[:, None, :]
    xr = x.reshape(T, n_heads, dh // 2, 2)
    a, b = xr[..., 0], xr[..., 1]
    out = np.stack([a * cos - b * sin, a * sin + b * cos], axis=-1)
    return out.reshape(T, n_heads * dh)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int, dh: int) -> np.ndarray:
    """Multi-head softmax attention without mask, readings <7>, <9>, <10>.

    q [Tq, H*dh], k and v [L, H*dh]; every query sees every key.
    """
    out = np.empty_like(q)
    scale = 1.0 / math.sqrt(dh)
    for h in range(n_heads):
        cols = slice(h * dh, (h + 1) * dh)
        s = (q[:, cols] @ k[:, cols].T) * scale
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, cols] = p @ v[:, cols]
    return out


# ---------------------------------------------------------------------------
# Model pieces
# ---------------------------------------------------------------------------

def step_times(S: int) -> np.ndarray:
    """t_s = 1 - s/S for s = 0..S: pure noise at t = 1, clean at t = 0."""
    return np.array([1.0 - s / S for s in range(S + 1)], dtype=np.float64)


def conditioning(cfg: dict, g: dict, blocks, cond: np.ndarray, dtype=np.float64):
    """Per-stream modulation tables, readings <1>-<5>.

    Returns mod [S, B, 6d] and fmod [S, 2d]: for each step s,
    temb = W_t2 SiLU(W_t1 emb(t_s) + b_t1) + b_t2, e = temb + cond,
    mod[s][b] = W_mod,b SiLU(e) + b_mod,b, fmod[s] = W_fmod SiLU(e) + b_fmod.
    ``blocks`` is a list of all block weight dicts, or a dict {b: weights}
    for a subset (rows of the other blocks are left as NaN).
    """
    S, B, d = cfg["S"], cfg["B"], cfg["d"]
    ts = step_times(S)
    items = blocks.items() if isinstance(blocks, dict) else enumerate(blocks)
    items = list(items)
    mod = np.full((S, B, 6 * d), np.nan, dtype=dtype)
    fmod = np.empty((S, 2 * d), dtype=dtype)
    cond = cond.astype(dtype)
    for s in range(S):
        emb = timestep_embedding(ts[s], cfg["t_embed"]).astype(dtype)
        temb = linear(silu(linear(emb, g["t1_w"], g["t1_b"])), g["t2_w"], g["t2_b"])
        se = silu(temb + cond)
        for b, bw in items:
            mod[s, b] = linear(se, bw["mod_w"], bw["mod_b"])
        fmod[s] = linear(se, g["fmod_w"], g["fmod_b"])
    return mod, fmod


def in_proj(g: dict, x: np.ndarray) -> np.ndarray:
    """Residual stream of a task: h = x W_in^T + b_in, reading <6>."""
    return linear(x, g["in_w"], g["in_b"])


def block_qkv(cfg: dict, bw: dict, mod_sb: np.ndarray, h: np.ndarray, pos: np.ndarray):
    """First half of a block up to the attention inputs.

    Returns (q, k, v) with RoPE applied to q and k at positions ``pos``.
    """
    d, H, dh = cfg["d"], cfg["H"], cfg["dh"]
    shift1, scale1 = mod_sb[0:d], mod_sb[d:2 * d]
    y = modulate(layer_norm(h, cfg["ln_eps"]), shift1, scale1)
    qkv = linear(y, bw["qkv_w"], bw["qkv_b"])
    q, k, v = qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:]
    q = rope(q, pos, H, dh, cfg["rope_theta"])
    k = rope(k, pos, H, dh, cfg["rope_theta"])
    return q, k, v


def block_rest(cfg: dict, bw: dict, mod_sb: np.ndarray, h: np.ndarray,
               q: np.ndarray, keys: np.ndarray, values: np.ndarray) -> np.ndarray:
    """Attention over the window, gated residual, MLP, gated residual."""
    d, H, dh = cfg["d"], cfg["H"], cfg["dh"]
    gate1 = mod_sb[2 * d:3 * d]
    shift2, scale2, gate2 = mod_sb[3 * d:4 * d], mod_sb[4 * d:5 * d], mod_sb[5 * d:6 * d]
    o = attention(q, keys, values, H, dh)
    h = h + gate1 * linear(o, bw["o_w"], bw["o_b"])
    y2 = modulate(layer_norm(h, cfg["ln_eps"]), shift2, scale2)
    u = gelu_tanh(linear(y2, bw["up_w"], bw["up_b"]))
    return h + gate2 * linear(u, bw["down_w"], bw["down_b"])


def block_forward(cfg: dict, bw: dict, mod_sb: np.ndarray, h: np.ndarray, pos: np.ndarray,
                  window: list):
    """One transformer block of one (chunk, step) task.

    ``window`` holds the (k, v) pairs that the W preceding chunks stored at
    this (block, step), oldest first; the task's own (k, v) is appended last.
    Returns (h_out, k, v); (k, v) is what this chunk leaves for its
    successors (post-RoPE, still noisy).
    """
    q, k, v = block_qkv(cfg, bw, mod_sb, h, pos)
    keys = np.concatenate([kv[0] for kv in window] + [k], axis=0)
    values = np.concatenate([kv[1] for kv in window] + [v], axis=0)
    return block_rest(cfg, bw, mod_sb, h, q, keys, values), k, v


def final_velocity(cfg: dict, g: dict, fmod_s: np.ndarray, h: np.ndarray) -> np.ndarray:
    """Final adaLN + linear head, reading <5>: v = (LN(h)(1+scale_f)+shift_f) W_out^T + b_out."""
    d = cfg["d"]
    shift_f, scale_f = fmod_s[0:d], fmod_s[d:2 * d]
    return linear(modulate(layer_norm(h, cfg["ln_eps"]), shift_f, scale_f), g["out_w"], g["out_b"])


def euler(x: np.ndarray, v: np.ndarray, t_s: float, t_next: float) -> np.ndarray:
    """x_{s+1} = x_s + (t_{s+1} - t_s) v."""
    return x + (t_next - t_s) * v


def positions(cfg: dict, c: int) -> np.ndarray:
    """Global token positions c*T + i of chunk c."""
    T = cfg["T"]
    return np.arange(c * T, (c + 1) * T, dtype=np.int64)
