"""Pins of the CPU oracle's block math against things other than itself.

Each test checks one oracle function against an independent fact: scalar
loops on tiny inputs, a closed form, an invariant, or a special case that
reduces to a textbook result.  A dropped term, a swapped split, a wrong sign
or a transposed operand in ``oracle/model.py`` fails at least one of them.
"""
import math

import numpy as np
import pytest

import synth
from oracle import model as M
from oracle.runner import OracleRunner


def _rng(seed=0):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- attention

def _attention_loops(q, k, v, H, dh):
    """Explicit softmax with a materialised score list, pure Python."""
    Tq, L = q.shape[0], k.shape[0]
    out = np.zeros_like(q)
    for h in range(H):
        for i in range(Tq):
            scores = []
            for j in range(L):
                acc = 0.0
                for e in range(dh):
                    acc += q[i, h * dh + e] * k[j, h * dh + e]
                scores.append(acc / math.sqrt(dh))
            m = max(scores)
            w = [math.exp(x - m) for x in scores]
            z = sum(w)
            for e in range(dh):
                out[i, h * dh + e] = sum(w[j] * v[j, h * dh + e] for j in range(L)) / z
    return out


@pytest.mark.parametrize("T,W,H,dh", [(4, 0, 2, 4), (8, 2, 2, 8), (5, 1, 2, 6)])
def test_attention_matches_scalar_loops(T, W, H, dh):
    r = _rng(T * 100 + W)
    d = H * dh
    q = r.standard_normal((T, d))
    k = r.standard_normal(((W + 1) * T, d)) * 2.0
    v = r.standard_normal(((W + 1) * T, d))
    np.testing.assert_allclose(M.attention(q, k, v, H, dh), _attention_loops(q, k, v, H, dh),
                               rtol=0, atol=1e-12)


def test_attention_key_permutation_invariance():
    r = _rng(1)
    q, k, v = r.standard_normal((6, 16)), r.standard_normal((18, 16)), r.standard_normal((18, 16))
    perm = r.permutation(18)
    np.testing.assert_allclose(M.attention(q, k, v, 2, 8), M.attention(q, k[perm], v[perm], 2, 8),
                               rtol=0, atol=1e-13)


def test_attention_special_cases():
    r = _rng(2)
    v = r.standard_normal((7, 8))
    # one key: output is that key's value
    q = r.standard_normal((3, 8))
    k1 = r.standard_normal((1, 8))
    np.testing.assert_allclose(M.attention(q, k1, v[:1], 2, 4), np.repeat(v[:1], 3, 0), atol=1e-15)
    # zero queries: uniform weights, output is the mean value
    out = M.attention(np.zeros((3, 8)), r.standard_normal((7, 8)), v, 2, 4)
    np.testing.assert_allclose(out, np.repeat(v.mean(0, keepdims=True), 3, 0), atol=1e-14)
    # a dominant key wins; the 1/sqrt(dh) scale is applied (exact ratio check)
    k = np.zeros((2, 4))
    k[0, 0] = 1.0
    qq = np.zeros((1, 4))
    qq[0, 0] = 2.0 * math.log(3.0)  # score gap = 2 ln3 / sqrt(4) = ln 3 -> weights 3:1
    vv = np.array([[1.0, 0, 0, 0], [0.0, 1, 0, 0]])
    np.testing.assert_allclose(M.attention(qq, k, vv, 1, 4)[0, :2], [0.75, 0.25], atol=1e-15)


# -------------------------------------------------------------- linear, LN

def test_linear_matches_loops():
    r = _rng(3)
    x, w, b = r.standard_normal((3, 5)), r.standard_normal((4, 5)), r.standard_normal(4)
    ref = np.array([[sum(x[i, k] * w[o, k] for k in range(5)) + b[o] for o in range(4)]
                    for i in range(3)])
    np.testing.assert_allclose(M.linear(x, w, b), ref, atol=1e-14)


def test_layer_norm_moments_and_invariances():
    r = _rng(4)
    h = r.standard_normal((5, 64)) * 3.0 + 7.0
    y = M.layer_norm(h, 1e-6)
    np.testing.assert_allclose(y.mean(1), 0, atol=1e-14)
    var = h.var(1)
    np.testing.assert_allclose(y.var(1), var / (var + 1e-6), rtol=1e-13)
    np.testing.assert_allclose(M.layer_norm(h + 11.0, 1e-6), y, atol=1e-12)
    np.testing.assert_allclose(M.layer_norm(h * 4.0, 1e-6 * 16.0), y, atol=1e-12)
    assert np.all(M.layer_norm(np.full((2, 8), 3.0), 1e-6) == 0)
    # modulation: zero shift/scale is plain LN
    np.testing.assert_array_equal(M.modulate(y, np.zeros(64), np.zeros(64)), y)


# ------------------------------------------------------------------- RoPE

def test_rope_matches_complex_rotation():
    r = _rng(5)
    H, dh, T = 2, 8, 5
    x = r.standard_normal((T, H * dh))
    pos = np.arange(100, 100 + T)
    out = M.rope(x, pos, H, dh, 1e4)
    for h in range(H):
        z = x[:, h * dh:(h + 1) * dh:2] + 1j * x[:, h * dh + 1:(h + 1) * dh:2]
        freq = np.array([1e4 ** (-(2 * j) / dh) for j in range(dh // 2)])
        zr = z * np.exp(1j * pos[:, None] * freq[None, :])
        np.testing.assert_allclose(out[:, h * dh:(h + 1) * dh:2], zr.real, atol=1e-12)
        np.testing.assert_allclose(out[:, h * dh + 1:(h + 1) * dh:2], zr.imag, atol=1e-12)


def test_rope_norm_and_relative_position():
    r = _rng(6)
    H, dh = 2, 16
    q, k = r.standard_normal((1, H * dh)), r.standard_normal((1, H * dh))
    rq = M.rope(q, np.array([37]), H, dh, 1e4)
    np.testing.assert_allclose(np.linalg.norm(rq), np.linalg.norm(q), rtol=1e-14)
    def score(pq, pk):
        return float((M.rope(q, np.array([pq]), H, dh, 1e4) @ M.rope(k, np.array([pk]), H, dh, 1e4).T)[0, 0])
    base = score(1560 * 7 + 3, 1560 * 5 + 9)
    shifted = score(1560 * 3 + 3, 1560 * 1 + 9)
    assert abs(base - shifted) < 1e-11
    np.testing.assert_array_equal(M.rope(q, np.array([0]), H, dh, 1e4), q)


# ------------------------------------------------ embedding, GELU, SiLU

def test_timestep_embedding_values():
    e0 = M.timestep_embedding(0.0, 256)
    np.testing.assert_array_equal(e0[:128], 1.0)
    np.testing.assert_array_equal(e0[128:], 0.0)
    t = 0.75
    e = M.timestep_embedding(t, 256)
    assert e[0] == math.cos(t) and e[128] == math.sin(t)
    f_last = 1e4 ** (-127 / 128)
    assert abs(e[127] - math.cos(t * f_last)) < 1e-15
    assert abs(e[255] - math.sin(t * f_last)) < 1e-15


def test_gelu_and_silu():
    x = np.linspace(-6, 6, 241)
    g = M.gelu_tanh(x)
    erf_gelu = np.array([0.5 * a * (1 + math.erf(a / math.sqrt(2))) for a in x])
    assert np.max(np.abs(g - erf_gelu)) < 1e-3
    np.testing.assert_allclose(g - M.gelu_tanh(-x), x, atol=1e-14)
    assert M.gelu_tanh(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(M.silu(x), x / (1 + np.exp(-x)), atol=0)
    np.testing.assert_allclose(M.silu(np.array([0.0, 30.0])), [0.0, 30.0], atol=1e-11)


# ------------------------------------------------------------ block wiring

def _tiny_cfg(**kw):
    return synth.config("tiny", **kw)


def _zero_like_weights(cfg):
    w = synth.make_weights(cfg, seed=0)
    for bw in w["blocks"]:
        for k in bw:
            bw[k] = np.zeros_like(bw[k], dtype=np.float64)
    w["global"] = {k: v.astype(np.float64) for k, v in w["global"].items()}
    return w


def test_zero_gates_make_block_identity():
    cfg = _tiny_cfg()
    w = synth.make_weights(cfg, seed=0)
    bw = {k: v.astype(np.float64) for k, v in w["blocks"][0].items()}
    r = _rng(7)
    h = r.standard_normal((cfg["T"], cfg["d"]))
    mod = r.standard_normal(6 * cfg["d"])
    d = cfg["d"]
    mod[2 * d:3 * d] = 0.0  # gate1
    mod[5 * d:6 * d] = 0.0  # gate2
    h_out, _, _ = M.block_forward(cfg, bw, mod, h, M.positions(cfg, 3), [])
    np.testing.assert_array_equal(h_out, h)


def test_block_closed_form_with_constant_values():
    """qkv_w = 0 and a constant v-bias u: attention returns u for every query,
    the MLP with zero up weights returns b_down, so
    h_out = h + gate1 (W_o u + b_o) + gate2 b_down  (checks the gate slots,
    the v slice, the W_o orientation and both residual adds)."""
    cfg = _tiny_cfg()
    d, F = cfg["d"], cfg["F"]
    r = _rng(8)
    bw = {"qkv_w": np.zeros((3 * d, d)), "qkv_b": np.zeros(3 * d),
          "o_w": r.standard_normal((d, d)), "o_b": r.standard_normal(d),
          "up_w": np.zeros((F, d)), "up_b": np.zeros(F),
          "down_w": r.standard_normal((d, F)), "down_b": r.standard_normal(d)}
    u = r.standard_normal(d)
    bw["qkv_b"][:d] = r.standard_normal(d)          # q bias: irrelevant
    bw["qkv_b"][2 * d:] = u
    mod = r.standard_normal(6 * d)
    h = r.standard_normal((cfg["T"], cfg["d"]))
    win = [(r.standard_normal((cfg["T"], d)), np.tile(u, (cfg["T"], 1)))]
    h_out, k, v = M.block_forward(cfg, bw, mod, h, M.positions(cfg, 1), win)
    gate1, gate2 = mod[2 * d:3 * d], mod[5 * d:6 * d]
    expect = h + gate1 * (bw["o_w"] @ u + bw["o_b"]) + gate2 * bw["down_b"]
    np.testing.assert_allclose(h_out, expect, atol=1e-12)
    np.testing.assert_allclose(v, np.tile(u, (cfg["T"], 1)), atol=0)
    np.testing.assert_array_equal(k, 0.0)


def test_block_closed_form_mean_of_modulated_ln():
    """q = k = 0 and v = y (identity v weights): every query averages the
    window's values, so with an empty window o = shift1 + (1+scale1) *
    mean_i LN(h_i); o_w = I then exposes o through gate1."""
    cfg = _tiny_cfg()
    d, F = cfg["d"], cfg["F"]
    r = _rng(9)
    bw = {"qkv_w": np.zeros((3 * d, d)), "qkv_b": np.zeros(3 * d),
          "o_w": np.eye(d), "o_b": np.zeros(d),
          "up_w": np.zeros((F, d)), "up_b": np.zeros(F),
          "down_w": np.zeros((d, F)), "down_b": np.zeros(d)}
    bw["qkv_w"][2 * d:] = np.eye(d)
    mod = r.standard_normal(6 * d)
    h = r.standard_normal((cfg["T"], d)) * 2 + 1
    h_out, _, _ = M.block_forward(cfg, bw, mod, h, M.positions(cfg, 0), [])
    ln = M.layer_norm(h, 1e-6)
    o = mod[:d] + (1 + mod[d:2 * d]) * ln.mean(0)
    np.testing.assert_allclose(h_out, h + mod[2 * d:3 * d] * o, atol=1e-12)


def test_block_mlp_branch_special_case():
    """o_w = 0 removes the attention branch; up = I, down = I (F = d) reduce
    the MLP branch to gate2 * GELU(LN(h)(1+scale2) + shift2)."""
    cfg = _tiny_cfg(F=128)
    d = cfg["d"]
    r = _rng(10)
    bw = {"qkv_w": r.standard_normal((3 * d, d)) * 0.1, "qkv_b": np.zeros(3 * d),
          "o_w": np.zeros((d, d)), "o_b": np.zeros(d),
          "up_w": np.eye(d), "up_b": np.zeros(d), "down_w": np.eye(d), "down_b": np.zeros(d)}
    mod = r.standard_normal(6 * d)
    h = r.standard_normal((cfg["T"], d))
    h_out, _, _ = M.block_forward(cfg, bw, mod, h, M.positions(cfg, 0), [])
    y2 = M.layer_norm(h, 1e-6) * (1 + mod[4 * d:5 * d]) + mod[3 * d:4 * d]
    expect = h + mod[5 * d:6 * d] * np.array([[0.5 * a * (1 + math.tanh(math.sqrt(2 / math.pi) * (a + 0.044715 * a ** 3)))
                                               for a in row] for row in y2])
    np.testing.assert_allclose(h_out, expect, atol=1e-12)


def test_conditioning_closed_form():
    """With W_mod = 0 the table is its bias; fmod likewise; and the time MLP
    reduces to explicit scalar SiLU loops on a single element."""
    cfg = _tiny_cfg()
    w = _zero_like_weights(cfg)
    r = _rng(11)
    for bw in w["blocks"]:
        bw["mod_b"] = r.standard_normal(6 * cfg["d"])
    w["global"]["fmod_w"][:] = 0
    w["global"]["fmod_b"] = r.standard_normal(2 * cfg["d"])
    cond = r.standard_normal(cfg["d"])
    mod, fmod = M.conditioning(cfg, w["global"], w["blocks"], cond)
    for s in range(cfg["S"]):
        for b in range(cfg["B"]):
            np.testing.assert_array_equal(mod[s, b], w["blocks"][b]["mod_b"])
        np.testing.assert_array_equal(fmod[s], w["global"]["fmod_b"])
    # element check of the whole chain for one output component
    g = {k: v for k, v in synth.make_weights(cfg, 1)["global"].items()}
    g = {k: v.astype(np.float64) for k, v in g.items()}
    blocks = [{k: v.astype(np.float64) for k, v in bw.items()} for bw in synth.make_weights(cfg, 1)["blocks"]]
    mod, fmod = M.conditioning(cfg, g, blocks, cond)
    s, b, o = 1, 1, 5
    t = 1 - s / cfg["S"]
    emb = [math.cos(t * math.exp(-math.log(1e4) * j / 128)) for j in range(128)] + \
          [math.sin(t * math.exp(-math.log(1e4) * j / 128)) for j in range(128)]
    sl = lambda a: a / (1 + math.exp(-a))
    a1 = [sl(sum(g["t1_w"][i, j] * emb[j] for j in range(256)) + g["t1_b"][i]) for i in range(cfg["d"])]
    temb = [sum(g["t2_w"][i, j] * a1[j] for j in range(cfg["d"])) + g["t2_b"][i] for i in range(cfg["d"])]
    se = [sl(temb[i] + cond[i]) for i in range(cfg["d"])]
    want = sum(blocks[b]["mod_w"][o, j] * se[j] for j in range(cfg["d"])) + blocks[b]["mod_b"][o]
    assert abs(mod[s, b, o] - want) < 1e-12


# ------------------------------------------------ stream-level invariants

def _runner(cfg, weights, n_streams=1, dtype=np.float64, conds=None):
    r = OracleRunner(cfg, weights, dtype)
    streams = synth.make_streams(cfg, n_streams)
    for i, st in enumerate(streams):
        r.open_stream(st.cond if conds is None else conds[i])
    return r, streams


def test_euler_constant_velocity_closed_form():
    for S in (2, 4):
        cfg = _tiny_cfg(S=S, B=1)
        w = synth.make_weights(cfg, 0)
        beta = np.random.default_rng(12).standard_normal(cfg["C"]).astype(np.float32)
        w["global"]["out_w"] = np.zeros_like(w["global"]["out_w"])
        w["global"]["out_b"] = beta
        r, st = _runner(cfg, w)
        x0 = st[0].noise(0).astype(np.float64)
        r.submit(0, st[0].noise(0))
        r.run_until_idle()
        xs = r.streams[0].outputs[0]
        err = np.abs(xs - (x0 - beta))
        bound = 4 * S * np.finfo(np.float64).eps * (np.abs(x0) + np.abs(beta))
        assert np.all(err <= bound)


def test_window_zero_gives_independent_chunks():
    """W = 0: a chunk sees only itself, and RoPE scores depend on position
    differences only, so chunk 2 of one stream equals chunk 0 of another
    stream given the same noise and conditioning."""
    cfg = _tiny_cfg(W=0)
    w = synth.make_weights(cfg, 0)
    st = synth.make_streams(cfg, 1)[0]
    r = OracleRunner(cfg, w)
    r.open_stream(st.cond)
    r.open_stream(st.cond)
    for c in range(3):
        r.submit(0, st.noise(c))
    r.submit(1, st.noise(2))
    r.run_until_idle()
    a, b = r.streams[0].outputs[2], r.streams[1].outputs[0]
    assert np.max(np.abs(a - b)) < 1e-9
    # and with W > 0 the predecessors do matter
    cfg3 = _tiny_cfg()
    r3 = OracleRunner(cfg3, w)
    r3.open_stream(st.cond)
    r3.open_stream(st.cond)
    for c in range(3):
        r3.submit(0, st.noise(c))
    r3.submit(1, st.noise(2))
    r3.run_until_idle()
    assert np.max(np.abs(r3.streams[0].outputs[2] - r3.streams[1].outputs[0])) > 1e-4


def test_window_history_enters_through_kv():
    """With W = 1 a perturbation of chunk 0 changes chunk 0's output and
    reaches chunk 1 through chunk 0's stored KV."""
    cfg = _tiny_cfg(W=1, B=1)
    w = synth.make_weights(cfg, 0)
    st = synth.make_streams(cfg, 1)[0]
    outs = []
    for perturb in (0.0, 1.0):
        r = OracleRunner(cfg, w)
        r.open_stream(st.cond)
        r.submit(0, st.noise(0) + perturb)
        r.submit(0, st.noise(1))
        r.run_until_idle()
        outs.append([r.streams[0].outputs[c] for c in range(2)])
    assert np.max(np.abs(outs[0][0] - outs[1][0])) > 1e-3
    assert np.max(np.abs(outs[0][1] - outs[1][1])) > 1e-6


def test_wave_order_equals_sequential_order_bitwise():
    cfg = _tiny_cfg()
    w = synth.make_weights(cfg, 0)
    ra, st = _runner(cfg, w)
    rb, _ = _runner(cfg, w)
    for c in range(cfg["n_chunks"]):
        ra.submit(0, st[0].noise(c))
        rb.submit(0, st[0].noise(c))
    ra.run_until_idle()
    rb.run_sequential(0)
    for c in range(cfg["n_chunks"]):
        np.testing.assert_array_equal(ra.streams[0].outputs[c], rb.streams[0].outputs[c])
    # the wave run really was batched: waves held several tasks
    assert ra.task_log != rb.task_log


def test_fp32_oracle_close_to_fp64():
    cfg = _tiny_cfg()
    w = synth.make_weights(cfg, 0)
    outs = {}
    for dt in (np.float64, np.float32):
        r, st = _runner(cfg, w, dtype=dt)
        for c in range(cfg["n_chunks"]):
            r.submit(0, st[0].noise(c))
        r.run_until_idle()
        outs[dt] = np.stack([r.streams[0].outputs[c] for c in range(cfg["n_chunks"])])
    x64, x32 = outs[np.float64], outs[np.float32].astype(np.float64)
    assert np.linalg.norm(x32 - x64) / np.linalg.norm(x64) < 1e-5


def test_chunk_conditioning_matches_stream_conditioning():
    """Per-chunk conditioning (reading <18>) with W = 0: chunk 2 of a stream,
    submitted with its own vector a, equals chunk 0 of a stream opened with a
    (same noise; RoPE scores depend on position differences only), while the
    neighbouring chunks keep the stream's vector."""
    cfg = _tiny_cfg(W=0)
    w = synth.make_weights(cfg, 0)
    st = synth.make_streams(cfg, 1)[0]
    a = np.random.default_rng(7).standard_normal(cfg["d"]).astype(np.float32)
    r = OracleRunner(cfg, w)
    r.open_stream(st.cond)
    r.open_stream(a)
    r.open_stream(st.cond)
    r.submit(0, st.noise(0))
    r.submit(0, st.noise(1))
    r.submit(0, st.noise(2), cond=a)
    r.submit(0, st.noise(3))
    r.submit(1, st.noise(2))
    r.submit(2, st.noise(3))
    r.run_until_idle()
    assert np.max(np.abs(r.streams[0].outputs[2] - r.streams[1].outputs[0])) < 1e-9
    # chunk 3 went back to the stream's vector
    assert np.max(np.abs(r.streams[0].outputs[3] - r.streams[2].outputs[0])) < 1e-9


def test_chunk_conditioning_is_causal():
    """With W > 0 a chunk's vector reaches later chunks only through its
    stored KV: chunks before it are bit-identical, it and later ones change;
    a vector equal to the stream's gives the unconditioned run bit for bit."""
    cfg = _tiny_cfg()
    w = synth.make_weights(cfg, 0)
    st = synth.make_streams(cfg, 1)[0]
    a = np.random.default_rng(8).standard_normal(cfg["d"]).astype(np.float32)

    def run(conds):
        r = OracleRunner(cfg, w)
        r.open_stream(st.cond)
        for c in range(5):
            r.submit(0, st.noise(c), cond=conds.get(c))
        r.run_until_idle()
        return r.streams[0].outputs

    base = run({})
    same = run({2: st.cond})
    moved = run({2: a})
    for c in range(5):
        assert np.array_equal(base[c], same[c])
    for c in (0, 1):
        assert np.array_equal(base[c], moved[c])
    for c in (2, 3, 4):
        assert np.max(np.abs(base[c] - moved[c])) > 1e-6


# ------------------------------------------------------------ final head, positions

def test_final_velocity_closed_form():
    """Final adaLN + head (reading <5>) on rows whose LayerNorm is known
    exactly: row r = mu_r + sigma_r * z with z = (+1, -1, +1, ...), so the
    row has mean mu_r, biased variance sigma_r^2 and LN(row) = z * sigma_r /
    sqrt(sigma_r^2 + eps).  The head reads column 2j+1 into output j
    (W_out[j, 2j+1] = 1), shift_f and scale_f are different constants and
    b_out is a ramp, so a swapped [shift_f, scale_f] split, a missing LN, an
    LN without the eps, a transposed or shifted head or a dropped bias gives
    another value."""
    d, C, eps = 16, 5, 1e-6
    cfg = {"d": d, "ln_eps": eps}
    z = np.array([1.0 if e % 2 == 0 else -1.0 for e in range(d)])
    mus, sigmas = [3.0, -0.5, 0.0], [2.0, 0.25, 1e-3]
    h = np.stack([m + s * z for m, s in zip(mus, sigmas)])
    shift_c, scale_c = 0.75, -0.4
    fmod = np.concatenate([np.full(d, shift_c), np.full(d, scale_c)])
    out_w = np.zeros((C, d))
    for j in range(C):
        out_w[j, 2 * j + 1] = 1.0
    out_b = np.arange(C) * 0.1
    g = {"out_w": out_w, "out_b": out_b}
    v = M.final_velocity(cfg, g, fmod, h)
    for r, s in enumerate(sigmas):
        ln_odd = -s / math.sqrt(s * s + eps)  # z = -1 on every odd column
        expect = [ln_odd * (1.0 + scale_c) + shift_c + out_b[j] for j in range(C)]
        np.testing.assert_allclose(v[r], expect, rtol=0, atol=1e-12)


def test_final_velocity_uses_its_step_fmod_in_the_runner():
    """Inside a run the head uses the fmod row of the task's own step: with
    identity blocks (zero adaLN weights, so zero gates) and a head that reads
    the modulated LN of h, only shift_f enters through b_fmod, which makes the
    velocity of every step the same constant and x_S = x_0 - (shift_f . head
    + b_out) in closed form, step by step."""
    cfg = _tiny_cfg(S=4, B=1)
    w = synth.make_weights(cfg, 0)
    d, C = cfg["d"], cfg["C"]
    for bw in w["blocks"]:
        bw["mod_w"] = np.zeros_like(bw["mod_w"])
        bw["mod_b"] = np.zeros_like(bw["mod_b"])
    # fmod = b_fmod whatever the step: shift_f = 0.5, scale_f = -1 (zeroes the LN term)
    w["global"]["fmod_w"] = np.zeros_like(w["global"]["fmod_w"])
    w["global"]["fmod_b"] = np.concatenate([np.full(d, 0.5), np.full(d, -1.0)]).astype(np.float32)
    head = np.random.default_rng(21).standard_normal((C, d)).astype(np.float32)
    w["global"]["out_w"] = head
    w["global"]["out_b"] = np.zeros(C, np.float32)
    r, st = _runner(cfg, w)
    x0 = st[0].noise(0).astype(np.float64)
    r.submit(0, st[0].noise(0))
    r.run_until_idle()
    vel = np.array([0.5 * head[j].astype(np.float64).sum() for j in range(C)])
    np.testing.assert_allclose(r.streams[0].outputs[0], x0 - vel[None, :], rtol=0, atol=1e-12)


def test_positions_offset_each_chunk_by_T():
    """RoPE positions are global, c*T + i (the configurations' definition).
    Three chunks with the same noise give the same pre-RoPE keys at block 0,
    step 0 (their block input depends only on their own x_0), so the stored
    keys of chunk c must equal chunk 0's keys with pair j of every head turned
    by the extra angle c*T*theta^(-2j/dh), checked as a complex product, and
    chunk 0's keys must be its un-rotated keys turned by i*theta^(-2j/dh).
    An offset of c*(T-1), (c+1)*T or none fails it."""
    cfg = _tiny_cfg(W=2, B=1, S=1)
    w = synth.make_weights(cfg, 0)
    T, H, dh, theta = cfg["T"], cfg["H"], cfg["dh"], cfg["rope_theta"]
    st = synth.make_streams(cfg, 1)[0]
    r = OracleRunner(cfg, w)
    r.open_stream(st.cond)
    for _ in range(3):
        r.submit(0, st.noise(0))
    r.run_until_idle()
    k0 = r.streams[0].kv[(0, 0, 0)][0]

    def as_complex(k):
        kr = k.reshape(T, H, dh // 2, 2)
        return kr[..., 0] + 1j * kr[..., 1]

    freqs = np.array([theta ** (-2.0 * j / dh) for j in range(dh // 2)])
    # chunk 0 sits at positions 0..T-1: its stored keys are the un-rotated
    # keys (RoPE at position 0 is the identity) turned by i * freq
    g = {k: v.astype(np.float64) for k, v in w["global"].items()}
    bw = {k: v.astype(np.float64) for k, v in w["blocks"][0].items()}
    h0 = M.in_proj(g, st.noise(0).astype(np.float64))
    _, k_plain, _ = M.block_qkv(cfg, bw, r.streams[0].mod[0, 0], h0, np.zeros(T, dtype=np.int64))
    turn0 = np.exp(1j * np.arange(T)[:, None, None] * freqs[None, None, :])
    np.testing.assert_allclose(as_complex(k0), as_complex(k_plain) * turn0, rtol=0, atol=1e-12)
    for c in (1, 2):
        kc = r.streams[0].kv[(0, 0, c)][0]
        turn = np.exp(1j * c * T * freqs)[None, None, :]
        np.testing.assert_allclose(as_complex(kc), as_complex(k0) * turn, rtol=0, atol=1e-12)
