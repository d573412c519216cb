"""Per-chunk (action) conditioning on the GPU, through the C ABI
(psv_submit_chunk_cond): parity with the oracle, and causality bit for bit.

Reading <18>: a chunk submitted with its own conditioning vector uses
e_s = temb(t_s) + cond_chunk at every step in place of the stream's vector
(AREX article, section 难题; BAAI announcement, section 新一代物理 AI 的基础设施).
Tolerance: rel-L2 <= 3e-2 per chunk's final latent (the end-to-end bound).
"""
import numpy as np
import pytest

import synth
from _harness import rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FLAG_CHUNK_COND = 4


def _vec(cfg, seed):
    return np.random.default_rng(seed).standard_normal(cfg["d"]).astype(np.float32)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_chunk_conditioning_matches_oracle(name):
    cfg = synth.config(name)
    w = synth.make_weights(cfg, 0)
    streams = synth.make_streams(cfg, 2)
    n = 6
    chunk_conds = [{1: _vec(cfg, 11), 3: _vec(cfg, 13)}, {0: _vec(cfg, 20), 4: streams[1].cond}]
    got, _ = run_gpu(cfg, w, streams, n, flags=FLAG_CHUNK_COND, chunk_conds=chunk_conds)
    ref = run_oracle(cfg, w, streams, n, chunk_conds=chunk_conds)
    for i in range(2):
        for c in range(n):
            e = rel_l2(got[i][c], ref[i][c])
            assert e <= 3e-2, (i, c, e)


def test_chunk_conditioning_causal_and_neutral_bitwise():
    """Chunks before the conditioned one are bit-identical to an
    unconditioned run; it and the later ones change; a vector equal to the
    stream's reproduces the unconditioned run bit for bit."""
    cfg = synth.config("tiny")
    w = synth.make_weights(cfg, 0)
    streams = synth.make_streams(cfg, 1)
    n = 6
    base, _ = run_gpu(cfg, w, streams, n, flags=FLAG_CHUNK_COND)
    same, _ = run_gpu(cfg, w, streams, n, flags=FLAG_CHUNK_COND, chunk_conds=[{2: streams[0].cond}])
    moved, _ = run_gpu(cfg, w, streams, n, flags=FLAG_CHUNK_COND, chunk_conds=[{2: _vec(cfg, 5)}])
    for c in range(n):
        assert np.array_equal(base[0][c], same[0][c]), c
    for c in (0, 1):
        assert np.array_equal(base[0][c], moved[0][c]), c
    for c in (2, 3, 4, 5):
        assert np.max(np.abs(base[0][c] - moved[0][c])) > 1e-6, c
