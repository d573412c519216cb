"""Latency-mode schedule on the GPU (PSV_FLAG_LATENCY): every wave runs each
stream's oldest ready chunk only.  Batch invariance makes the outputs equal,
bit for bit, to the wave schedule's, and a chunk's S steps run in S
consecutive waves; both match the oracle (rel-L2 <= 3e-2 on the final latent
and on its displacement)."""
import numpy as np
import pytest

import synth
from _harness import rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FLAG_LATENCY = 8


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_latency_mode_equals_wave_mode_bitwise(name):
    cfg = synth.config(name)
    w = synth.make_weights(cfg, 0)
    streams = synth.make_streams(cfg, 2)
    n = 6
    waves_out, n_waves = run_gpu(cfg, w, streams, n)
    lat_out, n_lat = run_gpu(cfg, w, streams, n, flags=FLAG_LATENCY)
    assert n_waves == n + cfg["S"] - 1
    assert n_lat == n * cfg["S"]
    ora = run_oracle(cfg, w, streams, n)
    for i in range(2):
        for c in range(n):
            assert np.array_equal(waves_out[i][c], lat_out[i][c]), (i, c)
            x0 = streams[i].noise(c).astype(np.float64)
            assert rel_l2(lat_out[i][c], ora[i][c]) <= 3e-2, (i, c)
            assert rel_l2(lat_out[i][c] - x0, ora[i][c] - x0) <= 3e-2, (i, c)
