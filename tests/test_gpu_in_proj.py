"""In-projection on the tensor cores against the oracle's f64 definition.

h = x W_inᵀ + b_in opens every (chunk, step) task (BAAI announcement, Fig. 1: each
chunk is denoised from its submitted noise); x is the f32 latent, W_in bf16.  The
library runs it as one bf16 GEMM of [hi(x) | lo(x)] against [W_in | W_in], with
hi = bf16(x) and lo = bf16(x - hi): x - hi is exact in f32 and at most 2^-8 |x|, and
lo keeps it to 2^-8 relative, so hi + lo carries x to within 2^-16 relative and each
product with a bf16 weight is exact in the f32 accumulator.  The result must therefore match the f64 definition
to f32 accumulation error, two orders of magnitude tighter than a plain bf16 product
of x (~4e-3 relative).  The block-0 tap of the first wave (one task: chunk 0, step 0)
captures h as the in-projection wrote it.

Cases: the three channel counts of the configurations (C = 16, 64, 192 -> K = 64, 128,
384 after the split), a nonzero bias, and latents far from N(0, 1) (large offsets and
magnitudes spanning several binades), which a split without the low part would get
wrong by ~1e-3.
"""
import numpy as np
import pytest

import synth
from _harness import rel_l2, weight_items
from oracle import model as M

pytestmark = pytest.mark.gpu

CASES = [("tiny", 1.0, 0.0), ("wan21_1p3b", 1.0, 0.0), ("wan22_5b", 1.0, 0.0),
         ("wan21_1p3b", 300.0, 37.0)]


def _tap_in_proj(cfg, weights, cond, x):
    import torch
    from autoregressive_denoising_dit_gb300 import Session, _psv as P

    T, d = cfg["T"], cfg["d"]
    sess = Session(cfg, max_streams=1, max_inflight=cfg["S"] + 2)
    try:
        sess.load_host_weights(weight_items(weights))
        sid = sess.open_stream(cond)
        sess.submit(sid, x)
        h_in = torch.empty(T * d, dtype=torch.float32, device="cuda")
        h_out = torch.empty_like(h_in)
        P.psv_debug_tap(sess.ctx, 0, h_in.data_ptr(), h_out.data_ptr())
        assert sess.run_wave() == 1
        sess.sync(120000)
        return h_in.cpu().numpy().reshape(T, d)
    finally:
        sess.close()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name,scale,offset", CASES,
                         ids=[f"{c[0]}-x{c[1]:g}+{c[2]:g}" for c in CASES])
def test_in_proj_matches_f64_definition(name, scale, offset):
    cfg = synth.config(name, B=1)
    weights = synth.make_weights(cfg, 0)
    rng = np.random.default_rng(7)
    weights["global"]["in_b"] = (0.5 * rng.standard_normal(cfg["d"])).astype(np.float32)
    st = synth.make_streams(cfg, 1)[0]
    x = st.noise(0).astype(np.float64) * scale + offset
    # magnitudes over several binades: scale each token row by 2^k, k in [-6, 6]
    x *= np.exp2(rng.integers(-6, 7, size=(cfg["T"], 1)))
    x = np.ascontiguousarray(x, dtype=np.float32)
    got = _tap_in_proj(cfg, weights, st.cond, x).astype(np.float64)
    g = {k: v.astype(np.float64) for k, v in weights["global"].items()}
    want = M.in_proj(g, x.astype(np.float64))
    assert np.all(np.isfinite(got))
    # hi + lo = x (1 + e), |e| <= 2^-16, and f32 accumulation over K = 2C terms: a few
    # 1e-6 relative in L2; x rounded to bf16 alone would be ~2e-3
    assert rel_l2(got, want) <= 2e-5, rel_l2(got, want)
    # elementwise against sum |x| |w| + |b|: 2^-16 from the split plus the accumulation
    bound = np.abs(x.astype(np.float64)) @ np.abs(g["in_w"]).T + np.abs(g["in_b"])
    assert np.max(np.abs(got - want) / bound) <= 5e-5
