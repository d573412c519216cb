"""Kernel-level parity of the window attention (psv_attention, through the C
ABI) against the oracle's explicit-softmax attention on the same bf16 inputs.

Cases span: dh 32 / 64 / 128, ragged query tiles (T not a multiple of 128
or 256), ragged key tiles, windows long enough to take the two-pair key split
(>= 64 key tiles of 256) and the single-key degenerate case.  Tolerance: rel-L2 <=
1e-2 per query block (bf16 P and bf16 output against f64).
"""
import numpy as np
import pytest

import synth
from _harness import rel_l2
from oracle import model as M

pytestmark = pytest.mark.gpu


def _bf16(x):
    return synth.round_to_bf16(np.asarray(x, dtype=np.float32))


def make_problem(n, T, H, dh, L, k_rows=None, vt_cols=None, seed=0):
    rng = np.random.default_rng(seed)
    d = H * dh
    k_rows = k_rows or L
    vt_cols = vt_cols or (L + 7) // 8 * 8
    q = _bf16(rng.standard_normal((n * T, d)) * 1.5)
    k = _bf16(rng.standard_normal((n, k_rows, d)))
    v = _bf16(rng.standard_normal((n, L, d)))
    vt = np.zeros((n, H, dh, vt_cols), dtype=np.float32)
    for i in range(n):
        vt[i, :, :, :L] = v[i].reshape(L, H, dh).transpose(1, 2, 0)
    return dict(n=n, T=T, H=H, dh=dh, L=L, k_rows=k_rows, vt_cols=vt_cols, q=q, k=k, v=v, vt=vt)


def run_op(pb, call=None):
    import torch
    from autoregressive_denoising_dit_gb300 import _psv as P

    prob = P.AttnProblem(n=pb["n"], T=pb["T"], H=pb["H"], dh=pb["dh"], L=pb["L"],
                         k_rows=pb["k_rows"], vt_cols=pb["vt_cols"])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype=torch.bfloat16)
    q, k, vt = dev(pb["q"]), dev(pb["k"]), dev(pb["vt"])
    o = torch.zeros_like(q)
    if call is None:
        nbytes = P.psv_attention_scratch_bytes(prob)
        scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
        base = (scratch.data_ptr() + 255) // 256 * 256
        P.psv_attention(prob, q.data_ptr(), k.data_ptr(), vt.data_ptr(), o.data_ptr(), base, nbytes,
                        torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        off = base - scratch.data_ptr()
        err = int(scratch[off:off + 4].cpu().numpy().view(np.int32)[0])
        assert err == 0, f"device error word {err}"
    else:
        call(prob, q, k, vt, o)
        torch.cuda.synchronize()
    return o.float().cpu().numpy()


def oracle(pb):
    T, H, dh, L = pb["T"], pb["H"], pb["dh"], pb["L"]
    out = []
    for i in range(pb["n"]):
        qi = pb["q"][i * T:(i + 1) * T].astype(np.float64)
        out.append(M.attention(qi, pb["k"][i, :L].astype(np.float64), pb["v"][i].astype(np.float64), H, dh))
    return np.concatenate(out)


CASES = [
    dict(n=2, T=200, H=2, dh=128, L=600),                              # ragged, no split
    dict(n=3, T=300, H=4, dh=64, L=2100, k_rows=2200, vt_cols=2240),   # ragged, tail query unit
    dict(n=1, T=64, H=4, dh=32, L=256),                                # dh = 32 (64-byte swizzle)
    dict(n=2, T=1560, H=2, dh=128, L=7800),                            # full-size window
    dict(n=8, T=300, H=8, dh=64, L=2100),                              # 192 work pieces > 76 pairs
    dict(n=2, T=300, H=2, dh=64, L=16500, k_rows=16600, vt_cols=16512),  # split, ragged last tile
    dict(n=2, T=130, H=1, dh=128, L=1),                                # single key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"n{c['n']}T{c['T']}H{c['H']}dh{c['dh']}L{c['L']}")
def test_attention_op_matches_oracle(case):
    pb = make_problem(**case)
    got = run_op(pb)
    ref = oracle(pb)
    T = pb["T"]
    for i in range(pb["n"]):
        e = rel_l2(got[i * T:(i + 1) * T], ref[i * T:(i + 1) * T])
        assert e <= 1e-2, (i, e)
    if pb["L"] == 1:
        # one key: every query returns that key's value (bf16 of it)
        np.testing.assert_allclose(got, np.repeat(pb["v"][:, 0], T, axis=0), rtol=0, atol=0)


def test_attention_op_rejects_bad_shapes():
    from autoregressive_denoising_dit_gb300 import _psv as P

    bad = P.AttnProblem(n=1, T=64, H=2, dh=96, L=64, k_rows=64, vt_cols=64)
    with pytest.raises(P.PSVError):
        P.psv_attention_scratch_bytes(bad)
    bad = P.AttnProblem(n=1, T=64, H=2, dh=64, L=65, k_rows=64, vt_cols=72)
    with pytest.raises(P.PSVError):
        P.psv_attention_scratch_bytes(bad)


def test_split_key_path_is_batch_invariant():
    """A long window (split into two key halves merged in a fixed order) gives
    the same bits for a problem alone and inside a batch of three."""
    big = make_problem(n=3, T=300, H=2, dh=64, L=16500, seed=3)
    one = {k: (v[:1] if k in ("k", "v", "vt") else v) for k, v in big.items()}
    one["n"] = 1
    one["q"] = big["q"][:300]
    got3 = run_op(big)
    got1 = run_op(one)
    np.testing.assert_array_equal(got1, got3[:300])
