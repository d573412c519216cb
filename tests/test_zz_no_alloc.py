"""The allocation-free attention entry point (psv_attention_noalloc).

It is for callers that cannot allocate device memory when they call (a
control loop that must not enter the CUDA allocator after start-up, or a
framework that owns all device memory); its scratch is a fixed array inside
the library.  Checked through the C ABI against psv_attention (caller
scratch) on the same inputs, on two calls in a row (the second call reuses
the array the first one left behind), with the call's status word read back
after each.  Kept in its own file, collected last.
"""
import numpy as np
import pytest

from _harness import rel_l2
from test_gpu_attention_op import make_problem, run_op

pytestmark = pytest.mark.gpu


def test_noalloc_matches_caller_scratch_on_two_calls():
    import torch
    from autoregressive_denoising_dit_gb300 import _psv as P

    # L = 16500: split-key path, so partials and counters are used
    pb = make_problem(n=2, T=300, H=2, dh=64, L=16500, k_rows=16600, vt_cols=16512, seed=7)
    prob = P.AttnProblem(n=pb["n"], T=pb["T"], H=pb["H"], dh=pb["dh"], L=pb["L"],
                         k_rows=pb["k_rows"], vt_cols=pb["vt_cols"])
    assert P.psv_attention_scratch_bytes(prob) <= P.PSV_ATTN_NOALLOC_SCRATCH_BYTES
    ref = run_op(pb)  # existing entry point, caller-provided scratch

    def noalloc(prob, q, k, vt, o):
        P.psv_attention_noalloc(prob, q.data_ptr(), k.data_ptr(), vt.data_ptr(), o.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)

    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        got = run_op(pb, call=noalloc)
        # no device-side wait of the call gave up (the word is read from the
        # library's own array, after the stream's work is done)
        assert P.psv_attention_noalloc_status(stream) == 0
        T = pb["T"]
        for i in range(pb["n"]):
            assert rel_l2(got[i * T:(i + 1) * T], ref[i * T:(i + 1) * T]) <= 1e-2
        np.testing.assert_array_equal(got, ref)


def test_noalloc_rejects_problems_over_the_fixed_scratch():
    from autoregressive_denoising_dit_gb300 import _psv as P

    big = P.AttnProblem(n=16, T=1560, H=12, dh=128, L=7800, k_rows=7800, vt_cols=7808)
    assert P.psv_attention_scratch_bytes(big) > P.PSV_ATTN_NOALLOC_SCRATCH_BYTES
    with pytest.raises(P.PSVError) as e:
        P.psv_attention_noalloc(big, 16, 16, 16, 16, 0)
    assert e.value.code == P.PSV_ENOMEM
