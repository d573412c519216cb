"""Failure paths of the C ABI on the GPU, reached without any device fault.

  * psv_sync with a zero deadline, right after several waves were issued,
    returns PSV_ETIMEDOUT (host-side polling only); the error is not sticky
    and the waves still finish with correct results;
  * a device error word raised from the host (a plain write into the arena,
    as a kernel does when one of its bounded waits gives up) makes
    psv_poll_chunk return PSV_EDEVICE, and every later call returns it too
    (sticky).  No kernel is made to time out or fault.
"""
import numpy as np
import pytest

import synth
from _harness import gpu_session, rel_l2, run_oracle

pytestmark = pytest.mark.gpu

PSV_ETIMEDOUT = -4
PSV_EDEVICE = -6


def test_sync_deadline_returns_etimedout_and_is_not_sticky():
    from autoregressive_denoising_dit_gb300 import Session, _psv as P

    # the 1.3B-shaped block at full width, 4 blocks: a wave takes milliseconds
    cfg = synth.config("wan21_1p3b", B=4)
    n = 8
    sess = Session(cfg, max_streams=1, max_inflight=n + cfg["S"])
    try:
        sess.load_device_weights(synth.iter_device_weights(cfg, seed=0))
        st = synth.make_streams(cfg, 1)[0]
        sid = sess.open_stream(st.cond)
        for c in range(n):
            sess.submit(sid, st.noise(c))
        issued = 0
        while sess.run_wave():
            issued += 1
        assert issued == n + cfg["S"] - 1
        with pytest.raises(P.PSVError) as e:
            sess.sync(0)
        assert e.value.code == PSV_ETIMEDOUT
        sess.sync(120000)  # not sticky: a later wait succeeds
        buf = np.empty((cfg["T"], cfg["C"]), dtype=np.float32)
        for c in range(n):
            assert sess.poll(sid, buf) == c
            assert np.all(np.isfinite(buf))
    finally:
        sess.close()


def test_device_error_word_gives_sticky_edevice():
    import torch
    from autoregressive_denoising_dit_gb300 import _psv as P

    cfg = synth.config("tiny")
    w = synth.make_weights(cfg, 0)
    st = synth.make_streams(cfg, 1)[0]
    ref = run_oracle(cfg, w, [st], 2)[0]
    sess = gpu_session(cfg, w, 1, max_inflight=2 + cfg["S"])
    try:
        sid = sess.open_stream(st.cond)
        sess.submit(sid, st.noise(0))
        sess.submit(sid, st.noise(1))
        while sess.run_wave():
            pass
        sess.sync(60000)
        buf = np.empty((cfg["T"], cfg["C"]), dtype=np.float32)
        assert sess.poll(sid, buf) == 0          # clean so far
        assert rel_l2(buf, ref[0]) <= 3e-2
        off = P.psv_debug_error_word(sess.ctx)
        idx = sess.arena_ptr - sess._arena.data_ptr() + off
        torch.cuda.synchronize()
        sess._arena[idx:idx + 4] = torch.tensor([7, 0, 0, 0], dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        with pytest.raises(P.PSVError) as e:
            sess.poll(sid, buf)
        assert e.value.code == PSV_EDEVICE
        # sticky: every later call reports it, whatever it is
        for call in (lambda: sess.poll(sid, buf), lambda: sess.run_wave(), lambda: sess.sync(1000)):
            with pytest.raises(P.PSVError) as e:
                call()
            assert e.value.code == PSV_EDEVICE
    finally:
        sess.close()
