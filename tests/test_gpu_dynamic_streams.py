"""Dynamic streams on one GPU through the C ABI: streams admitted and closed
mid-run (psv_admit_stream / psv_close_stream) do not disturb the streams
already running, and a reused ring set starts clean.  Batch invariance makes
this exact: every stream's outputs equal, bit for bit, a run of that stream
alone, and they match the oracle (which runs each stream by itself) within
the end-to-end tolerance, rel-L2 <= 3e-2 on the final latent and on its
displacement.  The admission model's prediction after timed steady waves
comes from the measured wave time."""
import numpy as np
import pytest

import synth
from _harness import gpu_session, rel_l2, run_oracle

pytestmark = pytest.mark.gpu


def _alone(cfg, w, st, n):
    sess = gpu_session(cfg, w, 1, max_inflight=n + cfg["S"])
    try:
        sid = sess.open_stream(st.cond)
        for c in range(n):
            sess.submit(sid, st.noise(c))
        while sess.run_wave():
            pass
        sess.sync(60000)
        out = []
        for c in range(n):
            buf = np.empty((cfg["T"], cfg["C"]), dtype=np.float32)
            assert sess.poll(sid, buf) == c
            out.append(buf)
        return out
    finally:
        sess.close()


def _poll_all(cfg, sess, sid, n, out):
    while len(out) < n:
        buf = np.empty((cfg["T"], cfg["C"]), dtype=np.float32)
        if sess.poll(sid, buf) is None:
            return
        out.append(buf)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_streams_admitted_and_closed_mid_run(name):
    cfg = synth.config(name)
    w = synth.make_weights(cfg, 0)
    sa, sb, sc = synth.make_streams(cfg, 3)
    n = 7
    sess = gpu_session(cfg, w, 2, max_inflight=n + cfg["S"])
    try:
        a, _ = sess.admit_stream(sa.cond, 0.0)
        for c in range(n):
            sess.submit(a, sa.noise(c))
        for _ in range(3):
            sess.run_wave()
        b, _ = sess.admit_stream(sb.cond, 0.0)          # joins while a is mid-stream
        for c in range(n):
            sess.submit(b, sb.noise(c))
        out = {a: [], b: []}
        while sess.run_wave():
            sess.sync(60000)
            _poll_all(cfg, sess, a, n, out[a])
            _poll_all(cfg, sess, b, n, out[b])
        sess.sync(60000)
        _poll_all(cfg, sess, a, n, out[a])
        _poll_all(cfg, sess, b, n, out[b])
        sess.close_stream(b)
        c_id, _ = sess.admit_stream(sc.cond, 0.0)       # reuses b's ring set
        assert c_id == b
        for c in range(n):
            sess.submit(c_id, sc.noise(c))
        out_c = []
        while sess.run_wave():
            pass
        sess.sync(60000)
        _poll_all(cfg, sess, c_id, n, out_c)
    finally:
        sess.close()
    for got, st in ((out[a], sa), (out[b], sb), (out_c, sc)):
        ref = _alone(cfg, w, st, n)
        ora = run_oracle(cfg, w, [st], n)[0]
        assert len(got) == n
        for c in range(n):
            assert np.array_equal(got[c], ref[c]), c
            x0 = st.noise(c).astype(np.float64)
            assert rel_l2(got[c], ora[c]) <= 3e-2, c
            assert rel_l2(got[c] - x0, ora[c] - x0) <= 3e-2, c


def test_prediction_uses_measured_steady_waves():
    cfg = synth.config("mid")
    w = synth.make_weights(cfg, 0)
    st = synth.make_streams(cfg, 1)[0]
    n = 24
    sess = gpu_session(cfg, w, 2, max_inflight=n + cfg["S"])
    try:
        flops_model = sess.predict_wave_ms(1)
        sid = sess.open_stream(st.cond)
        for c in range(n):
            sess.submit(sid, st.noise(c))
        while sess.run_wave():
            pass
        sess.sync(60000)
        measured = sess.predict_wave_ms(1)
        assert measured != flops_model and 0.0 < measured < 100.0
        # two streams: the one measured count scaled by the algorithmic FLOPs
        assert abs(sess.predict_wave_ms(2) - 2 * measured) < 1e-9 * measured
    finally:
        sess.close()
