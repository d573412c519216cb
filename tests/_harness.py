"""Shared helpers of the GPU parity tests: run a configuration through the
C ABI (libpsv) and through the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import synth
from oracle.runner import OracleRunner


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def weight_items(weights: dict):
    for name, arr in weights["global"].items():
        yield -1, name, arr
    for b, bw in enumerate(weights["blocks"]):
        for name, arr in bw.items():
            yield b, name, arr


def gpu_session(cfg, weights, n_streams, flags=0, max_inflight=0):
    from autoregressive_denoising_dit_gb300 import Session

    s = Session(cfg, max_streams=n_streams, max_inflight=max_inflight, flags=flags)
    s.load_host_weights(weight_items(weights))
    return s


def run_gpu(cfg, weights, streams, n_chunks, flags=0, conds=None, noises=None, chunk_conds=None):
    """outputs[sid][c] of a full run: every chunk submitted up front, waves
    until idle, then every chunk polled.  chunk_conds[sid] = {c: vector}
    submits those chunks with their own conditioning."""
    n_streams = len(streams)
    sess = gpu_session(cfg, weights, n_streams, flags, max_inflight=n_chunks + cfg["S"])
    try:
        for i, st in enumerate(streams):
            sid = sess.open_stream(st.cond if conds is None else conds[i])
            assert sid == i
            for c in range(n_chunks):
                x0 = st.noise(c) if noises is None else noises[i][c]
                cc = None if chunk_conds is None else chunk_conds[i].get(c)
                sess.submit(sid, np.ascontiguousarray(x0, dtype=np.float32),
                            None if cc is None else np.ascontiguousarray(cc, dtype=np.float32))
        waves = 0
        while sess.run_wave():
            waves += 1
        sess.sync(60000)
        outs = []
        for sid in range(n_streams):
            per = []
            for c in range(n_chunks):
                buf = np.empty((cfg["T"], cfg["C"]), dtype=np.float32)
                got = sess.poll(sid, buf)
                assert got == c
                per.append(buf)
            outs.append(per)
        return outs, waves
    finally:
        sess.close()


def run_oracle(cfg, weights, streams, n_chunks, dtype=np.float64, conds=None, noises=None,
               chunk_conds=None):
    r = OracleRunner(cfg, weights, dtype)
    for i, st in enumerate(streams):
        r.open_stream(st.cond if conds is None else conds[i])
        for c in range(n_chunks):
            r.submit(i, st.noise(c) if noises is None else noises[i][c],
                     cond=None if chunk_conds is None else chunk_conds[i].get(c))
    r.run_until_idle()
    return [[r.streams[i].outputs[c] for c in range(n_chunks)] for i in range(len(streams))]
