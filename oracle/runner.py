"""CPU oracle driver: streams, chunks, steps, the noisy-KV store, wave order.

TEST INFRASTRUCTURE: see ``oracle/model.py``.

A stream is a sequence of chunks; chunk c step s runs every block in order
and, at block b, attends to its own tokens plus the keys and values that
chunks max(0, c-W)..c-1 stored at the same (block b, step s) — the
still-noisy KV of the pages (AREX article, §难题; BAAI announcement, Fig. 1).
The store is logical, keyed (block, step, chunk); there is no ring here.
"""
from __future__ import annotations

import numpy as np

from . import model as M
from .schedule import WaveSimulator


class OracleStream:
    def __init__(self, runner, cond: np.ndarray):
        cfg = runner.cfg
        self.mod, self.fmod = M.conditioning(cfg, runner.g, runner.blocks, cond, runner.dtype)
        self.x = {}        # chunk -> current latent [T, C]
        self.step = {}     # chunk -> next step to run
        self.kv = {}       # (b, s, c) -> (k, v)
        self.outputs = {}  # chunk -> x_S
        self.chunk_mod = {}  # chunk -> (mod, fmod) of a chunk submitted with its own cond
        self.n_submitted = 0


class OracleRunner:
    """Runs (chunk, step) tasks one at a time in float64 (or float32)."""

    def __init__(self, cfg: dict, weights: dict, dtype=np.float64):
        self.cfg = cfg
        self.dtype = dtype
        self.g = {k: v.astype(dtype) for k, v in weights["global"].items()}
        self.blocks = [{k: v.astype(dtype) for k, v in bw.items()} for bw in weights["blocks"]]
        self.streams = []
        self.ts = M.step_times(cfg["S"])
        self.sim = WaveSimulator(cfg["S"])
        self.task_log = []

    def open_stream(self, cond: np.ndarray) -> int:
        self.streams.append(OracleStream(self, cond))
        return self.sim.open_stream()

    def submit(self, sid: int, noise: np.ndarray, cond: np.ndarray | None = None):
        """Next chunk of stream sid.  ``cond`` gives this chunk its own
        conditioning vector, used at every step of the chunk in place of the
        stream's (reading <18>: an action-conditioned world model conditions
        each generated chunk on the agent's action — AREX article, section
        难题; BAAI announcement, section 新一代物理 AI 的基础设施)."""
        st = self.streams[sid]
        c = st.n_submitted
        if cond is not None:
            st.chunk_mod[c] = M.conditioning(self.cfg, self.g, self.blocks, cond, self.dtype)
        st.x[c] = noise.reshape(self.cfg["T"], self.cfg["C"]).astype(self.dtype)
        st.step[c] = 0
        st.n_submitted += 1
        self.sim.submit(sid, 1)

    def run_task(self, sid: int, c: int, s: int, tap=None):
        """Chunk c, step s of stream sid: in-proj, B blocks, final head, Euler.

        ``tap(b, h_in, h_out)`` if given sees every block's input and output.
        """
        cfg, st = self.cfg, self.streams[sid]
        assert st.step[c] == s, "task run out of order"
        W = cfg["W"]
        pos = M.positions(cfg, c)
        mod, fmod = st.chunk_mod.get(c, (st.mod, st.fmod))
        h = M.in_proj(self.g, st.x[c])
        for b in range(cfg["B"]):
            window = [st.kv[(b, s, cc)] for cc in range(max(0, c - W), c)]
            h_out, k, v = M.block_forward(cfg, self.blocks[b], mod[s, b], h, pos, window)
            if tap is not None:
                tap(b, h, h_out)
            st.kv[(b, s, c)] = (k, v)
            st.kv.pop((b, s, c - W - 1), None)
            h = h_out
        vel = M.final_velocity(cfg, self.g, fmod[s], h)
        st.x[c] = M.euler(st.x[c], vel, self.ts[s], self.ts[s + 1])
        st.step[c] = s + 1
        if s + 1 == cfg["S"]:
            st.outputs[c] = st.x.pop(c)
            st.chunk_mod.pop(c, None)
        self.task_log.append((sid, c, s))

    def run_wave(self) -> list:
        """All ready tasks, in the fixed (stream, step) order, one at a time."""
        tasks = self.sim.wave()
        for sid, c, s in tasks:
            self.run_task(sid, c, s)
        return tasks

    def run_until_idle(self) -> int:
        n = 0
        while self.run_wave():
            n += 1
        return n

    def run_sequential(self, sid: int):
        """Strictly sequential per-chunk order: chunk 0 all steps, chunk 1 ..."""
        st = self.streams[sid]
        for c in range(st.n_submitted):
            for s in range(st.step.get(c, self.cfg["S"]), self.cfg["S"]):
                self.run_task(sid, c, s)
