"""CPU oracle of the task DAG, the wave plan and the KV ring (brute force).

TEST INFRASTRUCTURE: see ``oracle/model.py``.

The DAG (AREX article "vLLM 与 Physis-AI 联合介绍 PhysisServe 推理系统",
§难题 and §三层设计; BAAI announcement "智源悟界·PhysisServe", Fig. 1 and
Fig. 2): stage k of chunk c may run once chunk c has finished stage k-1 and
chunk c-1 has finished stage k.  With stages = denoising steps this is the
(chunk, step) task DAG the single-GPU wave runs; with stages = steps x blocks
it is the pages' one-stage-per-GPU pipeline (Fig. 2 draws 2 steps x 4 blocks
= 8 stages).

Everything here is found by scanning all tasks and testing the definition,
never by a closed form, so that closed forms can be checked against it.
"""
from __future__ import annotations


def ready_tasks(n_stages: int, submitted: list, done: set) -> list:
    """All tasks (sid, c, k) whose dependencies are met, by definition.

    ``submitted[sid]`` chunks of stream ``sid`` have been submitted (their
    noise exists); ``done`` is the set of finished (sid, c, k).
    Order: stream ascending, then stage ascending (a fixed tie-break; any
    fixed order is correct, the CUDA path must use the same one).
    """
    out = []
    for sid, n in enumerate(submitted):
        for c in range(n):
            for k in range(n_stages):
                if (sid, c, k) in done:
                    continue
                if k > 0 and (sid, c, k - 1) not in done:
                    continue
                if c > 0 and (sid, c - 1, k) not in done:
                    continue
                out.append((sid, c, k))
    out.sort(key=lambda t: (t[0], t[2], t[1]))
    return out


def oldest_per_stream(tasks: list) -> list:
    """Latency order: of the ready tasks, only each stream's oldest chunk
    (lowest c) runs, so a chunk goes through its stages back to back."""
    best = {}
    for t in tasks:
        if t[0] not in best or t[1] < best[t[0]][1]:
            best[t[0]] = t
    return [t for t in tasks if best[t[0]] is t]


class WaveSimulator:
    """Runs waves: every ready task runs (or, with ``latency``, each stream's
    oldest ready chunk only); all finish before the next wave."""

    def __init__(self, n_stages: int, latency: bool = False):
        self.n_stages = n_stages
        self.latency = latency
        self.submitted = []
        self.done = set()

    def open_stream(self) -> int:
        self.submitted.append(0)
        return len(self.submitted) - 1

    def submit(self, sid: int, n: int = 1):
        self.submitted[sid] += n

    def wave(self) -> list:
        tasks = ready_tasks(self.n_stages, self.submitted, self.done)
        if self.latency:
            tasks = oldest_per_stream(tasks)
        self.done.update(tasks)
        return tasks


def stage_pipeline_outputs(n_stages: int, n_chunks: int) -> list:
    """Interval index at which each chunk leaves the last stage.

    All chunks are available up front and every ready (chunk, stage) runs in
    each interval (one stage per GPU never holds two tasks at once, because
    chunk c+1 cannot be ready at stage k before chunk c finished it).
    """
    sim = WaveSimulator(n_stages)
    sid = sim.open_stream()
    sim.submit(sid, n_chunks)
    finished = {}
    interval = 0
    while len(finished) < n_chunks:
        for (_, c, k) in sim.wave():
            if k == n_stages - 1:
                finished[c] = interval
        interval += 1
    return [finished[c] for c in range(n_chunks)]


class KVRing:
    """One (stream, block, step) KV ring of W+1 slots, simulated by occupancy.

    A chunk writes into the lowest empty slot, else into the slot whose
    chunk has left the window (older than c - W).  After the write the
    occupied slots must hold exactly chunks max(0, c-W)..c.
    """

    def __init__(self, W: int):
        self.W = W
        self.slots = [None] * (W + 1)

    def write(self, c: int):
        """Returns (slot, kv_chunks) where kv_chunks = occupied slots' chunks."""
        target = None
        for i, occ in enumerate(self.slots):
            if occ is None:
                target = i
                break
        if target is None:
            for i, occ in enumerate(self.slots):
                if occ < c - self.W:
                    target = i
                    break
        if target is None:
            raise RuntimeError("ring overflow: no slot left the window")
        self.slots[target] = c
        window = sorted(x for x in self.slots if x is not None)
        if window != list(range(max(0, c - self.W), c + 1)):
            raise RuntimeError(f"ring window {window} is not chunks {max(0, c - self.W)}..{c}")
        return target, window
