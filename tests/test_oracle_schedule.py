"""Pins of the oracle's brute-force DAG / wave / ring simulators.

Checked against closed forms (the anti-diagonal w = c + s, the longest-path
recurrence under staggered submission, slot = c mod (W+1)) and against the
worked pipeline example the pages print (tests/golden/stage_pipeline_fig2.txt).
"""
import os

import pytest

from oracle.schedule import KVRing, WaveSimulator, ready_tasks, stage_pipeline_outputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "stage_pipeline_fig2.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def test_pages_worked_pipeline_example():
    g = _golden()
    assert g["n_stages"] == g["n_steps"] * g["n_blocks"] == g["n_gpus"]
    n_chunks = 12
    out = stage_pipeline_outputs(g["n_stages"], n_chunks)
    # the first chunk walks all 8 stages: it leaves the last one in interval 7
    assert out[0] == g["n_stages"] - 1
    # afterwards one chunk per interval
    gaps = [b - a for a, b in zip(out, out[1:])]
    assert gaps == [g["outputs_per_interval_after_fill"]] * (n_chunks - 1)


@pytest.mark.parametrize("S,N,n_streams", [(2, 6, 1), (4, 9, 1), (4, 5, 3), (1, 4, 2), (3, 1, 2)])
def test_all_submitted_waves_are_antidiagonals(S, N, n_streams):
    sim = WaveSimulator(S)
    for _ in range(n_streams):
        sim.submit(sim.open_stream(), N)
    w = 0
    while True:
        tasks = sim.wave()
        if not tasks:
            break
        expect = sorted(((sid, c, s) for sid in range(n_streams) for s in range(S)
                         for c in [w - s] if 0 <= c < N), key=lambda t: (t[0], t[2]))
        assert tasks == expect
        w += 1
    assert w == N + S - 1
    # first output at wave S-1, then one chunk per stream per wave
    assert len(sim.done) == n_streams * N * S


def _longest_path_waves(arrivals, S):
    """r(c, s) = max(r(c, s-1), r(c-1, s)) + 1 with r(c, -1) = a_c - 1 and
    r(-1, s) = -1, where chunk c is submitted before wave a_c."""
    r = {}
    for c, a in enumerate(arrivals):
        for s in range(S):
            left = r[(c, s - 1)] if s > 0 else a - 1
            up = r[(c - 1, s)] if c > 0 else -1
            r[(c, s)] = max(left, up) + 1
    return r


@pytest.mark.parametrize("arrivals,S", [([0, 0, 3, 3, 4, 9], 4), ([0, 5, 5, 6], 2), ([2, 2, 2], 3)])
def test_staggered_submission_matches_longest_path(arrivals, S):
    sim = WaveSimulator(S)
    sid = sim.open_stream()
    expect = _longest_path_waves(arrivals, S)
    got = {}
    w = 0
    while len(got) < len(arrivals) * S:
        sim.submit(sid, sum(1 for a in arrivals if a == w))
        for (_, c, s) in sim.wave():
            got[(c, s)] = w
        w += 1
        assert w < 100
    assert got == expect


def test_ready_set_never_holds_two_tasks_of_one_stream_step():
    sim = WaveSimulator(3)
    a, b = sim.open_stream(), sim.open_stream()
    sim.submit(a, 5)
    for w in range(12):
        if w == 2:
            sim.submit(b, 4)
        tasks = sim.wave()
        keys = [(t[0], t[2]) for t in tasks]
        assert len(keys) == len(set(keys))


def test_ready_tasks_order_and_definition():
    done = {(0, 0, 0), (0, 0, 1), (0, 1, 0), (1, 0, 0)}
    got = ready_tasks(3, [3, 2], done)
    assert got == [(0, 2, 0), (0, 1, 1), (0, 0, 2), (1, 1, 0), (1, 0, 1)]


@pytest.mark.parametrize("W", [0, 1, 3, 4])
def test_ring_slots_are_c_mod_window(W):
    ring = KVRing(W)
    for c in range(40):
        slot, window = ring.write(c)
        assert slot == c % (W + 1)
        assert window == list(range(max(0, c - W), c + 1))
        # the occupied slots are the prefix [0, len(window))
        occ = [i for i, x in enumerate(ring.slots) if x is not None]
        assert occ == list(range(len(window)))
