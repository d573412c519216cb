"""CPU tests of the C ABI: the library loads, exports every call psv.h
declares, validates descriptions, and its host scheduler (plan-only mode,
no device) matches the oracle's brute-force DAG and ring simulators
bit-exactly: task order, KV slots, window lengths, state slots."""
import os
import re

import numpy as np
import pytest

import synth
from autoregressive_denoising_dit_gb300 import _psv as P
from oracle.schedule import KVRing, WaveSimulator

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from autoregressive_denoising_dit_gb300 import build

    build.build()


def test_header_declarations_are_exported():
    hdr = open(os.path.join(ROOT, "include", "psv.h")).read()
    declared = set(re.findall(r"\b(psv_[a-z_]+)\s*\(", hdr))
    assert declared == set(P.EXPORTS)
    L = P.lib()
    for name in declared:
        assert hasattr(L, name), name
    syms = os.popen(f"nm -D --defined-only {P.LIB_PATH}").read()
    exported = {l.split()[-1] for l in syms.splitlines() if " T " in l}
    assert exported == declared, "only the psv_* calls may be exported"


def test_arena_bytes_and_validation():
    cfg = synth.config("wan21_1p3b")
    n = P.psv_arena_bytes(P.model_desc(cfg))
    # bf16 weights (~3.1 GB) + KV rings (5.75 GB) + activations
    assert 8.5e9 < n < 10.5e9
    bad = dict(cfg, dh=96, H=16)
    with pytest.raises(P.PSVError) as e:
        P.psv_arena_bytes(P.model_desc(bad))
    assert e.value.code == P.PSV_EINVAL and "dh" in str(e.value)
    with pytest.raises(P.PSVError):
        P.psv_arena_bytes(P.model_desc(dict(cfg, d=1000, H=10, dh=100)))


def _plan_ctx(cfg, max_streams, flags=0, max_inflight=0):
    return P.psv_create(P.model_desc(cfg, max_streams, max_inflight, P.PSV_FLAG_PLAN_ONLY | flags))


def _run_schedule(cfg, n_streams, events, latency=False):
    """events: list of ('submit', sid, k) / ('wave',) / ('poll', sid).
    Returns the list of wave plans from the library and the oracle."""
    W = cfg["W"]
    ctx = _plan_ctx(cfg, n_streams, P.PSV_FLAG_LATENCY if latency else 0, max_inflight=64)
    sim = WaveSimulator(cfg["S"], latency=latency)
    rings = {}
    for _ in range(n_streams):
        assert P.psv_open_stream(ctx, None) == sim.open_stream()
    lib_waves, ora_waves = [], []
    for ev in events:
        if ev[0] == "submit":
            for _ in range(ev[2]):
                P.psv_submit_chunk(ctx, ev[1], None)
            sim.submit(ev[1], ev[2])
        elif ev[0] == "wave":
            plan = P.psv_wave_plan(ctx)
            n = P.psv_run_wave(ctx)
            assert n == len(plan)
            tasks = sim.wave()
            exp = []
            for i, (sid, c, s) in enumerate(tasks):
                ring = rings.setdefault((sid, s), KVRing(W))
                slot, window = ring.write(c)
                exp.append((sid, c, s, slot, len(window) * cfg["T"], i * cfg["T"]))
            lib_waves.append([t[:6] for t in plan])
            ora_waves.append(exp)
    P.psv_destroy(ctx)
    return lib_waves, ora_waves


@pytest.mark.parametrize("name", ["tiny", "mid", "wan21_1p3b"])
def test_plan_matches_oracle_all_submitted(name):
    cfg = synth.config(name)
    n_streams = cfg["n_streams"]
    N = 9
    events = [("submit", s, N) for s in range(n_streams)] + [("wave",)] * (N + cfg["S"] + 2)
    lib_w, ora_w = _run_schedule(cfg, n_streams, events)
    assert lib_w == ora_w
    assert sum(len(w) for w in lib_w) == n_streams * N * cfg["S"]


def test_plan_matches_oracle_staggered_and_multistream():
    cfg = synth.config("mid", W=1, S=3)
    rng = np.random.default_rng(3)
    events = []
    for w in range(40):
        for sid in range(3):
            if rng.random() < 0.4:
                events.append(("submit", sid, int(rng.integers(1, 3))))
        events.append(("wave",))
    lib_w, ora_w = _run_schedule(cfg, 3, events)
    assert lib_w == ora_w


def test_window_zero_single_slot():
    cfg = synth.config("tiny", W=0)
    lib_w, ora_w = _run_schedule(cfg, 1, [("submit", 0, 5)] + [("wave",)] * 8)
    assert lib_w == ora_w
    assert all(t[3] == 0 and t[4] == cfg["T"] for w in lib_w for t in w)


def test_sequential_flag_runs_one_task_in_chunk_order():
    cfg = synth.config("tiny")
    ctx = _plan_ctx(cfg, 1, P.PSV_FLAG_SEQUENTIAL)
    sid = P.psv_open_stream(ctx, None)
    for _ in range(3):
        P.psv_submit_chunk(ctx, sid, None)
    order = []
    while True:
        plan = P.psv_wave_plan(ctx)
        if not plan:
            break
        assert P.psv_run_wave(ctx) == 1
        order.append(plan[0][1:3])
    assert order == [(c, s) for c in range(3) for s in range(cfg["S"])]
    P.psv_destroy(ctx)


def test_inflight_limit_and_poll_order():
    cfg = synth.config("tiny")
    ctx = _plan_ctx(cfg, 1, max_inflight=3)
    sid = P.psv_open_stream(ctx, None)
    for _ in range(3):
        P.psv_submit_chunk(ctx, sid, None)
    with pytest.raises(P.PSVError) as e:
        P.psv_submit_chunk(ctx, sid, None)
    assert e.value.code == P.PSV_EAGAIN
    assert P.psv_poll_chunk(ctx, sid, None) is None  # nothing finished yet
    got = []
    for _ in range(10):
        P.psv_run_wave(ctx)
        c = P.psv_poll_chunk(ctx, sid, None)
        if c is not None:
            got.append(c)
            P.psv_submit_chunk(ctx, sid, None)
    assert got == list(range(len(got))) and len(got) >= 5
    # state slots cycle through the in-flight window
    plan_slots = set()
    for _ in range(3):
        for t in P.psv_wave_plan(ctx):
            plan_slots.add(t[6])
        P.psv_run_wave(ctx)
    assert plan_slots <= {0, 1, 2}
    P.psv_destroy(ctx)


def test_stream_limit_and_errors():
    cfg = synth.config("tiny")
    ctx = _plan_ctx(cfg, 2)
    a = P.psv_open_stream(ctx, None)
    b = P.psv_open_stream(ctx, None)
    assert (a, b) == (0, 1)
    with pytest.raises(P.PSVError) as e:
        P.psv_open_stream(ctx, None)
    assert e.value.code == P.PSV_EAGAIN
    P.psv_close_stream(ctx, a)
    assert P.psv_open_stream(ctx, None) == 0
    with pytest.raises(P.PSVError) as e:
        P.psv_submit_chunk(ctx, 5, None)
    assert e.value.code == P.PSV_EINVAL
    with pytest.raises(P.PSVError):
        P.psv_load_weights(ctx, [(-1, "qkv_w", np.zeros(3 * 128 * 128, np.float32), P.PSV_LOC_HOST)])
    with pytest.raises(P.PSVError):
        P.psv_load_weights(ctx, [(-1, "in_w", np.zeros(7, np.float32), P.PSV_LOC_HOST)])
    P.psv_destroy(ctx)


def test_create_rejects_small_arena_without_device():
    cfg = synth.config("tiny")
    with pytest.raises(P.PSVError) as e:
        P.psv_create(P.model_desc(cfg), 0, 0, 0)
    assert e.value.code in (P.PSV_EINVAL, P.PSV_ENOMEM)


def test_chunk_conditioning_tables_in_plan():
    """A chunk submitted with its own conditioning reads table
    max_streams + state_slot at every step; the others read their stream's.
    Without PSV_FLAG_CHUNK_COND the call is refused, and the flag grows the
    arena by one table set per chunk slot."""
    cfg = synth.config("tiny")
    ctx = _plan_ctx(cfg, 2, P.PSV_FLAG_CHUNK_COND, max_inflight=8)
    s0 = P.psv_open_stream(ctx, None)
    s1 = P.psv_open_stream(ctx, None)
    P.psv_submit_chunk(ctx, s0, None)
    P.psv_submit_chunk_cond(ctx, s0, None, None)
    P.psv_submit_chunk_cond(ctx, s1, None, None)
    seen = {}
    while True:
        plan = P.psv_wave_plan(ctx, cond_tables=True)
        if not plan:
            break
        for (sid, c, s, slot, kv, row, state_slot, tab) in plan:
            want = sid if (sid, c) == (s0, 0) else 2 + state_slot
            assert tab == want, (sid, c, s, tab)
            seen[(sid, c, s)] = tab
        P.psv_run_wave(ctx)
    assert len(seen) == 3 * cfg["S"]
    P.psv_destroy(ctx)
    ctx = _plan_ctx(cfg, 1)
    sid = P.psv_open_stream(ctx, None)
    with pytest.raises(P.PSVError) as e:
        P.psv_submit_chunk_cond(ctx, sid, None, None)
    assert e.value.code == P.PSV_EINVAL
    P.psv_destroy(ctx)
    base = P.psv_arena_bytes(P.model_desc(cfg, 2, 8))
    more = P.psv_arena_bytes(P.model_desc(cfg, 2, 8, P.PSV_FLAG_CHUNK_COND))
    per_slot = cfg["S"] * (cfg["B"] * 6 + 2) * cfg["d"] * 4  # mod + fmod tables of one slot
    assert more - base >= 16 * per_slot


def _steady_flops(cfg, n_tasks):
    T, d, F, C, B = cfg["T"], cfg["d"], cfg["F"], cfg["C"], cfg["B"]
    Lk = (cfg["W"] + 1) * T
    return n_tasks * (2 * T * B * (4 * d * d + 2 * d * F) + 4 * T * Lk * d * B + 4 * T * C * d)


def test_admission_control_without_measurements():
    """Admission (one GPU, no migration): a stream is admitted only while a KV
    ring set is free and the predicted shared wave time meets its SLO and
    every admitted stream's SLO.  Without timed waves the prediction is the
    steady wave's algorithmic FLOPs at 1 PFLOP/s."""
    cfg = synth.config("tiny")
    ctx = _plan_ctx(cfg, 3)
    p1 = P.psv_predict_wave_ms(ctx, 1)
    assert abs(p1 - _steady_flops(cfg, cfg["S"]) / 1e15 * 1e3) < 1e-12 * max(1.0, p1)
    assert abs(P.psv_predict_wave_ms(ctx, 3) - 3 * p1) < 1e-9 * p1
    with pytest.raises(P.PSVError):
        P.psv_predict_wave_ms(ctx, 4)
    # the stream's own SLO
    with pytest.raises(P.PSVError) as e:
        P.psv_admit_stream(ctx, None, 0.5 * p1)
    assert e.value.code == P.PSV_EAGAIN and "SLO" in str(e.value)
    a, pa = P.psv_admit_stream(ctx, None, 2.0 * p1)      # tight: fits two streams
    assert abs(pa - p1) < 1e-9 * p1
    b, pb = P.psv_admit_stream(ctx, None, 0.0)           # no SLO of its own
    assert abs(pb - 2 * p1) < 1e-9 * p1
    with pytest.raises(P.PSVError) as e:                  # would break stream a's SLO
        P.psv_admit_stream(ctx, None, 0.0)
    assert e.value.code == P.PSV_EAGAIN and f"stream {a}" in str(e.value)
    P.psv_close_stream(ctx, b)
    c, pc = P.psv_admit_stream(ctx, None, 10 * p1)       # the freed ring set
    assert c == b and abs(pc - 2 * p1) < 1e-9 * p1
    P.psv_destroy(ctx)
    ctx = _plan_ctx(cfg, 1)
    P.psv_admit_stream(ctx, None, 0.0)
    with pytest.raises(P.PSVError) as e:
        P.psv_admit_stream(ctx, None, 0.0)
    assert e.value.code == P.PSV_EAGAIN and "ring" in str(e.value)
    P.psv_destroy(ctx)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_latency_mode_plan_matches_oracle(name):
    """Latency mode: each stream's oldest ready chunk only, so with all
    chunks submitted chunk c step s runs in wave c*S + s (its S steps back to
    back); with staggered submissions the library matches the oracle's
    brute-force simulator of the same rule."""
    cfg = synth.config(name)
    N, S = 5, cfg["S"]
    lib_w, ora_w = _run_schedule(cfg, 1, [("submit", 0, N)] + [("wave",)] * (N * S + 2), latency=True)
    assert lib_w == ora_w
    for w, plan in enumerate(lib_w[: N * S]):
        assert [(t[1], t[2]) for t in plan] == [(w // S, w % S)]
    assert lib_w[N * S:] == [[], []]
    rng = np.random.default_rng(5)
    events = []
    for _ in range(40):
        for sid in range(3):
            if rng.random() < 0.3:
                events.append(("submit", sid, int(rng.integers(1, 3))))
        events.append(("wave",))
    lib_w, ora_w = _run_schedule(synth.config(name, W=1), 3, events, latency=True)
    assert lib_w == ora_w
    assert all(len({t[0] for t in plan}) == len(plan) for plan in lib_w)
