"""ctypes binding of libpsv (include/psv.h): argument marshalling only.

Every compute step runs inside libpsv.so; this module converts Python/numpy
arguments to the C types, raises ``PSVError`` for negative status codes and
returns plain Python values.  Importing it does not load the library; the
first call does, and fails loudly if ``libpsv.so`` was not built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpsv.so")

PSV_OK = 0
PSV_EINVAL = -1
PSV_ENOMEM = -2
PSV_EAGAIN = -3
PSV_ETIMEDOUT = -4
PSV_ECUDA = -5
PSV_EDEVICE = -6

PSV_FLAG_PLAN_ONLY = 1
PSV_FLAG_SEQUENTIAL = 2
PSV_FLAG_CHUNK_COND = 4
PSV_FLAG_LATENCY = 8

PSV_DTYPE_F32 = 0
PSV_DTYPE_BF16 = 1
PSV_LOC_HOST = 0
PSV_LOC_DEVICE = 1

# tensor name -> weight id (names as in the synthetic weight generator)
WEIGHT_IDS = {
    "in_w": 0, "in_b": 1, "t1_w": 2, "t1_b": 3, "t2_w": 4, "t2_b": 5,
    "fmod_w": 6, "fmod_b": 7, "out_w": 8, "out_b": 9,
    "qkv_w": 16, "qkv_b": 17, "o_w": 18, "o_b": 19, "up_w": 20, "up_b": 21,
    "down_w": 22, "down_b": 23, "mod_w": 24, "mod_b": 25,
}

# Every exported entry point of psv.h.
EXPORTS = [
    "psv_arena_bytes", "psv_create", "psv_load_weights", "psv_open_stream",
    "psv_submit_chunk", "psv_submit_chunk_cond", "psv_run_wave", "psv_poll_chunk", "psv_sync",
    "psv_wave_plan", "psv_close_stream", "psv_predict_wave_ms", "psv_admit_stream",
    "psv_destroy", "psv_last_error",
    "psv_set_graphs", "psv_set_profiling", "psv_kernel_times", "psv_debug_tap",
    "psv_debug_read_kv", "psv_attention_scratch_bytes", "psv_attention",
    "psv_attention_noalloc", "psv_attention_noalloc_status", "psv_debug_error_word",
]

PSV_ATTN_NOALLOC_SCRATCH_BYTES = 16 << 20


class ModelDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "S", "d", "H", "dh", "F", "C", "T", "W",
                                              "max_streams", "max_inflight", "t_embed")] + \
               [("ln_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("flags", ctypes.c_int32)]


class Weight(ctypes.Structure):
    _fields_ = [("id", ctypes.c_int32), ("block", ctypes.c_int32), ("data", ctypes.c_void_p),
                ("dtype", ctypes.c_int32), ("location", ctypes.c_int32), ("numel", ctypes.c_int64)]


class Task(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("stream", "chunk", "step", "slot", "kv_len",
                                              "row_off", "state_slot", "cond_table")]

    def as_tuple(self):
        return (self.stream, self.chunk, self.step, self.slot, self.kv_len, self.row_off,
                self.state_slot)


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double)]


class AttnProblem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n", "T", "H", "dh", "L", "k_rows", "vt_cols")]


class PSVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libpsv error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpsv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "psv_arena_bytes": (i32, [ctypes.POINTER(ModelDesc), ctypes.POINTER(sz)]),
            "psv_create": (i32, [ctypes.POINTER(ModelDesc), vp, sz, vp, ctypes.POINTER(vp)]),
            "psv_load_weights": (i32, [vp, ctypes.POINTER(Weight), i32]),
            "psv_open_stream": (i32, [vp, vp, ctypes.POINTER(i32)]),
            "psv_submit_chunk": (i32, [vp, i32, vp]),
            "psv_submit_chunk_cond": (i32, [vp, i32, vp, vp]),
            "psv_run_wave": (i32, [vp, ctypes.POINTER(i32)]),
            "psv_poll_chunk": (i32, [vp, i32, vp, ctypes.POINTER(i64)]),
            "psv_sync": (i32, [vp, i32]),
            "psv_wave_plan": (i32, [vp, ctypes.POINTER(Task), i32, ctypes.POINTER(i32)]),
            "psv_close_stream": (i32, [vp, i32]),
            "psv_predict_wave_ms": (i32, [vp, i32, ctypes.POINTER(ctypes.c_double)]),
            "psv_admit_stream": (i32, [vp, vp, ctypes.c_double, ctypes.POINTER(i32),
                                       ctypes.POINTER(ctypes.c_double)]),
            "psv_destroy": (None, [vp]),
            "psv_last_error": (ctypes.c_char_p, [vp]),
            "psv_set_graphs": (i32, [vp, i32]),
            "psv_set_profiling": (i32, [vp, i32]),
            "psv_kernel_times": (i32, [vp, ctypes.POINTER(KernelTime), i32, ctypes.POINTER(i32)]),
            "psv_debug_tap": (i32, [vp, i32, vp, vp]),
            "psv_debug_read_kv": (i32, [vp, i32, i32, i32, vp, vp]),
            "psv_attention_scratch_bytes": (i32, [ctypes.POINTER(AttnProblem), ctypes.POINTER(sz)]),
            "psv_attention": (i32, [ctypes.POINTER(AttnProblem), vp, vp, vp, vp, vp, sz, vp]),
            "psv_attention_noalloc": (i32, [ctypes.POINTER(AttnProblem), vp, vp, vp, vp, vp]),
            "psv_attention_noalloc_status": (i32, [ctypes.POINTER(i32), vp]),
            "psv_debug_error_word": (i32, [vp, ctypes.POINTER(sz)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(ctx, code: int) -> int:
    if code < 0:
        raise PSVError(code, psv_last_error(ctx))
    return code


def _fptr(a: np.ndarray, n: int | None = None):
    if a.dtype != np.float32 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError("expected a C-contiguous float32 array")
    if n is not None and a.size != n:
        raise ValueError(f"expected {n} elements, got {a.size}")
    return a.ctypes.data_as(ctypes.c_void_p)


def model_desc(cfg: dict, max_streams: int | None = None, max_inflight: int = 0,
               flags: int = 0) -> ModelDesc:
    """psv_model_desc of a configuration dict (keys B, S, d, H, dh, F, C, T, W)."""
    return ModelDesc(B=cfg["B"], S=cfg["S"], d=cfg["d"], H=cfg["H"], dh=cfg["dh"], F=cfg["F"],
                     C=cfg["C"], T=cfg["T"], W=cfg["W"],
                     max_streams=max_streams if max_streams is not None else cfg["n_streams"],
                     max_inflight=max_inflight, t_embed=cfg.get("t_embed", 256),
                     ln_eps=cfg.get("ln_eps", 1e-6), rope_theta=cfg.get("rope_theta", 1e4),
                     flags=flags)


# ------------------------------------------------------------------ calls

def psv_arena_bytes(desc: ModelDesc) -> int:
    n = ctypes.c_size_t()
    _check(None, lib().psv_arena_bytes(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def psv_create(desc: ModelDesc, arena_ptr: int = 0, arena_bytes: int = 0, stream_ptr: int = 0):
    ctx = ctypes.c_void_p()
    _check(None, lib().psv_create(ctypes.byref(desc), ctypes.c_void_p(arena_ptr or None),
                                  arena_bytes, ctypes.c_void_p(stream_ptr or None),
                                  ctypes.byref(ctx)))
    return ctx


def psv_load_weights(ctx, weights) -> None:
    """weights: iterable of (block, name, data, location); data is a float32
    numpy array (host) or (ptr, numel, dtype) for device tensors."""
    items, keep = [], []
    for block, name, data, loc in weights:
        if loc == PSV_LOC_HOST:
            arr = np.ascontiguousarray(data, dtype=np.float32)
            keep.append(arr)
            items.append(Weight(WEIGHT_IDS[name], block, arr.ctypes.data, PSV_DTYPE_F32,
                                PSV_LOC_HOST, arr.size))
        else:
            ptr, numel, dtype = data
            items.append(Weight(WEIGHT_IDS[name], block, ptr, dtype, PSV_LOC_DEVICE, numel))
    arr_t = (Weight * len(items))(*items)
    _check(ctx, lib().psv_load_weights(ctx, arr_t, len(items)))


def psv_open_stream(ctx, cond: np.ndarray | None) -> int:
    sid = ctypes.c_int()
    ptr = None if cond is None else _fptr(cond)
    _check(ctx, lib().psv_open_stream(ctx, ptr, ctypes.byref(sid)))
    return sid.value


def psv_submit_chunk(ctx, sid: int, noise: np.ndarray | None) -> None:
    ptr = None if noise is None else _fptr(noise)
    _check(ctx, lib().psv_submit_chunk(ctx, sid, ptr))


def psv_submit_chunk_cond(ctx, sid: int, noise: np.ndarray | None, cond: np.ndarray | None) -> None:
    pn = None if noise is None else _fptr(noise)
    pc = None if cond is None else _fptr(cond)
    _check(ctx, lib().psv_submit_chunk_cond(ctx, sid, pn, pc))


def psv_run_wave(ctx) -> int:
    n = ctypes.c_int()
    _check(ctx, lib().psv_run_wave(ctx, ctypes.byref(n)))
    return n.value


def psv_poll_chunk(ctx, sid: int, out: np.ndarray | None):
    """Chunk index written to `out`, or None if nothing is ready (EAGAIN)."""
    idx = ctypes.c_int64()
    ptr = None if out is None else _fptr(out)
    r = lib().psv_poll_chunk(ctx, sid, ptr, ctypes.byref(idx))
    if r == PSV_EAGAIN:
        return None
    _check(ctx, r)
    return idx.value


def psv_sync(ctx, timeout_ms: int = -1) -> None:
    _check(ctx, lib().psv_sync(ctx, timeout_ms))


def psv_wave_plan(ctx, cond_tables: bool = False) -> list:
    """Tasks of the next wave as tuples (stream, chunk, step, slot, kv_len,
    row_off, state_slot), plus cond_table last when ``cond_tables``."""
    n = ctypes.c_int()
    _check(ctx, lib().psv_wave_plan(ctx, None, 0, ctypes.byref(n)))
    buf = (Task * max(1, n.value))()
    _check(ctx, lib().psv_wave_plan(ctx, buf, n.value, ctypes.byref(n)))
    if cond_tables:
        return [buf[i].as_tuple() + (buf[i].cond_table,) for i in range(n.value)]
    return [buf[i].as_tuple() for i in range(n.value)]


def psv_predict_wave_ms(ctx, n_streams: int) -> float:
    ms = ctypes.c_double()
    _check(ctx, lib().psv_predict_wave_ms(ctx, n_streams, ctypes.byref(ms)))
    return ms.value


def psv_admit_stream(ctx, cond: np.ndarray | None, slo_ms: float) -> tuple:
    """(stream id, predicted ms per chunk); PSVError with code PSV_EAGAIN when
    the stream is rejected (its .predicted_ms holds the prediction)."""
    sid = ctypes.c_int()
    pred = ctypes.c_double(float("nan"))
    ptr = None if cond is None else _fptr(cond)
    r = lib().psv_admit_stream(ctx, ptr, float(slo_ms), ctypes.byref(sid), ctypes.byref(pred))
    try:
        _check(ctx, r)
    except PSVError as e:
        e.predicted_ms = pred.value
        raise
    return sid.value, pred.value


def psv_close_stream(ctx, sid: int) -> None:
    _check(ctx, lib().psv_close_stream(ctx, sid))


def psv_destroy(ctx) -> None:
    lib().psv_destroy(ctx)


def psv_last_error(ctx) -> str:
    s = lib().psv_last_error(ctx)
    return s.decode() if s else ""


def psv_set_graphs(ctx, enabled: bool) -> None:
    _check(ctx, lib().psv_set_graphs(ctx, int(enabled)))


def psv_set_profiling(ctx, enabled: bool) -> None:
    _check(ctx, lib().psv_set_profiling(ctx, int(enabled)))


def psv_kernel_times(ctx) -> dict:
    n = ctypes.c_int()
    buf = (KernelTime * 16)()
    _check(ctx, lib().psv_kernel_times(ctx, buf, 16, ctypes.byref(n)))
    return {buf[i].name.decode(): dict(launches=buf[i].launches, total_ms=buf[i].total_ms,
                                       flops=buf[i].flops, bytes=buf[i].bytes)
            for i in range(min(n.value, 16))}


def psv_debug_tap(ctx, block: int, h_in_ptr: int, h_out_ptr: int) -> None:
    _check(ctx, lib().psv_debug_tap(ctx, block, ctypes.c_void_p(h_in_ptr), ctypes.c_void_p(h_out_ptr)))


def psv_debug_read_kv(ctx, sid: int, block: int, step: int, rows: int, d: int):
    k = np.empty((rows, d), dtype=np.float32)
    v = np.empty((rows, d), dtype=np.float32)
    _check(ctx, lib().psv_debug_read_kv(ctx, sid, block, step, _fptr(k), _fptr(v)))
    return k, v


def psv_debug_error_word(ctx) -> int:
    """Byte offset of the device error word within the context's arena."""
    off = ctypes.c_size_t()
    _check(ctx, lib().psv_debug_error_word(ctx, ctypes.byref(off)))
    return off.value


def psv_attention_scratch_bytes(prob: AttnProblem) -> int:
    n = ctypes.c_size_t()
    _check(None, lib().psv_attention_scratch_bytes(ctypes.byref(prob), ctypes.byref(n)))
    return n.value


def psv_attention(prob: AttnProblem, q_ptr: int, k_ptr: int, vt_ptr: int, o_ptr: int,
                  scratch_ptr: int, scratch_bytes: int, stream_ptr: int = 0) -> None:
    r = lib().psv_attention(ctypes.byref(prob), ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr),
                            ctypes.c_void_p(vt_ptr), ctypes.c_void_p(o_ptr),
                            ctypes.c_void_p(scratch_ptr), scratch_bytes,
                            ctypes.c_void_p(stream_ptr or None))
    if r < 0:
        raise PSVError(r, "psv_attention rejected its arguments")


def psv_attention_noalloc(prob: AttnProblem, q_ptr: int, k_ptr: int, vt_ptr: int, o_ptr: int,
                          stream_ptr: int = 0) -> None:
    """psv_attention with the library's fixed scratch array (no allocation)."""
    r = lib().psv_attention_noalloc(ctypes.byref(prob), ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr),
                                    ctypes.c_void_p(vt_ptr), ctypes.c_void_p(o_ptr),
                                    ctypes.c_void_p(stream_ptr or None))
    if r == PSV_ENOMEM:
        raise PSVError(r, "psv_attention_noalloc: the problem needs more scratch than the "
                          f"fixed {PSV_ATTN_NOALLOC_SCRATCH_BYTES >> 20} MiB array holds")
    if r < 0:
        raise PSVError(r, "psv_attention_noalloc rejected its arguments (shape or alignment)")


def psv_attention_noalloc_status(stream_ptr: int = 0) -> int:
    """Error word of the last psv_attention_noalloc call on the current device
    (waits for the stream first): 0, or nonzero if a device-side wait timed out."""
    st = ctypes.c_int()
    r = lib().psv_attention_noalloc_status(ctypes.byref(st), ctypes.c_void_p(stream_ptr or None))
    if r < 0:
        raise PSVError(r, "psv_attention_noalloc_status failed")
    return st.value
