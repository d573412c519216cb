"""psv: GB300-native serving of autoregressive-denoising DiT world models.

The product is the C-ABI library ``libpsv.so`` (include/psv.h) built from
``csrc/`` for sm_103a.  This package holds the build step and a thin ctypes
binding with the same call names; ``Session`` adds the PyTorch plumbing
(device arena and CUDA stream) around those calls.  There is no CPU path:
every call that computes runs in libpsv's kernels.
"""
from __future__ import annotations

from . import _psv
from ._psv import *  # noqa: F401,F403


class Session:
    """One libpsv context on the current CUDA device.

    The arena is a torch uint8 CUDA tensor (kept alive by the session); the
    context issues its work on ``stream`` (default: torch's current stream).
    """

    def __init__(self, cfg: dict, max_streams: int | None = None, max_inflight: int = 0,
                 flags: int = 0, stream=None):
        import torch

        self.cfg = cfg
        self.desc = _psv.model_desc(cfg, max_streams, max_inflight, flags)
        nbytes = _psv.psv_arena_bytes(self.desc)
        self.torch_stream = stream if stream is not None else torch.cuda.current_stream()
        self._arena = torch.empty(nbytes + 1024, dtype=torch.uint8, device="cuda")
        base = self._arena.data_ptr()
        self.arena_ptr = (base + 1023) // 1024 * 1024
        self.arena_bytes = nbytes
        self.ctx = _psv.psv_create(self.desc, self.arena_ptr, nbytes, self.torch_stream.cuda_stream)

    # host-numpy weights, one tensor at a time: iterable of (block, name, array)
    def load_host_weights(self, items) -> None:
        for block, name, arr in items:
            _psv.psv_load_weights(self.ctx, [(block, name, arr, _psv.PSV_LOC_HOST)])

    # device torch tensors (bf16 matrices / f32 biases): iterable of (block, name, tensor)
    def load_device_weights(self, items) -> None:
        import torch

        batch = []
        keep = []
        for block, name, t in items:
            t = t.contiguous()
            keep.append(t)
            dt = _psv.PSV_DTYPE_BF16 if t.dtype == torch.bfloat16 else _psv.PSV_DTYPE_F32
            batch.append((block, name, (t.data_ptr(), t.numel(), dt), _psv.PSV_LOC_DEVICE))
        _psv.psv_load_weights(self.ctx, batch)

    def open_stream(self, cond):
        return _psv.psv_open_stream(self.ctx, cond)

    def admit_stream(self, cond, slo_ms: float = 0.0):
        """Open a stream under admission control: (stream id, predicted ms per
        chunk), or PSVError (code PSV_EAGAIN) if it is rejected."""
        return _psv.psv_admit_stream(self.ctx, cond, slo_ms)

    def close_stream(self, sid):
        _psv.psv_close_stream(self.ctx, sid)

    def predict_wave_ms(self, n_streams: int) -> float:
        return _psv.psv_predict_wave_ms(self.ctx, n_streams)

    def submit(self, sid, noise, cond=None):
        """Submit the stream's next chunk; ``cond`` [d] gives the chunk its own
        conditioning vector (needs ``flags`` with PSV_FLAG_CHUNK_COND)."""
        if cond is None:
            _psv.psv_submit_chunk(self.ctx, sid, noise)
        else:
            _psv.psv_submit_chunk_cond(self.ctx, sid, noise, cond)

    def run_wave(self) -> int:
        return _psv.psv_run_wave(self.ctx)

    def poll(self, sid, out):
        return _psv.psv_poll_chunk(self.ctx, sid, out)

    def sync(self, timeout_ms: int = -1):
        _psv.psv_sync(self.ctx, timeout_ms)

    def plan(self):
        return _psv.psv_wave_plan(self.ctx)

    def close(self):
        if getattr(self, "ctx", None) is not None:
            _psv.psv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
