"""ctypes binding of liblf_decode.so: argument marshalling only.

Every function here validates torch tensors (dtype, device, shape, layout),
passes their data pointers and the stream to the C ABI declared in
``include/lf_decode.h`` and raises ``LFError`` on a non-OK status. All of the
decode step's arithmetic runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

LF_OK = 0
LF_ERR_INVALID_ARG = 1
LF_ERR_UNSUPPORTED = 2
LF_ERR_CUDA = 3
LF_ERR_NO_MEMORY = 4

LF_DEVERR_BAD_WRITE_SLOT = 0x1
LF_DEVERR_WAIT_TIMEOUT = 0x2

LF_KERNEL_DECODE_STEP = 0
LF_KERNEL_ATTENTION = 1
LF_KERNEL_SCORE = 2
KERNEL_NAMES = {LF_KERNEL_DECODE_STEP: "lf_decode_step_kernel",
                LF_KERNEL_ATTENTION: "lf_decode_step_kernel (attention-only variant)",
                LF_KERNEL_SCORE: "lf_score_kernel"}

LF_STEP_FILL_EMPTY_FIRST = 0x1
LF_STEP_MASK_EVICTED = 0x2
LF_STEP_LOG2_SCORES = 0x4
LF_MAX_TOPK = 1024

# Every exported symbol of include/lf_decode.h.
EXPORTED = (
    "lf_decode_step", "lf_decode_step_scores", "lf_decode_step_ex", "lf_decode_attention",
    "lf_decode_step_host", "lf_decode_step_noalloc", "lf_step_prepare", "lf_step_run",
    "lf_step_errors", "lf_step_destroy", "lf_step_plan", "lf_device_errors",
    "lf_profile_enable", "lf_profile_collect", "lf_release_workspace", "lf_status_string",
    "lf_last_error", "lf_version",
)


class LFError(RuntimeError):
    """A non-OK lf_status from the library."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Load (once) and bind the shared library. Raises if it is missing.

    The environment variable LF_LIBRARY names another build of the same
    library (for comparing two builds in one session)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or os.environ.get("LF_LIBRARY") or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        step_args = [P] * 9 + [I] * 6 + [F, P]
        lib.lf_decode_step.argtypes = step_args
        lib.lf_decode_step_host.argtypes = step_args
        lib.lf_decode_step_noalloc.argtypes = step_args
        lib.lf_decode_step_noalloc.restype = I
        lib.lf_decode_step_scores.argtypes = [P] * 10 + [I] * 6 + [F, P]
        lib.lf_decode_step_ex.argtypes = [P] * 9 + [I, I, P] + [I] * 6 + [F, P]
        lib.lf_decode_step_ex.restype = I
        lib.lf_decode_attention.argtypes = [P] * 8 + [I] * 5 + [F, P]
        lib.lf_decode_attention.restype = I
        for fn in (lib.lf_decode_step, lib.lf_decode_step_host, lib.lf_decode_step_scores):
            fn.restype = I
        lib.lf_step_prepare.argtypes = [P] * 9 + [I] * 6 + [F, P, ctypes.POINTER(P)]
        lib.lf_step_prepare.restype = I
        lib.lf_step_run.argtypes = [P]
        lib.lf_step_run.restype = I
        lib.lf_step_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), I]
        lib.lf_step_errors.restype = I
        lib.lf_step_destroy.argtypes = [P]
        lib.lf_step_destroy.restype = I
        lib.lf_step_plan.argtypes = [I] * 6 + [ctypes.POINTER(ctypes.c_int32)]
        lib.lf_step_plan.restype = I
        lib.lf_device_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), I]
        lib.lf_device_errors.restype = I
        lib.lf_profile_enable.argtypes = [I]
        lib.lf_profile_enable.restype = I
        lib.lf_profile_collect.argtypes = [I, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int64)]
        lib.lf_profile_collect.restype = I
        lib.lf_release_workspace.argtypes = []
        lib.lf_release_workspace.restype = I
        lib.lf_status_string.argtypes = [I]
        lib.lf_status_string.restype = ctypes.c_char_p
        lib.lf_last_error.argtypes = []
        lib.lf_last_error.restype = ctypes.c_char_p
        lib.lf_version.argtypes = []
        lib.lf_version.restype = I
        if path is None:
            _lib = lib
        return lib


def _check(lib, status: int):
    if status != LF_OK:
        msg = lib.lf_last_error().decode(errors="replace")
        name = lib.lf_status_string(status).decode(errors="replace")
        raise LFError(status, f"{name}: {msg}")


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype, shape, cuda: bool):
    # One combined test on the common path; the detailed ones name the fault.
    if (isinstance(t, torch.Tensor) and t.dtype is dtype and t.shape == shape
            and t.is_cuda is cuda and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not cuda and t.is_cuda:
        raise ValueError(f"{name}: must be a host tensor")


def _shapes(q, k_cache):
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B,Hq,d] and k_cache [B,Hkv,S,d]")
    B, Hq, d = q.shape
    _, Hkv, S, _ = k_cache.shape
    return int(B), int(Hq), int(Hkv), int(d), int(S)


def _check_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot,
                io_on_device=True, k=None):
    B, Hq, Hkv, d, S = _shapes(q, k_cache)
    bf, i32 = torch.bfloat16, torch.int32
    _need(q, "q", bf, (B, Hq, d), io_on_device)
    _need(k_cache, "k_cache", bf, (B, Hkv, S, d), True)
    _need(v_cache, "v_cache", bf, (B, Hkv, S, d), True)
    _need(mask, "mask", i32, (B, Hkv, S), True)
    _need(new_k, "new_k", bf, (B, Hkv, d), io_on_device)
    _need(new_v, "new_v", bf, (B, Hkv, d), io_on_device)
    _need(write_slot, "write_slot", i32, (B, Hkv), io_on_device)
    _need(out, "out", bf, (B, Hq, d), io_on_device)
    _need(next_slot, "next_slot", i32, (B, Hkv) if k is None else (B, Hkv, int(k)), io_on_device)
    return B, Hq, Hkv, d, S


def decode_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, W, scale,
                stream=None):
    """lf_decode_step on CUDA tensors (see include/lf_decode.h). Asynchronous."""
    lib = load_library()
    B, Hq, Hkv, d, S = _check_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out,
                                   next_slot)
    _check(lib, lib.lf_decode_step(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(), new_k.data_ptr(),
        new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(), next_slot.data_ptr(),
        B, Hq, Hkv, d, S, int(W), float(scale), _stream_handle(stream)))


def decode_step_scores(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot,
                       scores, W, scale, stream=None):
    """lf_decode_step_scores: also fills scores [B,Hkv,S] fp32 (+inf on masked slots)."""
    lib = load_library()
    B, Hq, Hkv, d, S = _check_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out,
                                   next_slot)
    _need(scores, "scores", torch.float32, (B, Hkv, S), True)
    _check(lib, lib.lf_decode_step_scores(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(), new_k.data_ptr(),
        new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(), next_slot.data_ptr(),
        scores.data_ptr(), B, Hq, Hkv, d, S, int(W), float(scale), _stream_handle(stream)))


def decode_step_ex(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slots, W,
                   scale, k=1, flags=0, scores=None, stream=None):
    """lf_decode_step_ex: next_slots [B,Hkv,k] int32 gets the k lowest-(score, slot)
    candidates per unit; flags are LF_STEP_* bits; scores optional [B,Hkv,S]
    (log2 I_j with LF_STEP_LOG2_SCORES)."""
    lib = load_library()
    B, Hq, Hkv, d, S = _check_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out,
                                   next_slots, k=k)
    if scores is not None:
        _need(scores, "scores", torch.float32, (B, Hkv, S), True)
    _check(lib, lib.lf_decode_step_ex(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(), new_k.data_ptr(),
        new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(), next_slots.data_ptr(), int(k),
        int(flags), None if scores is None else scores.data_ptr(), B, Hq, Hkv, d, S, int(W),
        float(scale), _stream_handle(stream)))


def decode_attention(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, scale,
                     stream=None):
    """lf_decode_attention: slot write and attention only (no score, no eviction)."""
    lib = load_library()
    B, Hq, Hkv, d, S = _shapes(q, k_cache)
    bf, i32 = torch.bfloat16, torch.int32
    _need(q, "q", bf, (B, Hq, d), True)
    _need(k_cache, "k_cache", bf, (B, Hkv, S, d), True)
    _need(v_cache, "v_cache", bf, (B, Hkv, S, d), True)
    _need(mask, "mask", i32, (B, Hkv, S), True)
    _need(new_k, "new_k", bf, (B, Hkv, d), True)
    _need(new_v, "new_v", bf, (B, Hkv, d), True)
    _need(write_slot, "write_slot", i32, (B, Hkv), True)
    _need(out, "out", bf, (B, Hq, d), True)
    _check(lib, lib.lf_decode_attention(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(), new_k.data_ptr(),
        new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(), B, Hq, Hkv, d, S, float(scale),
        _stream_handle(stream)))


def decode_step_host(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, W,
                     scale, stream=None):
    """lf_decode_step_host: per-step I/O in host tensors, caches and mask on the
    device. Pinned tensors are read and written by the kernel in place; others
    are staged through device memory. Outputs are valid after the stream syncs."""
    lib = load_library()
    B, Hq, Hkv, d, S = _check_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out,
                                   next_slot, io_on_device=False)
    _check(lib, lib.lf_decode_step_host(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(), new_k.data_ptr(),
        new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(), next_slot.data_ptr(),
        B, Hq, Hkv, d, S, int(W), float(scale), _stream_handle(stream)))


def decode_step_noalloc(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, W,
                        scale, stream=None):
    """lf_decode_step_noalloc: lf_decode_step with the library's fixed 16 MiB
    scratch instead of cudaMalloc, for callers that cannot allocate device
    memory. Calls that overlap on the GPU share that scratch and race."""
    lib = load_library()
    B, Hq, Hkv, d, S = _check_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out,
                                   next_slot)
    _check(lib, lib.lf_decode_step_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(), new_k.data_ptr(),
        new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(), next_slot.data_ptr(),
        B, Hq, Hkv, d, S, int(W), float(scale), _stream_handle(stream)))


class PreparedStep:
    """lf_step_prepare / lf_step_run: one layer's decode step with its buffers,
    shape, plan and stream fixed once; ``run()`` then enqueues the step with
    no argument checks (see include/lf_decode.h). The per-step buffers (q,
    new_k, new_v, write_slot, out, next_slot) may each be CUDA tensors, pinned
    host tensors (read and written in place) or other host tensors (staged);
    the caches and the mask are CUDA tensors. The object keeps the tensors
    alive; write each token's inputs into the same tensors."""

    def __init__(self, q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, W,
                 scale, stream=None):
        lib = load_library()
        B, Hq, Hkv, d, S = _shapes(q, k_cache)
        bf, i32 = torch.bfloat16, torch.int32
        _need(k_cache, "k_cache", bf, (B, Hkv, S, d), True)
        _need(v_cache, "v_cache", bf, (B, Hkv, S, d), True)
        _need(mask, "mask", i32, (B, Hkv, S), True)
        for t, name, dt, shape in ((q, "q", bf, (B, Hq, d)), (new_k, "new_k", bf, (B, Hkv, d)),
                                   (new_v, "new_v", bf, (B, Hkv, d)),
                                   (write_slot, "write_slot", i32, (B, Hkv)),
                                   (out, "out", bf, (B, Hq, d)),
                                   (next_slot, "next_slot", i32, (B, Hkv))):
            _need(t, name, dt, shape, t.is_cuda if isinstance(t, torch.Tensor) else True)
        if stream is None:
            stream = torch.cuda.current_stream()
        self._keep = (q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, stream)
        self._lib = lib
        self._h = ctypes.c_void_p(0)
        _check(lib, lib.lf_step_prepare(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), mask.data_ptr(),
            new_k.data_ptr(), new_v.data_ptr(), write_slot.data_ptr(), out.data_ptr(),
            next_slot.data_ptr(), B, Hq, Hkv, d, S, int(W), float(scale),
            _stream_handle(stream), ctypes.byref(self._h)))
        self._run = lib.lf_step_run

    def run(self):
        """Enqueue one step on the prepare-time stream (asynchronous)."""
        st = self._run(self._h)
        if st:
            _check(self._lib, st)

    def errors(self, clear: bool = True) -> int:
        """OR of LF_DEVERR_* bits of this handle's runs (syncs its stream)."""
        flags = ctypes.c_uint32(0)
        _check(self._lib, self._lib.lf_step_errors(self._h, ctypes.byref(flags), int(clear)))
        return int(flags.value)

    def close(self):
        """Synchronise the stream and free the handle (idempotent)."""
        if self._h and self._h.value:
            h, self._h = self._h, ctypes.c_void_p(0)
            _check(self._lib, self._lib.lf_step_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def step_plan(B: int, Hq: int, Hkv: int, d: int, S: int, topk: int = 1) -> dict:
    """The launch plan a step of this shape takes on the current device."""
    lib = load_library()
    plan = (ctypes.c_int32 * 6)()
    _check(lib, lib.lf_step_plan(int(B), int(Hq), int(Hkv), int(d), int(S), int(topk), plan))
    return {"nchunk": plan[0], "chunk_tiles": plan[1], "stages": plan[2],
            "cluster": bool(plan[3]), "split": bool(plan[4]), "cluster_fit": plan[5]}


def device_errors(stream=None, clear: bool = True) -> int:
    """OR of LF_DEVERR_* bits raised on `stream` since the last clear (syncs the stream)."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    _check(lib, lib.lf_device_errors(_stream_handle(stream), ctypes.byref(flags), int(clear)))
    return int(flags.value)


def profile_enable(on: bool = True):
    lib = load_library()
    _check(lib, lib.lf_profile_enable(int(on)))


def profile_collect(kernel_id: int):
    """(total event milliseconds, launches) for one kernel id since the last collect."""
    lib = load_library()
    ms = ctypes.c_double(0)
    n = ctypes.c_int64(0)
    _check(lib, lib.lf_profile_collect(int(kernel_id), ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def release_workspace():
    lib = load_library()
    _check(lib, lib.lf_release_workspace())


def status_string(status: int) -> str:
    return load_library().lf_status_string(int(status)).decode()


def version() -> int:
    return int(load_library().lf_version())
