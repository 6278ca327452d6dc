"""fp64 CPU oracle of the LongFlow decode step (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library and its Python binding
never do, and the two implementations share no code.

The arithmetic lives in ``lf_oracle.c`` (plain C, fp64, one OpenMP thread per
(b, kvh) unit). This module compiles it with gcc on first use, on whichever
machine runs it, and marshals numpy arrays to it with ctypes.

Parity status of each piece, against "LongFlow: Efficient KV Cache Compression
for Reasoning Models":

* slot write, mask ageing, softmax, output, score and argmin are pinned by the
  ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``. Those tests use brute
  force, closed forms, library routines and invariants, and never re-run this
  code's own formula.
* LongFlowScore against the paper's own definition is **parity unpinned**. The
  paper prints no formula, so the score definition
  ``I_j = sum_h sum_c |p_hj * v_jc|`` is the contract, not something checked
  against the paper.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lf_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liblf_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile lf_oracle.c into oracle/_build/liblf_oracle.so (portable flags)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(_LIB_PATH))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError as e:  # pragma: no cover - toolchain failure
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.lfo_decode_step.argtypes = [P] * 11 + [i] * 6 + [ctypes.c_float, i, P, i]
    lib.lfo_decode_step.restype = i
    lib.lfo_decode_step_ex.argtypes = [P] * 11 + [i] * 6 + [ctypes.c_float] + [i] * 5 + [P, i]
    lib.lfo_decode_step_ex.restype = i
    lib.lfo_max_threads.argtypes = []
    lib.lfo_max_threads.restype = i
    return lib


def bind_library(path: str):
    """Bind another build of lf_oracle.c (the planted-mistake tests use this)."""
    return _bind(path)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle uses by default on this machine."""
    return int(_load().lfo_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _need(a, dtype, shape, name):
    if a.dtype != dtype or tuple(a.shape) != tuple(shape) or not a.flags.c_contiguous:
        raise ValueError(f"{name}: want {np.dtype(dtype).name}{tuple(shape)} C-contiguous, "
                         f"got {a.dtype}{tuple(a.shape)}")


def decode_step(q, k_cache, v_cache, mask, new_k, new_v, write_slot, W, scale, *,
                want_p=False, want_scores=False, nthreads=0, units=None, lib=None,
                topk=1, fill_first=False, mask_evicted=False, attention_only=False):
    """Run one decode step in fp64.

    bf16 arrays are numpy ``uint16`` bit patterns. ``k_cache``, ``v_cache`` and
    ``mask`` are updated in place, like the library's. ``units`` (optional)
    restricts the work to those (b * Hkv + kvh) units; the outputs of other units
    are then left as NaN / -2.

    Returns a dict: ``out`` float64 [B,Hq,d], ``next_slot`` int32 [B,Hkv],
    ``invalid_writes`` int, and ``p`` [B,Hq,S] / ``scores`` [B,Hkv,S] on request
    (scores are +inf on masked slots). ``lib`` selects another build bound with
    ``bind_library``.

    Options: ``topk`` > 1 returns ``next_slot`` as [B,Hkv,topk], the topk
    candidates in ascending (class, score, slot) order, -1 past the last;
    ``fill_first`` makes empty slots candidates ranked before every score;
    ``mask_evicted`` sets the mask of returned slots to -1; ``attention_only``
    writes and attends only (the written slot becomes live, nothing ages, no
    selection; ``next_slot`` is None).
    """
    B, Hq, d = q.shape
    _, Hkv, S, _ = k_cache.shape
    _need(q, np.uint16, (B, Hq, d), "q")
    _need(k_cache, np.uint16, (B, Hkv, S, d), "k_cache")
    _need(v_cache, np.uint16, (B, Hkv, S, d), "v_cache")
    _need(mask, np.int32, (B, Hkv, S), "mask")
    _need(new_k, np.uint16, (B, Hkv, d), "new_k")
    _need(new_v, np.uint16, (B, Hkv, d), "new_v")
    _need(write_slot, np.int32, (B, Hkv), "write_slot")
    out = np.full((B, Hq, d), np.nan, dtype=np.float64)
    nxt = np.full((B, Hkv, int(topk)), -2, dtype=np.int32)
    p = np.zeros((B, Hq, S), dtype=np.float64) if want_p else None
    sc = np.full((B, Hkv, S), np.nan, dtype=np.float64) if want_scores else None
    u = None
    if units is not None:
        u = np.ascontiguousarray(np.asarray(units, dtype=np.int32))
    rc = (lib or _load()).lfo_decode_step_ex(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask), _ptr(new_k), _ptr(new_v),
        _ptr(write_slot), _ptr(out), _ptr(nxt), _ptr(p), _ptr(sc), B, Hq, Hkv, d, S, int(W),
        float(scale), int(topk), int(bool(fill_first)), int(bool(mask_evicted)),
        int(bool(attention_only)), int(nthreads), _ptr(u), 0 if u is None else int(u.size))
    if rc == -1:
        raise ValueError("oracle: invalid arguments")
    if rc == -2:
        raise MemoryError("oracle: out of memory")
    if attention_only:
        nxt = None
    elif topk == 1:
        nxt = np.ascontiguousarray(nxt[:, :, 0])
    res = {"out": out, "next_slot": nxt, "invalid_writes": int(rc)}
    if want_p:
        res["p"] = p
    if want_scores:
        res["scores"] = sc
    return res
