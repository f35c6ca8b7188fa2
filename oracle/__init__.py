"""fp64 CPU oracle for multi-head scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The product package never
imports this module, and this module imports nothing from the product package.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one row at a time,
the three stages scores -> softmax weights -> weighted sum of V that the
realizar ``cached/attention.rs`` page and the ripvec-core ``Driver`` page
describe).  This file only builds that C file with gcc and marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_CAUSAL_WINDOW = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, -O2, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """ctypes handle on a compiled oracle library at ``path`` (argument types set)."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_attention_rows
    f.restype = ctypes.c_int
    f.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
        ctypes.c_double, ctypes.c_void_p, ctypes.c_longlong,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _as_f32(x) -> np.ndarray:
    """Exact float32 copy of a torch tensor (bf16/fp16/fp32) or numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only needed for torch inputs
        if x.dtype != torch.float32:
            x = x.to(torch.float32)  # bf16 -> fp32 is exact
        x = x.numpy()
    a = np.asarray(x)
    if a.dtype != np.float32:
        if a.dtype not in (np.float16,):
            raise TypeError(f"oracle inputs must be exactly representable in fp32, got {a.dtype}")
        a = a.astype(np.float32)
    return np.ascontiguousarray(a)


def attention(q, k, v, *, pos_offset: int = 0, mask_mode: int = MASK_NONE, window: int = 0,
              key_lens=None, scale: float | None = None, rows=None,
              return_weights: bool = False, nthreads: int = 0, lib=None):
    """fp64 attention output for q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D].

    rows: None for the whole output ([B,Hq,Lq,D] float64 array), or a sequence of
    flat row indices (b*Hq + h)*Lq + i, returning [len(rows), D].
    scale: None means 1/sqrt(D) rounded to fp32 (the value the library receives).
    return_weights: also return the stage-2 softmax weights, [nrows, Lk].
    lib: a handle from load_library() to use instead of the default build.
    """
    qa, ka, va = _as_f32(q), _as_f32(k), _as_f32(v)
    if qa.ndim != 4 or ka.ndim != 4 or va.ndim != 4:
        raise ValueError("q, k, v must be 4-D [B, H, L, D]")
    B, Hq, Lq, D = qa.shape
    Bk, Hkv, Lk, Dk = ka.shape
    if va.shape != ka.shape or Bk != B or Dk != D:
        raise ValueError("shape mismatch between q, k, v")
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(D)))
    kl = None
    if key_lens is not None:
        if hasattr(key_lens, "detach"):
            key_lens = key_lens.detach().cpu().numpy()
        kl = np.ascontiguousarray(np.asarray(key_lens, dtype=np.int32))
        if kl.shape != (B,):
            raise ValueError("key_lens must have shape [B]")
    if rows is None:
        rr = None
        nrows = B * Hq * Lq
    else:
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = int(rr.shape[0])
    out = np.zeros((nrows, D), dtype=np.float64)
    w = np.zeros((nrows, Lk), dtype=np.float64) if return_weights else None
    lib = lib if lib is not None else _load()
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = lib.oracle_attention_rows(
        ptr(qa), ptr(ka), ptr(va), B, Hq, Hkv, Lq, Lk, D,
        int(pos_offset), int(mask_mode), int(window), ptr(kl),
        float(scale), ptr(rr), nrows, ptr(out), ptr(w), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    if rows is None:
        out = out.reshape(B, Hq, Lq, D)
        if w is not None:
            w = w.reshape(B, Hq, Lq, Lk)
    return (out, w) if return_weights else out
