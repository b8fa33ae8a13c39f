"""CPU fp64 oracle for dense video-token attention, AdaLN modulate and the
gated residual.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import this package; the product package
never does.  It shares no code with the CUDA path; the two meet only in the
seeded inputs of ``workloads.py``.

The arithmetic lives in ``oracle.c`` (plain C, double precision, the
definitions written out; see its header for the passages each function
follows).  This module only marshals numpy/torch arrays into it.

Pins: every function here is checked in ``tests/test_oracle.py`` against
closed forms, invariants, brute force on tiny inputs and library routines
(torch's float64 scaled_dot_product_attention and layer_norm on the CPU).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build
from . import delta  # noqa: F401  (fp64 Video Delta Attention, numpy)
from . import vsa  # noqa: F401  (VSA-style block-sparse attention, numpy)


def default_threads() -> int:
    return os.cpu_count() or 1


def _bf16_bits(t) -> np.ndarray:
    """bfloat16 torch tensor (or uint16 ndarray of bf16 bits) -> contiguous uint16 ndarray."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """The oracle's functions bound to one build of ``oracle.c`` (the tests
    also bind deliberately broken copies, to show that the pins catch them)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_double, i64p, ctypes.c_int64, f64p, f64p,
                                         ctypes.c_int]
        lib.oracle_attn_rows.restype = ctypes.c_int
        lib.oracle_modulate.argtypes = [u16p, ctypes.c_int64, f32p, f32p, ctypes.c_double, i64p,
                                        ctypes.c_int64, f64p, ctypes.c_int]
        lib.oracle_modulate.restype = ctypes.c_int
        lib.oracle_gated_residual.argtypes = [u16p, u16p, ctypes.c_int64, f32p, i64p, ctypes.c_int64,
                                              f64p, u16p, ctypes.c_int]
        lib.oracle_gated_residual.restype = ctypes.c_int
        lib.oracle_attn_rows_window.argtypes = [u16p, u16p, u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int64, i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int]
        lib.oracle_attn_rows_window.restype = ctypes.c_int
        lib.oracle_window_allowed.argtypes = [ctypes.c_int64] * 6
        lib.oracle_window_allowed.restype = ctypes.c_int
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_double
        self.lib = lib

    def attn_rows(self, q, k, v, head: int, rows, scale: float, head_dim: int = 128, threads: int | None = None):
        """fp64 attention output and LSE of ``head`` for query ``rows``.

        q, k, v: bfloat16 [N, H*head_dim] (or bf16 bit arrays); returns
        (O: float64 [len(rows), head_dim], lse: float64 [len(rows)]).
        """
        qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
        n, ld = qb.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.empty((len(rows), head_dim), dtype=np.float64)
        lse = np.empty(len(rows), dtype=np.float64)
        rc = self.lib.oracle_attn_rows(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                       _ptr(vb, ctypes.c_uint16), n, ld, head_dim, head, float(scale),
                                       _ptr(rows, ctypes.c_int64), len(rows), _ptr(o, ctypes.c_double),
                                       _ptr(lse, ctypes.c_double), threads or default_threads())
        if rc != 0:
            raise ValueError("oracle_attn_rows: bad arguments")
        return o, lse

    def attn_rows_window(self, q, k, v, head: int, rows, scale: float, frame_tokens: int, chunk_frames: int = 5,
                         window_chunks: int = 1, head_dim: int = 128, threads: int | None = None):
        """fp64 windowed attention (local chunk window + first/last frame anchors)
        of ``head`` for query ``rows``; returns (O [len(rows), head_dim], lse)."""
        qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
        n, ld = qb.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.empty((len(rows), head_dim), dtype=np.float64)
        lse = np.empty(len(rows), dtype=np.float64)
        rc = self.lib.oracle_attn_rows_window(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                              _ptr(vb, ctypes.c_uint16), n, ld, head_dim, head, float(scale),
                                              frame_tokens, chunk_frames, window_chunks, _ptr(rows, ctypes.c_int64),
                                              len(rows), _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                              threads or default_threads())
        if rc != 0:
            raise ValueError("oracle_attn_rows_window: bad arguments")
        return o, lse

    def window_allowed(self, i: int, j: int, n: int, frame_tokens: int, chunk_frames: int = 5,
                       window_chunks: int = 1) -> bool:
        return bool(self.lib.oracle_window_allowed(i, j, n, frame_tokens, chunk_frames, window_chunks))

    def modulate(self, x, shift_row, scale_row, eps: float, rows=None, threads: int | None = None):
        """fp64 LN(x)*(1+scale_row)+shift_row for ``rows`` of x (bf16 [N, C])."""
        xb = _bf16_bits(x)
        n, c = xb.shape
        rows = (np.arange(n, dtype=np.int64) if rows is None
                else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
        sh = np.ascontiguousarray(np.asarray(shift_row, dtype=np.float32))
        sc = np.ascontiguousarray(np.asarray(scale_row, dtype=np.float32))
        assert sh.shape == (c,) and sc.shape == (c,)
        y = np.empty((len(rows), c), dtype=np.float64)
        rc = self.lib.oracle_modulate(_ptr(xb, ctypes.c_uint16), c, _ptr(sh, ctypes.c_float),
                                      _ptr(sc, ctypes.c_float), float(eps), _ptr(rows, ctypes.c_int64),
                                      len(rows), _ptr(y, ctypes.c_double), threads or default_threads())
        if rc != 0:
            raise ValueError("oracle_modulate: bad arguments")
        return y

    def gated_residual(self, x, a, gate_row, rows=None, threads: int | None = None):
        """(fp64 x + gate_row*a, the same rounded to bf16 as uint16 bits) for ``rows``."""
        xb, ab = _bf16_bits(x), _bf16_bits(a)
        n, c = xb.shape
        assert ab.shape == xb.shape
        rows = (np.arange(n, dtype=np.int64) if rows is None
                else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
        g = np.ascontiguousarray(np.asarray(gate_row, dtype=np.float32))
        assert g.shape == (c,)
        y = np.empty((len(rows), c), dtype=np.float64)
        yb = np.empty((len(rows), c), dtype=np.uint16)
        rc = self.lib.oracle_gated_residual(_ptr(xb, ctypes.c_uint16), _ptr(ab, ctypes.c_uint16), c,
                                            _ptr(g, ctypes.c_float), _ptr(rows, ctypes.c_int64), len(rows),
                                            _ptr(y, ctypes.c_double), _ptr(yb, ctypes.c_uint16),
                                            threads or default_threads())
        if rc != 0:
            raise ValueError("oracle_gated_residual: bad arguments")
        return y, yb

    def round_bf16(self, x: float) -> float:
        """Nearest bfloat16 value of a double, ties to even (the oracle's rounding)."""
        return self.lib.oracle_round_bf16(float(x))


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def attn_rows(*args, **kwargs):
    return default().attn_rows(*args, **kwargs)


def modulate(*args, **kwargs):
    return default().modulate(*args, **kwargs)


def attn_rows_window(*args, **kwargs):
    return default().attn_rows_window(*args, **kwargs)


def window_allowed(*args, **kwargs):
    return default().window_allowed(*args, **kwargs)


def gated_residual(*args, **kwargs):
    return default().gated_residual(*args, **kwargs)


def round_bf16(x: float) -> float:
    return default().round_bf16(x)
