"""Seeded synthetic inputs for the two-pool KV cache (ctypes binding of
``libkvgen.so``; the definition is in ``kvgen.h``).

The generator is counter based: element ``i`` of stream ``s`` under ``seed``
is a pure function of ``(seed, s, i)``, so the GPU can fill a 64 GiB prefill
in place while the CPU regenerates any sampled element bit for bit.  This
module holds none of the KV-cache method's arithmetic.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))

K, V, IDXK, Q, QIDX, GATE_CSA, GATE_HCA, GATE_IDX, LEN = 1, 2, 3, 4, 5, 6, 7, 8, 9
OUT_F32, OUT_BF16, OUT_BF16_F32 = 0, 1, 2  # the last one host only


class Run(C.Structure):
    _fields_ = [("stream", C.c_uint64), ("index0", C.c_int64), ("count", C.c_int64), ("out_offset", C.c_int64)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        from .._build import build_lib
        L = C.CDLL(build_lib("kvgen"))
        L.kvgen_fill_host.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_int, C.c_void_p]
        L.kvgen_fill_device.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_int, C.c_void_p, C.c_void_p]
        L.kvgen_u64_host.argtypes = [C.c_void_p, C.c_uint64, C.c_uint64, C.c_int64, C.c_int64]
        _lib = L
    return _lib


def stream_id(kind: int, layer: int, request: int) -> int:
    return (kind << 56) | ((layer & 0xFFFF) << 40) | (request & 0xFFFFFFFFFF)


def _runs_array(runs):
    arr = (Run * max(len(runs), 1))()
    for i, (s, i0, cnt, off) in enumerate(runs):
        arr[i] = Run(s, i0, cnt, off)
    return arr


def fill_host(n_values: int, out_dtype: int, seed: int, runs, out: np.ndarray | None = None) -> np.ndarray:
    """runs: list of (stream, index0, count, out_offset).  Returns float32 values
    (OUT_F32), uint16 bfloat16 bits (OUT_BF16) or float32 bfloat16 values
    (OUT_BF16_F32); `out` (contiguous, n_values elements of that type) is
    filled in place when given."""
    dt = np.uint16 if out_dtype == OUT_BF16 else np.float32
    if out is None:
        out = np.zeros(n_values, dt)
    elif out.dtype != dt or out.size != n_values or not out.flags.c_contiguous:
        raise ValueError("fill_host: out must be a contiguous array of n_values elements of the output type")
    arr = _runs_array(runs)
    rc = lib().kvgen_fill_host(out.ctypes.data_as(C.c_void_p), out_dtype, seed, len(runs), arr)
    if rc != 0:
        raise ValueError(f"kvgen_fill_host: {rc}")
    return out


def fill_device(ptr: int, out_dtype: int, seed: int, runs, stream: int = 0) -> None:
    arr = _runs_array(runs)
    rc = lib().kvgen_fill_device(C.c_void_p(ptr), out_dtype, seed, len(runs), arr, C.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"kvgen_fill_device: {rc}")


def u64(seed: int, stream: int, index0: int, count: int) -> np.ndarray:
    out = np.zeros(max(count, 1), np.uint64)
    rc = lib().kvgen_u64_host(out.ctypes.data_as(C.c_void_p), seed, stream, index0, count)
    if rc != 0:
        raise ValueError(f"kvgen_u64_host: {rc}")
    return out[:count]


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def token_runs(kind: int, layer: int, reqs, pos0s, counts, row_len: int, base_offset: int = 0):
    """Runs that lay out, row after row, the tokens [pos0, pos0+count) of each
    workload request in turn (batch order, then position order)."""
    runs, off = [], base_offset
    for r, p0, c in zip(reqs, pos0s, counts):
        if c > 0:
            runs.append((stream_id(kind, layer, int(r)), int(p0) * row_len, int(c) * row_len, off))
        off += int(c) * row_len
    return runs


def gate_logits(seed: int, kind: int, n_layers: int, groups: int, width: int) -> np.ndarray:
    """fp32 gate logits [n_layers][groups][width] ~ Irwin-Hall N(0,1) stand-in."""
    runs = [(stream_id(kind, l, 0), 0, groups * width, l * groups * width) for l in range(n_layers)]
    return fill_host(n_layers * groups * width, OUT_F32, seed, runs).reshape(n_layers, groups, width)
