"""CPU oracle of the two-pool KV cache decode step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  The oracle is a plain single-threaded C model of
the method (``kvoracle.c``) written from the design pages; it is what the CUDA
path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  It
shares no code with the product library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvoracle.c")
HDR = os.path.join(HERE, "kvoracle.h")
LIB = os.path.join(HERE, "libkvoracle.so")

F32, BF16, FP8, FP4 = 0, 1, 2, 3  # FP4: indexer entries only
SWA_ONLY, CSA, HCA, CSA_HCA = 0, 1, 2, 3
OK, ERR_INVALID_ARG, ERR_OUT_OF_BLOCKS, ERR_OUT_OF_REQUESTS, ERR_BAD_REQUEST, ERR_NOT_SHAREABLE = 0, -1, -2, -3, -4, -5
ERR_CAPACITY = -8
ERR_BAD_IMAGE = -9
IMAGE_WINDOW = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no FMA contraction)."""
    with _lock:
        newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
        if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
            tmp = LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                                   "-Wall", "-o", tmp, SRC, "-lm"])
            os.replace(tmp, LIB)
    return LIB


class _Config(C.Structure):
    _fields_ = [("m", C.c_int32), ("m_prime", C.c_int32), ("n_win", C.c_int32),
                ("heads", C.c_int32), ("head_dim", C.c_int32), ("idx_heads", C.c_int32), ("idx_dim", C.c_int32),
                ("in_dtype", C.c_int32), ("cache_dtype", C.c_int32), ("n_layers", C.c_int32),
                ("layer_kinds", C.POINTER(C.c_int32)),
                ("max_requests", C.c_int32), ("max_blocks", C.c_int32), ("max_blocks_per_request", C.c_int32),
                ("gate_csa", C.POINTER(C.c_float)), ("gate_hca", C.POINTER(C.c_float)),
                ("gate_idx", C.POINTER(C.c_float)), ("idx_fp4", C.c_int32), ("csa_hot_slots", C.c_int32),
                ("csa_host_slots", C.c_int32), ("idx_per_token", C.c_int32)]


class _Info(C.Structure):
    _fields_ = [("length", C.c_int64), ("n_csa", C.c_int64), ("n_hca", C.c_int64),
                ("csa_tail", C.c_int32), ("hca_tail", C.c_int32), ("n_blocks", C.c_int32), ("window", C.c_int32)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        vp, i32, i64, f32p = C.c_void_p, C.c_int32, C.c_int64, C.POINTER(C.c_float)
        L.kvo_bf16_from_f32.restype = C.c_uint16
        L.kvo_bf16_from_f32.argtypes = [C.c_float]
        L.kvo_f32_from_bf16.restype = C.c_float
        L.kvo_f32_from_bf16.argtypes = [C.c_uint16]
        L.kvo_e4m3_from_f32.restype = C.c_uint8
        L.kvo_e4m3_from_f32.argtypes = [C.c_float]
        L.kvo_f32_from_e4m3.restype = C.c_float
        L.kvo_f32_from_e4m3.argtypes = [C.c_uint8]
        L.kvo_e2m1_from_f32.restype = C.c_uint8
        L.kvo_e2m1_from_f32.argtypes = [C.c_float]
        L.kvo_f32_from_e2m1.restype = C.c_float
        L.kvo_f32_from_e2m1.argtypes = [C.c_uint8]
        L.kvo_softmax_f32.argtypes = [vp, C.c_int, vp]
        L.kvo_encode.argtypes = [C.c_int, vp, C.c_int, vp, vp]
        L.kvo_decode.restype = C.c_double
        L.kvo_decode.argtypes = [C.c_int, vp, vp, C.c_int]
        L.kvo_compress_kv.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp]
        L.kvo_compress_idx.argtypes = [vp, C.c_int, vp, vp, vp]
        L.kvo_score.restype = C.c_float
        L.kvo_score.argtypes = [vp, vp, vp, vp]
        L.kvo_score_tokens.restype = C.c_float
        L.kvo_score_tokens.argtypes = [vp, C.c_int, vp, vp, vp]
        L.kvo_topk.argtypes = [vp, i64, C.c_int, vp]
        L.kvo_attend_sources.argtypes = [vp, i64, vp, vp, vp, vp]
        L.kvo_create.argtypes = [C.POINTER(_Config), C.POINTER(vp)]
        L.kvo_destroy.argtypes = [vp]
        L.kvo_destroy.restype = None
        L.kvo_alloc_request.argtypes = [vp, C.POINTER(i32)]
        L.kvo_free_request.argtypes = [vp, i32]
        L.kvo_append.argtypes = [vp, C.c_int, vp, vp, vp, vp, vp]
        L.kvo_share_prefix.argtypes = [vp, i32, i32, i64, vp, vp]
        L.kvo_decode_attend.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp, C.c_int, vp, vp]
        L.kvo_request_info.argtypes = [vp, i32, C.POINTER(_Info), vp, i32]
        L.kvo_block_refcount.argtypes = [vp, i32]
        L.kvo_free_block_count.argtypes = [vp]
        L.kvo_block_entry.argtypes = [vp, C.c_int, i32, C.c_int, C.c_int, vp, vp]
        L.kvo_request_entry.argtypes = [vp, C.c_int, i32, C.c_int, i64, vp, vp]
        L.kvo_window_token.argtypes = [vp, C.c_int, i32, i64, vp, vp]
        L.kvo_request_scores.argtypes = [vp, C.c_int, i32, vp, vp]
        L.kvo_value_bytes.argtypes = [C.c_int]
        L.kvo_fnv1a64.restype = C.c_uint64
        L.kvo_fnv1a64.argtypes = [vp, i64]
        L.kvo_fingerprint.restype = C.c_uint64
        L.kvo_fingerprint.argtypes = [vp]
        L.kvo_image_bytes.restype = i64
        L.kvo_image_bytes.argtypes = [vp, i64, C.c_uint32]
        L.kvo_export_prefix.argtypes = [vp, i32, i64, C.c_uint32, vp, i64]
        L.kvo_import_prefix.argtypes = [vp, i32, vp, i64, vp, vp]
        L.kvo_block_location.argtypes = [vp, i32, C.POINTER(i32), C.POINTER(C.c_uint32)]
        L.kvo_epoch.restype = C.c_uint32
        L.kvo_epoch.argtypes = [vp]
        L.kvo_inactive_blocks.argtypes = [vp, C.c_uint32, vp, i32]
        L.kvo_offload.argtypes = [vp, C.c_int, vp]
        L.kvo_fetch.argtypes = [vp, C.c_int, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def value_bytes(dtype: int) -> int:
    return 4 if dtype == F32 else 2 if dtype == BF16 else 1


def code_bytes(dtype: int, n: int) -> int:
    """Bytes of n encoded values (FP4: two per byte)."""
    return (n + 1) // 2 if dtype == FP4 else n * value_bytes(dtype)


# ---- scalar codecs -----------------------------------------------------
def bf16_from_f32(x: float) -> int:
    return lib().kvo_bf16_from_f32(float(x))


def f32_from_bf16(b: int) -> float:
    return lib().kvo_f32_from_bf16(int(b))


def e4m3_from_f32(x: float) -> int:
    return lib().kvo_e4m3_from_f32(float(x))


def f32_from_e4m3(c: int) -> float:
    return lib().kvo_f32_from_e4m3(int(c))


def e2m1_from_f32(x: float) -> int:
    return lib().kvo_e2m1_from_f32(float(x))


def f32_from_e2m1(c: int) -> float:
    return lib().kvo_f32_from_e2m1(int(c))


def softmax_f32(logits) -> np.ndarray:
    g = _f32(logits)
    out = np.zeros_like(g)
    lib().kvo_softmax_f32(_p(g), g.size, _p(out))
    return out


def encode(dtype: int, x):
    """-> (codes uint8 array, scale uint16)"""
    x = _f32(x)
    code = np.zeros(code_bytes(dtype, x.size), np.uint8)
    scale = np.zeros(1, np.uint16)
    lib().kvo_encode(dtype, _p(x), x.size, _p(code), _p(scale))
    return code, int(scale[0])


def decode(dtype: int, code, scale: int, n: int) -> np.ndarray:
    code = np.ascontiguousarray(code, dtype=np.uint8)
    sc = np.array([scale], np.uint16)
    return np.array([lib().kvo_decode(dtype, _p(code), _p(sc), i) for i in range(n)])


def fnv1a64(data: bytes) -> int:
    b = np.frombuffer(bytes(data), np.uint8).copy()
    return int(lib().kvo_fnv1a64(_p(b) if b.size else None, b.size))


def topk(scores, top_k: int) -> np.ndarray:
    s = _f32(scores)
    out = np.zeros(max(top_k, 1), np.int32)
    rc = lib().kvo_topk(_p(s), s.size, top_k, _p(out))
    assert rc == OK
    return out[:top_k]


class Oracle:
    """The stateful two-pool cache.  Arrays are numpy; K/V/indexer inputs are
    the fp32 values of the input-dtype tensors."""

    def __init__(self, *, m, m_prime, n_win, heads, head_dim, idx_heads, idx_dim, in_dtype, cache_dtype,
                 layer_kinds, max_requests, max_blocks, max_blocks_per_request, gate_csa, gate_hca, gate_idx,
                 idx_fp4=0, csa_hot_slots=0, csa_host_slots=0, idx_per_token=0):
        self.L = lib()
        self.kinds = np.ascontiguousarray(layer_kinds, dtype=np.int32)
        n_layers = self.kinds.size
        self.g_csa = _f32(gate_csa).reshape(-1)
        self.g_hca = _f32(gate_hca).reshape(-1)
        self.g_idx = _f32(gate_idx).reshape(-1)
        fp = C.POINTER(C.c_float)
        cfg = _Config(m, m_prime, n_win, heads, head_dim, idx_heads, idx_dim, in_dtype, cache_dtype, n_layers,
                      self.kinds.ctypes.data_as(C.POINTER(C.c_int32)), max_requests, max_blocks,
                      max_blocks_per_request, self.g_csa.ctypes.data_as(fp), self.g_hca.ctypes.data_as(fp),
                      self.g_idx.ctypes.data_as(fp), int(idx_fp4), int(csa_hot_slots), int(csa_host_slots),
                      int(idx_per_token))
        h = C.c_void_p()
        rc = self.L.kvo_create(C.byref(cfg), C.byref(h))
        if rc != OK:
            raise ValueError(f"kvo_create failed: {rc}")
        self.h = h
        self.m, self.m_prime, self.n_win = m, m_prime, n_win
        self.heads, self.head_dim, self.idx_heads, self.idx_dim = heads, head_dim, idx_heads, idx_dim
        self.HD, self.XD = heads * head_dim, idx_heads * idx_dim
        self.cache_dtype, self.in_dtype, self.n_layers = cache_dtype, in_dtype, n_layers
        self.vs = value_bytes(cache_dtype)
        self.esz = 2 * self.HD * self.vs
        self.idx_dtype = FP4 if idx_fp4 else cache_dtype
        self.xsz = code_bytes(self.idx_dtype, self.XD)
        self.CB = m_prime // m

    def __del__(self):
        if getattr(self, "h", None):
            self.L.kvo_destroy(self.h)
            self.h = None

    # lifecycle ---------------------------------------------------------
    def alloc_request(self):
        r = C.c_int32()
        rc = self.L.kvo_alloc_request(self.h, C.byref(r))
        return (rc, r.value)

    def free_request(self, r):
        return self.L.kvo_free_request(self.h, r)

    def append(self, req_ids, n_new, k, v, idx_k):
        req = np.ascontiguousarray(req_ids, dtype=np.int32)
        nn = np.ascontiguousarray(n_new, dtype=np.int32)
        k, v = _f32(k), _f32(v)
        idx = None if idx_k is None else _f32(idx_k)
        return self.L.kvo_append(self.h, req.size, _p(req), _p(nn), _p(k), _p(v), _p(idx))

    def share_prefix(self, dst, src, n_tokens, win_k, win_v):
        wk = None if win_k is None else _f32(win_k)
        wv = None if win_v is None else _f32(win_v)
        return self.L.kvo_share_prefix(self.h, dst, src, n_tokens, _p(wk), _p(wv))

    # prefix images -------------------------------------------------------
    def fingerprint(self) -> int:
        return int(self.L.kvo_fingerprint(self.h))

    def image_bytes(self, n_tokens, flags=0) -> int:
        return int(self.L.kvo_image_bytes(self.h, n_tokens, flags))

    def export_prefix(self, r, n_tokens, flags=0, cap=None):
        """(rc, image as uint8 array)"""
        n = self.image_bytes(n_tokens, flags)
        cap = max(n, 0) if cap is None else cap
        img = np.zeros(max(cap, 1), np.uint8)
        rc = self.L.kvo_export_prefix(self.h, r, n_tokens, flags, _p(img), cap)
        return rc, img[:max(n, 0)]

    def import_prefix(self, dst, image, win_k=None, win_v=None):
        img = np.ascontiguousarray(image, np.uint8)
        wk = None if win_k is None else _f32(win_k)
        wv = None if win_v is None else _f32(win_v)
        return self.L.kvo_import_prefix(self.h, dst, _p(img), img.size, _p(wk), _p(wv))

    # HiSparse placement ------------------------------------------------------
    def block_location(self, b):
        """(rc, loc, last_used): loc >= 0 hot slot, < 0 host slot -1-loc."""
        loc, lu = C.c_int32(), C.c_uint32()
        rc = self.L.kvo_block_location(self.h, b, C.byref(loc), C.byref(lu))
        return rc, loc.value, lu.value

    def epoch(self) -> int:
        return int(self.L.kvo_epoch(self.h))

    def inactive_blocks(self, idle, cap=1 << 16):
        ids = np.zeros(max(cap, 1), np.int32)
        n = self.L.kvo_inactive_blocks(self.h, idle, _p(ids), cap)
        return ids[:min(n, cap)].copy() if n >= 0 else n

    def offload(self, ids):
        a = np.ascontiguousarray(ids, np.int32)
        return self.L.kvo_offload(self.h, a.size, _p(a))

    def fetch(self, ids):
        a = np.ascontiguousarray(ids, np.int32)
        return self.L.kvo_fetch(self.h, a.size, _p(a))

    def decode_attend(self, layer, req_ids, q, q_idx, top_k):
        req = np.ascontiguousarray(req_ids, dtype=np.int32)
        n = req.size
        q = _f32(q)
        qi = None if q_idx is None else _f32(q_idx)
        out = np.zeros((n, self.HD), np.float64)
        tk = np.zeros((n, max(top_k, 1)), np.int32)
        rc = self.L.kvo_decode_attend(self.h, layer, n, _p(req), _p(q), _p(qi), top_k, _p(out), _p(tk))
        return rc, out.reshape(n, self.heads, self.head_dim), tk[:, :top_k]

    # pure steps -----------------------------------------------------------
    def compress_kv(self, layer, kind, tokens):
        t = _f32(tokens)
        code = np.zeros(self.esz, np.uint8)
        sc = np.zeros(2, np.uint16)
        rc = self.L.kvo_compress_kv(self.h, layer, kind, _p(t), _p(code), _p(sc))
        assert rc == OK
        return code, sc

    def compress_idx(self, layer, keys):
        t = _f32(keys)
        code = np.zeros(self.xsz, np.uint8)
        sc = np.zeros(1, np.uint16)
        rc = self.L.kvo_compress_idx(self.h, layer, _p(t), _p(code), _p(sc))
        assert rc == OK
        return code, sc

    def score(self, code, scale, q_idx):
        code = np.ascontiguousarray(code, np.uint8)
        sc = np.ascontiguousarray(np.atleast_1d(scale), np.uint16)
        return self.L.kvo_score(self.h, _p(code), _p(sc), _p(_f32(q_idx)))

    def score_tokens(self, layer, codes, scales, q_idx):
        """Score of one CSA entry from its m tokens' encoded keys (per-token
        indexer keys): codes [m][xsz] uint8, scales [m] uint16."""
        codes = np.ascontiguousarray(codes, np.uint8)
        sc = np.ascontiguousarray(np.atleast_1d(scales), np.uint16)
        return self.L.kvo_score_tokens(self.h, layer, _p(codes), _p(sc), _p(_f32(q_idx)))

    def attend_sources(self, codes, scales, q):
        codes = np.ascontiguousarray(codes, np.uint8)
        scales = np.ascontiguousarray(scales, np.uint16)
        n_src = codes.size // self.esz
        out = np.zeros(self.HD, np.float64)
        rc = self.L.kvo_attend_sources(self.h, n_src, _p(codes), _p(scales), _p(_f32(q)), _p(out))
        return rc, out.reshape(self.heads, self.head_dim)

    # inspection --------------------------------------------------------
    def request_info(self, r, cap=1 << 20):
        info = _Info()
        ids = np.zeros(max(cap, 1), np.int32)
        rc = self.L.kvo_request_info(self.h, r, C.byref(info), _p(ids), cap)
        if rc != OK:
            return rc, None, None
        d = {f: getattr(info, f) for f, _ in _Info._fields_}
        return rc, d, ids[:info.n_blocks].copy()

    def block_refcount(self, b):
        return self.L.kvo_block_refcount(self.h, b)

    def free_block_count(self):
        return self.L.kvo_free_block_count(self.h)

    def block_entry(self, layer, block_id, kind, slot):
        n = self.xsz if kind == 3 else self.esz
        code = np.zeros(n, np.uint8)
        sc = np.zeros(2, np.uint16)
        rc = self.L.kvo_block_entry(self.h, layer, block_id, kind, slot, _p(code), _p(sc))
        return rc, code, sc

    def request_entry(self, layer, r, kind, e):
        n = self.xsz if kind == 3 else self.esz
        code = np.zeros(n, np.uint8)
        sc = np.zeros(2, np.uint16)
        rc = self.L.kvo_request_entry(self.h, layer, r, kind, e, _p(code), _p(sc))
        return rc, code, sc

    def window_token(self, layer, r, pos):
        code = np.zeros(self.esz, np.uint8)
        sc = np.zeros(2, np.uint16)
        rc = self.L.kvo_window_token(self.h, layer, r, pos, _p(code), _p(sc))
        return rc, code, sc

    def request_scores(self, layer, r, q_idx, n_csa):
        out = np.zeros(max(n_csa, 1), np.float32)
        rc = self.L.kvo_request_scores(self.h, layer, r, _p(_f32(q_idx)), _p(out))
        return rc, out[:n_csa]

    # decoding helpers (the oracle's own codecs) ------------------------
    def entry_values(self, code, scale) -> np.ndarray:
        """fp64 values [2][H][d] of an encoded K/V entry."""
        L, HD = self.L, self.HD
        code = np.ascontiguousarray(code, np.uint8)
        sc = np.ascontiguousarray(scale, np.uint16)
        out = np.empty(2 * HD)
        for half in range(2):
            sub = np.ascontiguousarray(code[half * HD * self.vs:(half + 1) * HD * self.vs])
            s = np.ascontiguousarray(sc[half:half + 1])
            for i in range(HD):
                out[half * HD + i] = L.kvo_decode(self.cache_dtype, _p(sub), _p(s), i)
        return out.reshape(2, self.heads, self.head_dim)
