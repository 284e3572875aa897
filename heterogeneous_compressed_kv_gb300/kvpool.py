"""Thin Python binding of the kvpool C ABI (``include/kvpool.h``).

Argument marshalling only: torch tensors are passed as raw device pointers,
the current (or given) torch CUDA stream as a ``cudaStream_t``.  Every step of
the path runs in the CUDA kernels of ``libkvpool.so``; there is no CPU or
PyTorch fallback -- if the library cannot be built or loaded this module
raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

F32, BF16, FP8_E4M3, FP4_E2M1 = 0, 1, 2, 3  # FP4: indexer entries only (PoolConfig.idx_fp4)
SWA_ONLY, CSA, HCA, CSA_HCA = 0, 1, 2, 3
FLAG_NO_DEVICE = 1
OK, ERR_INVALID_ARG, ERR_OUT_OF_BLOCKS, ERR_OUT_OF_REQUESTS, ERR_BAD_REQUEST = 0, -1, -2, -3, -4
ERR_NOT_SHAREABLE, ERR_CUDA, ERR_DEVICE_CHECK, ERR_CAPACITY, ERR_BAD_IMAGE = -5, -6, -7, -8, -9
KERNEL_APPEND, KERNEL_SCORE, KERNEL_SELECT, KERNEL_ATTEND, KERNEL_COMBINE, KERNEL_IMAGE = range(6)
KERNEL_NAMES = ["append", "score", "select", "attend", "combine", "image"]
IMAGE_WINDOW = 1  # prefix image flag: include the SWA window (a checkpoint)
PROFILE_COUNT = 1 << 16  # profiling flag: count launches and bytes without events

EXPORTS = ["kvpool_required_bytes", "kvpool_create", "kvpool_destroy", "kvpool_alloc_request",
           "kvpool_free_request", "kvpool_share_prefix", "kvpool_append", "kvpool_decode_attend",
           "kvpool_request_info", "kvpool_block_refcount", "kvpool_free_block_count", "kvpool_get_layout",
           "kvpool_check_device", "kvpool_profile_enable", "kvpool_profile_read", "kvpool_last_error",
           "kvpool_topk_static", "kvpool_profile_timeline", "kvpool_fingerprint", "kvpool_image_bytes",
           "kvpool_export_prefix", "kvpool_import_prefix", "kvpool_host_slot_bytes", "kvpool_set_host_pool",
           "kvpool_offload", "kvpool_fetch", "kvpool_block_location", "kvpool_epoch", "kvpool_block_activity",
           "kvpool_inactive_blocks", "kvpool_wait_selftest", "kvpool_topk_static_check"]


class KvpoolError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kvpool error {code}: {msg}")
        self.code = code


class _Config(C.Structure):
    _fields_ = [("m", C.c_int32), ("m_prime", C.c_int32), ("n_win", C.c_int32), ("heads", C.c_int32),
                ("head_dim", C.c_int32), ("idx_heads", C.c_int32), ("idx_dim", C.c_int32),
                ("in_dtype", C.c_int32), ("cache_dtype", C.c_int32), ("n_layers", C.c_int32),
                ("layer_kinds", C.POINTER(C.c_int32)), ("max_requests", C.c_int32), ("max_blocks", C.c_int32),
                ("max_blocks_per_request", C.c_int32), ("max_batch", C.c_int32), ("max_top_k", C.c_int32),
                ("gate_csa", C.POINTER(C.c_float)), ("gate_hca", C.POINTER(C.c_float)),
                ("gate_idx", C.POINTER(C.c_float)), ("flags", C.c_uint32), ("idx_fp4", C.c_int32),
                ("csa_hot_slots", C.c_int32), ("csa_host_slots", C.c_int32), ("idx_per_token", C.c_int32)]


class _Info(C.Structure):
    _fields_ = [("length", C.c_int64), ("n_csa", C.c_int64), ("n_hca", C.c_int64), ("csa_tail", C.c_int32),
                ("hca_tail", C.c_int32), ("n_blocks", C.c_int32), ("window", C.c_int32)]


class _Layout(C.Structure):
    _fields_ = [("entry_bytes", C.c_int64), ("idx_entry_bytes", C.c_int64), ("csa_per_block", C.c_int32),
                ("staging_base", C.c_int32), ("table_offset", C.c_int64), ("error_offset", C.c_int64),
                ("total_bytes", C.c_int64), ("csa_staging_base", C.c_int32), ("csa_hot_slots", C.c_int32),
                ("host_slot_bytes", C.c_int64), ("csa_loc_offset", C.c_int64), ("activity_offset", C.c_int64)]


class _LayerLayout(C.Structure):
    _fields_ = [("kind", C.c_int32), ("pad", C.c_int32), ("csa_offset", C.c_int64), ("csa_block_bytes", C.c_int64),
                ("idx_offset", C.c_int64), ("idx_block_bytes", C.c_int64), ("idx_scale_offset", C.c_int64),
                ("hca_offset", C.c_int64), ("hca_block_bytes", C.c_int64), ("ring_offset", C.c_int64),
                ("ring_request_bytes", C.c_int64), ("acc_offset", C.c_int64), ("acc_request_bytes", C.c_int64),
                ("csa_host_offset", C.c_int64)]


_lib = None


def lib():
    """Load libkvpool.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        from ._build import build_lib
        path = build_lib("kvpool")
        L = C.CDLL(path)
        vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        L.kvpool_required_bytes.restype = C.c_size_t
        L.kvpool_required_bytes.argtypes = [C.POINTER(_Config)]
        L.kvpool_create.argtypes = [C.POINTER(_Config), vp, C.c_size_t, vp, C.POINTER(vp)]
        L.kvpool_destroy.argtypes = [vp]
        L.kvpool_alloc_request.argtypes = [vp, C.POINTER(i32)]
        L.kvpool_free_request.argtypes = [vp, i32]
        L.kvpool_share_prefix.argtypes = [vp, i32, i32, i64, vp, vp, vp]
        L.kvpool_append.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
        L.kvpool_decode_attend.argtypes = [vp, i32, i32, vp, vp, vp, i32, vp, vp, vp]
        L.kvpool_request_info.argtypes = [vp, i32, C.POINTER(_Info), vp, i32]
        L.kvpool_block_refcount.argtypes = [vp, i32]
        L.kvpool_free_block_count.argtypes = [vp]
        L.kvpool_get_layout.argtypes = [vp, C.POINTER(_Layout), i32, C.POINTER(_LayerLayout)]
        L.kvpool_check_device.argtypes = [vp, vp, C.POINTER(C.c_uint32)]
        L.kvpool_profile_enable.argtypes = [vp, C.c_int]
        L.kvpool_profile_read.argtypes = [vp, i32, C.POINTER(C.c_double), C.POINTER(i64), C.POINTER(i64)]
        L.kvpool_topk_static.argtypes = [vp, i32, i32, i32, vp, vp]
        L.kvpool_topk_static_check.argtypes = [vp, C.POINTER(C.c_uint32)]
        L.kvpool_profile_timeline.argtypes = [vp, i32, vp]
        L.kvpool_fingerprint.restype = C.c_uint64
        L.kvpool_fingerprint.argtypes = [vp]
        L.kvpool_image_bytes.restype = i64
        L.kvpool_image_bytes.argtypes = [vp, i64, C.c_uint32]
        L.kvpool_export_prefix.argtypes = [vp, i32, i64, C.c_uint32, vp, i64, vp]
        L.kvpool_import_prefix.argtypes = [vp, i32, vp, i64, vp, vp, vp]
        L.kvpool_host_slot_bytes.restype = i64
        L.kvpool_host_slot_bytes.argtypes = [vp]
        L.kvpool_set_host_pool.argtypes = [vp, vp, i64]
        L.kvpool_offload.argtypes = [vp, i32, vp, vp]
        L.kvpool_fetch.argtypes = [vp, i32, vp, vp]
        L.kvpool_block_location.argtypes = [vp, i32, C.POINTER(i32)]
        L.kvpool_epoch.restype = C.c_uint32
        L.kvpool_epoch.argtypes = [vp]
        L.kvpool_block_activity.argtypes = [vp, i32, vp, vp, vp]
        L.kvpool_inactive_blocks.restype = i32
        L.kvpool_inactive_blocks.argtypes = [vp, C.c_uint32, vp, i32, vp]
        L.kvpool_wait_selftest.argtypes = [vp, vp]
        L.kvpool_last_error.restype = C.c_char_p
        L.kvpool_last_error.argtypes = [vp]
        _lib = L
    return _lib


def library_path() -> str:
    return lib()._name


@dataclass
class PoolConfig:
    m: int
    m_prime: int
    n_win: int
    heads: int
    head_dim: int
    idx_heads: int
    idx_dim: int
    in_dtype: int
    cache_dtype: int
    layer_kinds: Sequence[int]
    max_requests: int
    max_blocks: int
    max_blocks_per_request: int
    max_batch: int
    max_top_k: int
    gate_csa: np.ndarray  # [n_layers][heads][m] logits
    gate_hca: np.ndarray  # [n_layers][heads][m_prime]
    gate_idx: np.ndarray  # [n_layers][idx_heads][m]
    flags: int = 0
    idx_fp4: int = 0  # 1: indexer entries in FP4 (e2m1 + one bf16 scale)
    csa_hot_slots: int = 0  # HiSparse: GPU slots for sealed blocks' CSA entries (0 = off)
    csa_host_slots: int = 0  # HiSparse: host slots for offloaded CSA entries
    idx_per_token: int = 0  # 1: one indexer key per token (128 per block) instead of one per CSA entry
    _keep: list = field(default_factory=list, repr=False)

    def to_c(self) -> _Config:
        kinds = np.ascontiguousarray(self.layer_kinds, dtype=np.int32)
        g = [np.ascontiguousarray(x, dtype=np.float32).reshape(-1) for x in (self.gate_csa, self.gate_hca,
                                                                             self.gate_idx)]
        self._keep = [kinds] + g
        fp = C.POINTER(C.c_float)
        return _Config(self.m, self.m_prime, self.n_win, self.heads, self.head_dim, self.idx_heads, self.idx_dim,
                       self.in_dtype, self.cache_dtype, kinds.size, kinds.ctypes.data_as(C.POINTER(C.c_int32)),
                       self.max_requests, self.max_blocks, self.max_blocks_per_request, self.max_batch,
                       self.max_top_k, g[0].ctypes.data_as(fp), g[1].ctypes.data_as(fp), g[2].ctypes.data_as(fp),
                       self.flags, self.idx_fp4, self.csa_hot_slots, self.csa_host_slots, self.idx_per_token)


def required_bytes(cfg: PoolConfig) -> int:
    c = cfg.to_c()
    return int(lib().kvpool_required_bytes(C.byref(c)))


def topk_static(scores, top_k: int, out, stream=None) -> int:
    """Top-k of each row of a [n_rows][n_cols] fp32 device tensor into
    ``out`` ([n_rows][top_k] int32) using only the library's static device
    scratch (no allocation); see kvpool_topk_static in include/kvpool.h.
    Raises ValueError for tensors the kernels cannot take as they are."""
    import torch
    if scores.dim() != 2 or scores.dtype != torch.float32 or not scores.is_cuda or not scores.is_contiguous():
        raise ValueError("topk_static: scores must be a contiguous 2-D float32 CUDA tensor")
    n_rows, n_cols = scores.shape
    if (out.dtype != torch.int32 or not out.is_cuda or not out.is_contiguous() or out.device != scores.device
            or tuple(out.shape) != (n_rows, top_k)):
        raise ValueError("topk_static: out must be a contiguous int32 [n_rows][top_k] tensor on the scores' device")
    return lib().kvpool_topk_static(scores.data_ptr(), n_rows, n_cols, top_k, out.data_ptr(), _stream(stream))


def topk_static_check(stream=None) -> tuple:
    """(return code, device error flags) of the last topk_static call on the
    current device; synchronizes the stream."""
    w = C.c_uint32(0)
    rc = lib().kvpool_topk_static_check(_stream(stream), C.byref(w))
    return int(rc), int(w.value)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host_buffer(x):
    """(address, bytes) of a host buffer: a numpy array or a CPU torch tensor."""
    if isinstance(x, np.ndarray):
        return x.ctypes.data, x.nbytes
    return x.data_ptr(), x.numel() * x.element_size()


def _i32(a) -> np.ndarray:
    if type(a) is np.ndarray and a.dtype == np.int32 and a.flags.c_contiguous:
        return a
    return np.ascontiguousarray(a, dtype=np.int32)


class Pool:
    """A two-pool KV cache living in a caller-owned device arena."""

    def __init__(self, cfg: PoolConfig, arena=None, stream=None):
        self.L = lib()
        self.cfg = cfg
        self._c = cfg.to_c()
        self.arena = arena
        h = C.c_void_p()
        if cfg.flags & FLAG_NO_DEVICE:
            rc = self.L.kvpool_create(C.byref(self._c), None, 0, None, C.byref(h))
        else:
            nbytes = arena.numel() * arena.element_size()
            rc = self.L.kvpool_create(C.byref(self._c), arena.data_ptr(), nbytes, _stream(stream), C.byref(h))
        if rc != OK:
            raise KvpoolError(rc, "kvpool_create refused the configuration")
        self.h = h
        self.n_layers = len(cfg.layer_kinds)
        self.HD = cfg.heads * cfg.head_dim
        self.XD = cfg.idx_heads * cfg.idx_dim

    def __del__(self):
        if getattr(self, "h", None):
            self.L.kvpool_destroy(self.h)
            self.h = None

    def last_error(self) -> str:
        return self.L.kvpool_last_error(self.h).decode()

    def _check(self, rc: int, what: str) -> int:
        if rc != OK:
            raise KvpoolError(rc, f"{what}: {self.last_error()}")
        return rc

    # ---- lifecycle ----
    def alloc_request(self) -> int:
        r = C.c_int32()
        self._check(self.L.kvpool_alloc_request(self.h, C.byref(r)), "alloc_request")
        return r.value

    def free_request(self, req: int) -> None:
        self._check(self.L.kvpool_free_request(self.h, req), "free_request")

    def share_prefix(self, dst, src, n_tokens, win_k, win_v, stream=None, check=True) -> int:
        rc = self.L.kvpool_share_prefix(self.h, dst, src, n_tokens, _ptr(win_k), _ptr(win_v), _stream(stream))
        return self._check(rc, "share_prefix") if check else rc

    # ---- prefix images (sealed blocks in page-locked host memory) ----
    def fingerprint(self) -> int:
        return int(self.L.kvpool_fingerprint(self.h))

    def image_bytes(self, n_tokens: int, flags: int = 0) -> int:
        return int(self.L.kvpool_image_bytes(self.h, n_tokens, flags))

    def export_prefix(self, req, n_tokens, flags=0, out=None, stream=None, check=True):
        """Write the image of req's first n_tokens tokens into `out` (a
        page-locked uint8 host tensor; allocated when None) and return it.  The
        copy runs in stream order: the image is complete once the stream has
        reached it."""
        if out is None:
            import torch
            out = torch.empty(max(self.image_bytes(n_tokens, flags), 64), dtype=torch.uint8, pin_memory=True)
        addr, nbytes = _host_buffer(out)
        rc = self.L.kvpool_export_prefix(self.h, req, n_tokens, flags, addr, nbytes, _stream(stream))
        if check:
            self._check(rc, "export_prefix")
            return out
        return rc

    def import_prefix(self, dst, image, win_k=None, win_v=None, stream=None, check=True) -> int:
        """Restore an image (page-locked host memory) into the fresh request
        dst; win_k / win_v: the recomputed window for an image without one."""
        addr, nbytes = _host_buffer(image)
        rc = self.L.kvpool_import_prefix(self.h, dst, addr, nbytes, _ptr(win_k), _ptr(win_v), _stream(stream))
        return self._check(rc, "import_prefix") if check else rc

    # ---- HiSparse: inactive CSA entries off the GPU ----
    def host_slot_bytes(self) -> int:
        return int(self.L.kvpool_host_slot_bytes(self.h))

    def set_host_pool(self, pool=None, check=True):
        """Give the pool its host slots (a page-locked uint8 host tensor; one is
        allocated when None) and return it; the caller keeps it alive."""
        if pool is None:
            import torch
            pool = torch.empty(max(self.cfg.csa_host_slots * self.host_slot_bytes(), 16), dtype=torch.uint8,
                               pin_memory=True)
        addr, nbytes = _host_buffer(pool)
        rc = self.L.kvpool_set_host_pool(self.h, addr, nbytes)
        if check:
            self._check(rc, "set_host_pool")
            self._host_pool = pool
            return pool
        return rc

    def offload(self, block_ids, stream=None, check=True) -> int:
        ids = _i32(block_ids)
        rc = self.L.kvpool_offload(self.h, ids.size, ids.ctypes.data, _stream(stream))
        return self._check(rc, "offload") if check else rc

    def fetch(self, block_ids, stream=None, check=True) -> int:
        ids = _i32(block_ids)
        rc = self.L.kvpool_fetch(self.h, ids.size, ids.ctypes.data, _stream(stream))
        return self._check(rc, "fetch") if check else rc

    def block_location(self, block_id: int):
        """(rc, loc): loc >= 0 a GPU slot, < 0 host slot -1 - loc."""
        loc = C.c_int32()
        rc = self.L.kvpool_block_location(self.h, block_id, C.byref(loc))
        return rc, loc.value

    def epoch(self) -> int:
        return int(self.L.kvpool_epoch(self.h))

    def block_activity(self, block_ids, stream=None) -> np.ndarray:
        ids = _i32(block_ids)
        out = np.zeros(max(ids.size, 1), np.uint32)
        rc = self.L.kvpool_block_activity(self.h, ids.size, ids.ctypes.data,
                                          out.ctypes.data, _stream(stream))
        self._check(rc, "block_activity")
        return out[:ids.size]

    def inactive_blocks(self, idle: int, cap: int = 1 << 20, stream=None) -> np.ndarray:
        ids = np.zeros(max(cap, 1), np.int32)
        n = self.L.kvpool_inactive_blocks(self.h, idle, ids.ctypes.data, cap, _stream(stream))
        if n < 0:
            self._check(n, "inactive_blocks")
        return ids[:min(n, cap)].copy()

    def append(self, req_ids, n_new, k, v, idx_k, stream=None, check=True) -> int:
        req, nn = _i32(req_ids), _i32(n_new)
        rc = self.L.kvpool_append(self.h, req.size, req.ctypes.data, nn.ctypes.data,
                                  _ptr(k), _ptr(v), _ptr(idx_k), _stream(stream))
        return self._check(rc, "append") if check else rc

    def decode_attend(self, layer, req_ids, q, q_idx, top_k, out, topk_out=None, stream=None, check=True) -> int:
        req = _i32(req_ids)
        rc = self.L.kvpool_decode_attend(self.h, layer, req.size, req.ctypes.data, _ptr(q),
                                         _ptr(q_idx), top_k, _ptr(out), _ptr(topk_out), _stream(stream))
        return self._check(rc, "decode_attend") if check else rc

    # ---- queries ----
    def request_info(self, req: int, cap: int = 1 << 16):
        info = _Info()
        ids = np.zeros(max(cap, 1), np.int32)
        rc = self.L.kvpool_request_info(self.h, req, C.byref(info), ids.ctypes.data, cap)
        if rc != OK:
            return rc, None, None
        d = {f: getattr(info, f) for f, _ in _Info._fields_}
        return rc, d, ids[:info.n_blocks].copy()

    def block_refcount(self, b: int) -> int:
        return self.L.kvpool_block_refcount(self.h, b)

    def free_block_count(self) -> int:
        return self.L.kvpool_free_block_count(self.h)

    def layout(self, layer: Optional[int] = None):
        lo = _Layout()
        ll = _LayerLayout()
        rc = self.L.kvpool_get_layout(self.h, C.byref(lo), -1 if layer is None else layer,
                                      None if layer is None else C.byref(ll))
        self._check(rc, "get_layout")
        d = {f: getattr(lo, f) for f, _ in _Layout._fields_}
        if layer is not None:
            d.update({f: getattr(ll, f) for f, _ in _LayerLayout._fields_})
        return d

    def wait_selftest(self, stream=None) -> None:
        """A kernel whose barrier wait runs out (see kvpool_wait_selftest)."""
        self._check(self.L.kvpool_wait_selftest(self.h, _stream(stream)), "wait_selftest")

    def check_device(self, stream=None) -> int:
        w = C.c_uint32()
        rc = self.L.kvpool_check_device(self.h, _stream(stream), C.byref(w))
        if rc != OK:
            raise KvpoolError(rc, f"check_device: {self.last_error()} (flags {w.value:#x})")
        return w.value

    def profile_enable(self, on: bool = True, kinds=None, count: bool = False) -> None:
        """Record the launches of the given kernel kinds (indexes into
        KERNEL_NAMES; all kinds when None), or stop recording.  count: every
        launch of every kind also adds its kernel count and algorithmic bytes
        to the totals, with no events (kinds=[] counts without timing)."""
        mask = 0
        if on:
            mask = (1 << len(KERNEL_NAMES)) - 1 if kinds is None else sum(1 << int(k) for k in set(kinds))
            if count:
                mask |= PROFILE_COUNT
        self._check(self.L.kvpool_profile_enable(self.h, mask), "profile_enable")

    def profile_timeline(self, cap: int = 4096):
        """[(kernel name, start ms, end ms)] of the recorded launches."""
        buf = np.zeros((cap, 3), np.float32)
        n = self.L.kvpool_profile_timeline(self.h, cap, buf.ctypes.data)
        if n < 0:
            raise KvpoolError(n, "profile_timeline")
        return [(KERNEL_NAMES[int(k)], float(a), float(b)) for k, a, b in buf[:n]]

    def profile_read(self, kernel: int):
        ms, n, b = C.c_double(), C.c_int64(), C.c_int64()
        self._check(self.L.kvpool_profile_read(self.h, kernel, C.byref(ms), C.byref(n), C.byref(b)), "profile_read")
        return ms.value, n.value, b.value
