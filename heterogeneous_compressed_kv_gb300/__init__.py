"""GB300-native (sm_103a) two-pool KV cache for DeepSeek-V4-style decoding.

Classical/Block pool: immutable, refcounted, lcm(m, m')-aligned blocks of
compressed CSA / indexer / HCA entries.  State pool: per-request SWA window
ring and compressor state.  The decode-step hot path (append + compress +
seal, indexer top-k, three-source split-K attention) runs in the CUDA kernels
of ``libkvpool.so`` behind the C ABI in ``include/kvpool.h``; ``kvpool`` is
its Python binding.
"""
from .kvpool import (  # noqa: F401
    BF16, CSA, CSA_HCA, F32, FP8_E4M3, HCA, SWA_ONLY, KvpoolError, Pool, PoolConfig, lib, required_bytes,
)
