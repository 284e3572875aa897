"""The five synthetic workloads of the decode-step hot path and their input
recipes.  Pure data plus seeded draws; none of the method's arithmetic.

Every tensor is drawn from the counter generator in ``kvgen.h``: K, V,
indexer keys and queries ~ N(0,1) stand-in rounded to the input dtype, gate
logits ~ N(0,1) stand-in in fp32.  Lengths are drawn from the LEN stream.
"""
from __future__ import annotations

import numpy as np

from . import LEN, stream_id, u64, fill_host, OUT_F32

F32, BF16, FP8 = 0, 1, 2
SWA_ONLY, CSA, HCA, CSA_HCA = 0, 1, 2, 3

COMMON = dict(m=4, m_prime=128)

TINY = dict(COMMON, name="tiny", n_layers=1, layer_kinds=[CSA_HCA], heads=4, head_dim=64, idx_heads=1, idx_dim=32,
            in_dtype=F32, cache_dtype=F32, n_win=128, top_k=16, seed=0, n_requests=1, prefix=130,
            decode_steps=8)

DECODE_BATCH = dict(COMMON, name="decode_batch", n_layers=1, layer_kinds=[CSA_HCA], heads=16, head_dim=128,
                    idx_heads=4, idx_dim=64, in_dtype=BF16, cache_dtype=BF16, n_win=128, top_k=512, seed=1,
                    n_requests=32, len_lo=1, len_hi=8192, decode_steps=100)

CHUNKED_PREFILL = dict(COMMON, name="chunked_prefill", n_layers=1, layer_kinds=[CSA_HCA], heads=16, head_dim=128,
                       idx_heads=4, idx_dim=64, in_dtype=BF16, cache_dtype=BF16, n_win=128, top_k=512, seed=2,
                       n_requests=4, tokens=32768, chunk=2048, shared=16384)

LONG_CONTEXT = dict(COMMON, name="long_context", n_layers=1, layer_kinds=[CSA_HCA], heads=16, head_dim=128,
                    idx_heads=4, idx_dim=64, in_dtype=BF16, cache_dtype=FP8, n_win=128, top_k=2048, seed=3,
                    n_requests=8, length=1 << 20, chunk=2048)

MIXED_SERVING = dict(COMMON, name="mixed_serving", n_layers=4, layer_kinds=[SWA_ONLY, CSA, HCA, CSA], heads=16,
                     head_dim=128, idx_heads=4, idx_dim=64, in_dtype=BF16, cache_dtype=BF16, n_win=4096,
                     top_k=1024, seed=4, n_requests=256, len_median=4096, len_sigma=1.0, len_cap=131072,
                     churn=0.10, decode_steps=200, chunk=2048)

ALL = [TINY, DECODE_BATCH, CHUNKED_PREFILL, LONG_CONTEXT, MIXED_SERVING]


def uniform_lengths(seed: int, n: int, lo: int, hi: int, index0: int = 0) -> np.ndarray:
    """L_i = lo + (u64 draw i mod (hi - lo + 1))."""
    u = u64(seed, stream_id(LEN, 0, 0), index0, n)
    return (lo + (u % np.uint64(hi - lo + 1))).astype(np.int64)


def lognormal_lengths(seed: int, n: int, median: int, sigma: float, cap: int, index0: int = 0) -> np.ndarray:
    """L_i = clip(round(median * exp(sigma * z_i)), 1, cap), z_i the N(0,1)
    stand-in of the LEN stream (sigma is not given by the workload text; 1.0)."""
    z = fill_host(n, OUT_F32, seed, [(stream_id(LEN, 1, 0), index0, n, 0)]).astype(np.float64)
    lens = np.rint(median * np.exp(sigma * z))
    return np.clip(lens, 1, cap).astype(np.int64)


def churn_picks(seed: int, step: int, n_active: int, count: int) -> np.ndarray:
    """`count` distinct positions in [0, n_active) to retire at `step`
    (partial Fisher-Yates driven by the LEN stream of layer 2)."""
    u = u64(seed, stream_id(LEN, 2, step), 0, count)
    order = list(range(n_active))
    for j in range(count):
        r = j + int(u[j] % np.uint64(n_active - j))
        order[j], order[r] = order[r], order[j]
    return np.array(order[:count], np.int64)


def churn_count(cfg) -> int:
    """Requests that finish (and arrive) per step: round-half-even of churn * B."""
    return int(round(cfg["churn"] * cfg["n_requests"]))


def mixed_schedule(cfg, steps: int):
    """The mixed-serving schedule on the host: the initial lengths, and per
    decode step the slots that finish, the arrivals (slot, workload id,
    length) and the peak number of sealed blocks.  Lengths are lognormal
    (median 4096, capped); arrivals take the lowest free slots; step 0 has no
    churn; every active request grows by one token per step."""
    B, n_ch, mp_ = cfg["n_requests"], churn_count(cfg), cfg["m_prime"]
    lens = [int(x) for x in lognormal_lengths(cfg["seed"], B, cfg["len_median"], cfg["len_sigma"], cfg["len_cap"])]
    cur = {s: L for s, L in enumerate(lens)}
    free, wid, plan, peak = [], B, [], 0
    for step in range(steps):
        gone, arrivals = [], []
        if step > 0:
            order = sorted(cur)
            gone = [order[j] for j in churn_picks(cfg["seed"], step, len(order), n_ch)]
            for s in gone:
                del cur[s]
            free = sorted(free + gone)
            for L in lognormal_lengths(cfg["seed"], n_ch, cfg["len_median"], cfg["len_sigma"], cfg["len_cap"],
                                       index0=B + (step - 1) * n_ch):
                s = free.pop(0)
                arrivals.append((s, wid, int(L)))
                cur[s] = int(L)
                wid += 1
        for s in cur:
            cur[s] += 1
        plan.append((gone, arrivals))
        peak = max(peak, sum(L // mp_ for L in cur.values()))
    return lens, plan, peak


def blocks_needed(lengths, m_prime: int) -> int:
    return int(sum(int(L) // m_prime for L in lengths))


def describe(cfg) -> str:
    keys = [k for k in ("n_requests", "length", "tokens", "len_hi", "len_median") if k in cfg]
    return cfg["name"] + "(" + ", ".join(f"{k}={cfg[k]}" for k in keys) + ")"
