"""Shared test helpers: seeded inputs (through the generator module) and
oracle construction for the workloads."""
from __future__ import annotations

import numpy as np

from heterogeneous_compressed_kv_gb300 import gen
from heterogeneous_compressed_kv_gb300.gen import workloads as W

import oracle as O


def gates(cfg):
    nl = cfg["n_layers"]
    g_csa = gen.gate_logits(cfg["seed"], gen.GATE_CSA, nl, cfg["heads"], cfg["m"])
    g_hca = gen.gate_logits(cfg["seed"], gen.GATE_HCA, nl, cfg["heads"], cfg["m_prime"])
    g_idx = gen.gate_logits(cfg["seed"], gen.GATE_IDX, nl, cfg["idx_heads"], cfg["m"])
    return g_csa, g_hca, g_idx


def make_oracle(cfg, max_requests, max_blocks, max_blocks_per_request, gate_override=None):
    g_csa, g_hca, g_idx = gate_override if gate_override is not None else gates(cfg)
    return O.Oracle(m=cfg["m"], m_prime=cfg["m_prime"], n_win=cfg["n_win"], heads=cfg["heads"],
                    head_dim=cfg["head_dim"], idx_heads=cfg["idx_heads"], idx_dim=cfg["idx_dim"],
                    in_dtype=cfg["in_dtype"], cache_dtype=cfg["cache_dtype"], layer_kinds=cfg["layer_kinds"],
                    max_requests=max_requests, max_blocks=max_blocks,
                    max_blocks_per_request=max_blocks_per_request, gate_csa=g_csa, gate_hca=g_hca,
                    gate_idx=g_idx, idx_fp4=cfg.get("idx_fp4", 0), csa_hot_slots=cfg.get("csa_hot_slots", 0),
                    csa_host_slots=cfg.get("csa_host_slots", 0), idx_per_token=cfg.get("idx_per_token", 0))


def _values(cfg, n_values, runs, out=None):
    return gen.fill_host(n_values, gen.OUT_F32 if cfg["in_dtype"] == W.F32 else gen.OUT_BF16_F32, cfg["seed"], runs,
                         out)


def tokens(cfg, reqs, pos0s, counts):
    """K, V [n_layers][T][H*d] and indexer keys [n_layers][T][Ih*Id] (fp32
    values of the input dtype) for workload requests `reqs`, positions
    [pos0, pos0+count)."""
    HD = cfg["heads"] * cfg["head_dim"]
    XD = cfg["idx_heads"] * cfg["idx_dim"]
    T = int(sum(counts))
    nl = cfg["n_layers"]
    k = np.empty((nl, T, HD), np.float32)
    v = np.empty((nl, T, HD), np.float32)
    x = np.empty((nl, T, XD), np.float32)
    for l in range(nl):
        _values(cfg, T * HD, gen.token_runs(gen.K, l, reqs, pos0s, counts, HD), k[l].reshape(-1))
        _values(cfg, T * HD, gen.token_runs(gen.V, l, reqs, pos0s, counts, HD), v[l].reshape(-1))
        _values(cfg, T * XD, gen.token_runs(gen.IDXK, l, reqs, pos0s, counts, XD), x[l].reshape(-1))
    return k, v, x


def queries(cfg, layer, reqs, step):
    """q [n][H*d] and q_idx [n][Ih*Id] of decode step `step`."""
    HD = cfg["heads"] * cfg["head_dim"]
    XD = cfg["idx_heads"] * cfg["idx_dim"]
    n = len(reqs)
    q = _values(cfg, n * HD, gen.token_runs(gen.Q, layer, reqs, [step] * n, [1] * n, HD))
    qi = _values(cfg, n * XD, gen.token_runs(gen.QIDX, layer, reqs, [step] * n, [1] * n, XD))
    return q.reshape(n, HD), qi.reshape(n, XD)
