"""Pieces of a single-request oracle decode step at 1M-token context, run in
spawned worker processes (test infrastructure: only the parity tests call
it).  Every piece is a pure oracle step on tokens drawn from the seeded
generator: indexer entries and their scores, HCA entries, CSA entries."""
from __future__ import annotations

import numpy as np

import oracle as O

from heterogeneous_compressed_kv_gb300 import gen
from tests import harness as H

_ORACLES = {}


def _oracle(cfg):
    key = (cfg["name"], cfg["seed"], cfg.get("idx_fp4", 0), cfg.get("idx_per_token", 0))
    if key not in _ORACLES:
        _ORACLES[key] = H.make_oracle(cfg, 1, 1, 1)
    return _ORACLES[key]


def _rows(cfg, kind, wid, pos0, count, width, layer=0):
    out = np.empty(count * width, np.float32)
    H._values(cfg, count * width, gen.token_runs(kind, layer, [wid], [pos0], [count], width), out)
    return out.reshape(count, width)


def idx_scores(cfg, wid, q_idx, e0, e1, layer=0):
    """Indexer scores of CSA entries [e0, e1) of workload request `wid`."""
    o = _oracle(cfg)
    m, XD = cfg["m"], cfg["idx_heads"] * cfg["idx_dim"]
    keys = _rows(cfg, gen.IDXK, wid, e0 * m, (e1 - e0) * m, XD, layer)
    out = np.empty(e1 - e0, np.float32)
    if cfg.get("idx_per_token", 0):  # each token's key encoded alone; the entry mixes its m tokens
        for j in range(e1 - e0):
            enc = [O.encode(o.idx_dtype, keys[j * m + i]) for i in range(m)]
            codes = np.concatenate([c for c, _ in enc])
            scales = np.array([sc for _, sc in enc], np.uint16)
            out[j] = o.score_tokens(layer, codes, scales, q_idx)
        return out
    for j in range(e1 - e0):
        code, sc = o.compress_idx(layer, keys[j * m:(j + 1) * m])
        out[j] = o.score(code, sc, q_idx)
    return out


def token_keys(cfg, wid, ts, layer=0):
    """Per-token indexer keys (codes, scale) of tokens `ts`."""
    o = _oracle(cfg)
    XD = cfg["idx_heads"] * cfg["idx_dim"]
    return [O.encode(o.idx_dtype, _rows(cfg, gen.IDXK, wid, t, 1, XD, layer)[0]) for t in ts]


def idx_entries(cfg, wid, es, layer=0):
    """Indexer entries (codes, scales) of the CSA entries `es`."""
    o = _oracle(cfg)
    m, XD = cfg["m"], cfg["idx_heads"] * cfg["idx_dim"]
    res = []
    for e in es:
        code, sc = o.compress_idx(layer, _rows(cfg, gen.IDXK, wid, e * m, m, XD, layer))
        res.append((code, sc))
    return res


def _kv_rows(cfg, wid, pos0, count, layer=0):
    HD = cfg["heads"] * cfg["head_dim"]
    return np.concatenate([_rows(cfg, gen.K, wid, pos0, count, HD, layer),
                           _rows(cfg, gen.V, wid, pos0, count, HD, layer)], axis=1)


def kv_entries(cfg, wid, kind, groups, layer=0):
    """CSA (kind 1, groups of m tokens) or HCA (kind 2, groups of m' tokens)
    entries of `groups` -> (codes [n][esz], scales [n][2])."""
    o = _oracle(cfg)
    g = cfg["m"] if kind == 1 else cfg["m_prime"]
    codes = np.empty((len(groups), o.esz), np.uint8)
    scales = np.empty((len(groups), 2), np.uint16)
    for j, e in enumerate(groups):
        codes[j], scales[j] = o.compress_kv(layer, kind, _kv_rows(cfg, wid, e * g, g, layer))
    return codes, scales


def window_entries(cfg, wid, pos0, count, layer=0):
    """Window tokens [pos0, pos0 + count): K and V halves encoded with one
    scale each."""
    from oracle import encode
    HD = cfg["heads"] * cfg["head_dim"]
    rows = _kv_rows(cfg, wid, pos0, count, layer)
    o = _oracle(cfg)
    codes = np.empty((count, o.esz), np.uint8)
    scales = np.empty((count, 2), np.uint16)
    for t in range(count):
        ck, sk = encode(cfg["cache_dtype"], rows[t, :HD])
        cv, sv = encode(cfg["cache_dtype"], rows[t, HD:])
        codes[t] = np.concatenate([ck, cv])
        scales[t] = (sk, sv)
    return codes, scales
