"""GPU-side helpers for the parity tests: a pool in a torch-allocated arena,
device inputs from the seeded generator (the same values the oracle gets
from the host generator), and readers that decode the arena's documented
layout into the oracle's entry encoding."""
from __future__ import annotations

import numpy as np
import torch

from heterogeneous_compressed_kv_gb300 import gen
from heterogeneous_compressed_kv_gb300 import kvpool as K
from tests import harness as H


def tol(cache_dtype):
    """(max-abs, rel-L2) bound on the attention output: fp32 cache 1e-4 / 1e-5;
    bf16 2e-2 / 5e-3; fp8 6e-2 / 5e-3.

    The fp8 max-abs bound alone cannot tell a right output from a wrong one at
    long context: the output is a softmax average over ~10^4 sources, so its
    entries are of order 1e-2 and an all-zero output is within 6e-2.  The
    rel-L2 bound is the one with teeth there.  Both sides read the same
    decoded codes; the GPU's own error sources are the query carried as two
    e4m3 pieces (below 2^-17 of a head's largest element) and each weight
    p * V-scale rounded to f16 (relative 2^-11 at most, about 2.8e-4 RMS, which
    is the expected rel-L2 of the output), plus fp32 summation order.  5e-3 is
    the bf16 bound: over ten times that expectation, and far below what a
    missing source does (tests/test_parity_bounds.py)."""
    return {K.F32: (1e-4, 1e-5), K.BF16: (2e-2, 5e-3), K.FP8_E4M3: (6e-2, 5e-3)}[cache_dtype]


def check_out(gpu, ref, cache_dtype):
    """Both bounds of tol(cache_dtype) on an attention output against the
    oracle's; returns (max-abs error, rel-L2 error)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    amax, rl2 = tol(cache_dtype)
    err = np.max(np.abs(gpu - ref))
    rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= amax, f"max-abs error {err} > {amax}"
    assert rel <= rl2, f"rel-L2 error {rel} > {rl2}"
    return err, rel


class GpuCase:
    def __init__(self, w, max_requests, max_blocks, mbpr, max_batch, max_top_k, gates=None):
        g = H.gates(w) if gates is None else gates
        self.w = w
        self.cfg = K.PoolConfig(m=w["m"], m_prime=w["m_prime"], n_win=w["n_win"], heads=w["heads"],
                                head_dim=w["head_dim"], idx_heads=w["idx_heads"], idx_dim=w["idx_dim"],
                                in_dtype=w["in_dtype"], cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"],
                                max_requests=max_requests, max_blocks=max_blocks, max_blocks_per_request=mbpr,
                                max_batch=max_batch, max_top_k=max_top_k, gate_csa=g[0], gate_hca=g[1],
                                gate_idx=g[2], idx_fp4=w.get("idx_fp4", 0), csa_hot_slots=w.get("csa_hot_slots", 0),
                                csa_host_slots=w.get("csa_host_slots", 0), idx_per_token=w.get("idx_per_token", 0))
        # indexer entries carry a bf16 scale when they are fp8 or fp4
        self.idx_scaled = w["cache_dtype"] == K.FP8_E4M3 or bool(w.get("idx_fp4", 0))
        nbytes = K.required_bytes(self.cfg)
        assert nbytes > 0
        self.arena = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        self.pool = K.Pool(self.cfg, self.arena)
        self.host_pool = self.pool.set_host_pool() if self.cfg.csa_host_slots > 0 else None
        self.nl = len(w["layer_kinds"])
        self.HD = w["heads"] * w["head_dim"]
        self.XD = w["idx_heads"] * w["idx_dim"]
        self.tdtype = torch.float32 if w["in_dtype"] == K.F32 else torch.bfloat16
        self.gdtype = gen.OUT_F32 if w["in_dtype"] == K.F32 else gen.OUT_BF16
        self.vs = {K.F32: 4, K.BF16: 2, K.FP8_E4M3: 1}[w["cache_dtype"]]
        self._host = None

    # ---- inputs on the device (seeded generator, same values as the oracle's) ----
    def _fill(self, t, kind, layer, wids, pos0s, counts, row_len):
        runs = gen.token_runs(kind, layer, wids, pos0s, counts, row_len)
        gen.fill_device(t.data_ptr(), self.gdtype, self.w["seed"], runs, torch.cuda.current_stream().cuda_stream)

    def tokens(self, wids, pos0s, counts):
        T = int(sum(counts))
        k = torch.empty((self.nl, max(T, 1), self.HD), dtype=self.tdtype, device="cuda")
        v = torch.empty_like(k)
        x = torch.empty((self.nl, max(T, 1), self.XD), dtype=self.tdtype, device="cuda")
        for l in range(self.nl):
            self._fill(k[l], gen.K, l, wids, pos0s, counts, self.HD)
            self._fill(v[l], gen.V, l, wids, pos0s, counts, self.HD)
            self._fill(x[l], gen.IDXK, l, wids, pos0s, counts, self.XD)
        return k, v, x

    def queries(self, layer, wids, step):
        n = len(wids)
        q = torch.empty((n, self.HD), dtype=self.tdtype, device="cuda")
        qi = torch.empty((n, self.XD), dtype=self.tdtype, device="cuda")
        self._fill(q, gen.Q, layer, wids, [step] * n, [1] * n, self.HD)
        self._fill(qi, gen.QIDX, layer, wids, [step] * n, [1] * n, self.XD)
        return q, qi

    def append(self, slots, wids, pos0s, counts, check=True):
        k, v, x = self.tokens(wids, pos0s, counts)
        return self.pool.append(slots, counts, k, v, x, check=check)

    def attend(self, layer, slots, wids, step, top_k):
        q, qi = self.queries(layer, wids, step)
        n = len(slots)
        out = torch.empty((n, self.HD), dtype=torch.float32, device="cuda")
        tk = torch.empty((n, max(top_k, 1)), dtype=torch.int32, device="cuda")
        self.pool.decode_attend(layer, slots, q, qi, top_k, out, tk)
        return out, tk[:, :top_k]

    # ---- reading the arena ----
    def host(self, refresh=True):
        if refresh or self._host is None:
            torch.cuda.synchronize()
            self._host = self.arena.cpu().numpy()
        return self._host

    def bytes_at(self, off, n, host=None):
        if host is not None:
            return host[off:off + n]
        return self.arena[off:off + n].cpu().numpy()

    def entry(self, off, host=None):
        lo = self.pool.layout()
        raw = self.bytes_at(off, lo["entry_bytes"], host)
        code = raw[:2 * self.HD * self.vs]
        sc = raw[2 * self.HD * self.vs:2 * self.HD * self.vs + 4].copy().view(np.uint16) if self.vs == 1 \
            else np.zeros(2, np.uint16)
        return code, sc

    def _bid(self, d, slot, e, ids):
        seg = e // d["csa_per_block"]
        return int(ids[seg]) if seg < len(ids) else d["staging_base"] + slot

    def csa_entry(self, layer, slot, e, ids, host=None):
        """A CSA entry where the block's location puts it: the staging slot, a
        GPU slot, or (offloaded) a slot of the host pool."""
        d = self.pool.layout(layer)
        CB = d["csa_per_block"]
        seg = e // CB
        if seg >= len(ids):
            s_ = d["csa_staging_base"] + slot
        else:
            rc, s_ = self.pool.block_location(int(ids[seg]))
            assert rc == 0
        if s_ < 0:
            torch.cuda.synchronize()
            raw = self.host_pool.numpy()
            off = (-1 - s_) * d["host_slot_bytes"] + d["csa_host_offset"] + (e % CB) * d["entry_bytes"]
            return self.entry(off, raw)
        return self.entry(d["csa_offset"] + s_ * d["csa_block_bytes"] + (e % CB) * d["entry_bytes"], host)

    def idx_entry(self, layer, slot, e, ids, host=None):
        """Indexer key e: of CSA entry e, or with per-token keys of token e
        (run e % m' // CB of its block, key e % CB of the run)."""
        d = self.pool.layout(layer)
        CB = d["csa_per_block"]
        if self.w.get("idx_per_token", 0):
            mp, runs = self.w["m_prime"], self.w["m"]
            seg = e // mp
            bid = int(ids[seg]) if seg < len(ids) else d["staging_base"] + slot
            base = d["idx_offset"] + bid * d["idx_block_bytes"] + (e % mp) // CB * (d["idx_block_bytes"] // runs)
        else:
            base = d["idx_offset"] + self._bid(d, slot, e, ids) * d["idx_block_bytes"]
        n_chunks = d["idx_entry_bytes"] // 16
        code = np.concatenate([self.bytes_at(base + (c * CB + e % CB) * 16, 16, host) for c in range(n_chunks)])
        sc = np.zeros(1, np.uint16)
        if self.idx_scaled:
            sc = self.bytes_at(base + d["idx_scale_offset"] + 2 * (e % CB), 2, host).copy().view(np.uint16)
        return code, sc

    def hca_entry(self, layer, bid, host=None):
        d = self.pool.layout(layer)
        return self.entry(d["hca_offset"] + bid * d["hca_block_bytes"], host)

    def window_token(self, layer, slot, pos, host=None):
        d = self.pool.layout(layer)
        return self.entry(d["ring_offset"] + slot * d["ring_request_bytes"] + (pos % self.w["n_win"]) * d["entry_bytes"],
                          host)


def compare_request_state(case, oracle, slot, layers=None, sample=None, rng=None):
    """Block ids, counts and tails bit-exact; every (or a sample of) CSA,
    indexer and HCA entry and window token byte-identical to the oracle's."""
    rc1, i1, ids1 = oracle.request_info(slot)
    rc2, i2, ids2 = case.pool.request_info(slot)
    assert rc1 == rc2 == 0
    assert i1 == i2, (i1, i2)
    assert ids1.tolist() == ids2.tolist()
    host = case.host()
    layers = range(case.nl) if layers is None else layers
    for l in layers:
        kind = case.w["layer_kinds"][l]
        n_csa = i1["n_csa"] if kind in (K.CSA, K.CSA_HCA) else 0
        es = range(n_csa)
        if sample is not None and n_csa > sample:
            es = sorted(set(rng.integers(0, n_csa, sample).tolist()) | {n_csa - 1, 0})
        for e in es:
            rc, c_ref, s_ref = oracle.request_entry(l, slot, 1, e)
            c, s = case.csa_entry(l, slot, e, ids2, host)
            assert np.array_equal(c, c_ref), f"CSA entry {e} of layer {l} differs"
            if case.vs == 1:
                assert np.array_equal(s, s_ref), f"CSA entry {e} scales differ"
            if case.w.get("idx_per_token", 0):
                continue
            rc, c_ref, s_ref = oracle.request_entry(l, slot, 3, e)
            c, s = case.idx_entry(l, slot, e, ids2, host)
            assert np.array_equal(c, c_ref), f"indexer entry {e} of layer {l} differs"
            if case.idx_scaled:
                assert s[0] == s_ref[0], f"indexer entry {e} scale differs"
        if n_csa and case.w.get("idx_per_token", 0):  # one key per token
            ts = range(i1["length"])
            if sample is not None and i1["length"] > 4 * sample:
                ts = sorted(set(rng.integers(0, i1["length"], 4 * sample).tolist()) | {i1["length"] - 1, 0})
            for t in ts:
                rc, c_ref, s_ref = oracle.request_entry(l, slot, 3, t)
                assert rc == 0
                c, s = case.idx_entry(l, slot, t, ids2, host)
                assert np.array_equal(c, c_ref), f"indexer key of token {t} of layer {l} differs"
                if case.idx_scaled:
                    assert s[0] == s_ref[0], f"indexer key of token {t} scale differs"
        if kind in (K.HCA, K.CSA_HCA):
            ts = range(len(ids1))
            if sample is not None and len(ids1) > sample:
                ts = sorted(set(rng.integers(0, len(ids1), sample).tolist()))
            for t in ts:
                rc, c_ref, s_ref = oracle.block_entry(l, int(ids1[t]), 2, 0)
                c, s = case.hca_entry(l, int(ids2[t]), host)
                assert np.array_equal(c, c_ref), f"HCA entry {t} of layer {l} differs"
                if case.vs == 1:
                    assert np.array_equal(s, s_ref)
        L = i1["length"]
        for p in range(max(0, L - case.w["n_win"]), L):
            rc, c_ref, s_ref = oracle.window_token(l, slot, p)
            c, s = case.window_token(l, slot, p, host)
            assert np.array_equal(c, c_ref), f"window token {p} of layer {l} differs"
            if case.vs == 1:
                assert np.array_equal(s, s_ref)
