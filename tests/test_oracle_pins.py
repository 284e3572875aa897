"""Pins of the CPU oracle against what the design pages and mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a
worked example printed on the pages (tests/golden/), a closed form, a library
routine (torch casts, scipy softmax, torch scaled-dot-product attention), a
special case with a known answer, or an error bound.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O
from heterogeneous_compressed_kv_gb300 import gen
from tests import harness as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


U = 2.0 ** -24  # fp32 unit roundoff


def small_cfg(**kw):
    cfg = dict(m=4, m_prime=16, n_win=32, heads=2, head_dim=4, idx_heads=2, idx_dim=4, in_dtype=O.F32,
               cache_dtype=O.F32, n_layers=1, layer_kinds=[O.CSA_HCA], seed=11)
    cfg.update(kw)
    return cfg


def oracle_for(cfg, max_requests=4, max_blocks=64, mbpr=64, gates=None):
    return H.make_oracle(cfg, max_requests, max_blocks, mbpr, gate_override=gates)


# --------------------------------------------------------------------------
# codecs: against torch's casts (library routines)
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([(rng.standard_normal(20000) * 10 ** rng.uniform(-30, 30, 20000)).astype(np.float32),
                        np.float32([0.0, -0.0, 1.0, -3.5, 1e-40, -1e-42])])
    # exact ties: lower 16 bits 0x8000 with odd and even kept parts
    e = np.arange(100, 150, dtype=np.uint32)[:, None]
    mhi = np.arange(0, 128, dtype=np.uint32)[None, :]  # odd and even kept parts
    ties = ((e << 23) | (mhi << 16) | 0x8000).astype(np.uint32).reshape(-1).view(np.float32)
    x = np.concatenate([x, ties, -ties]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.bf16_from_f32(v) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([O.f32_from_bf16(b) for b in ref], np.float32)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 10 ** rng.uniform(-4, 2.6, 20000)).astype(np.float32)
    # every e4m3 value and every midpoint between neighbours (ties to even)
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    finite = np.sort(vals[np.isfinite(vals) & (vals >= 0)])
    mids = ((finite[1:].astype(np.float64) + finite[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, finite, -finite, mids, -mids, np.float32([0.0, -0.0, 463.9, -463.9])])
    x = x[np.abs(x) < 464.0]  # torch does not saturate above the last midpoint
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_from_f32(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_saturates_and_decodes_every_code():
    for v in [448.0, 464.0, 470.0, 1e6, 3.4e38]:
        assert O.e4m3_from_f32(v) == 0x7E
        assert O.e4m3_from_f32(-v) == 0xFE
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        if c in (0x7F, 0xFF):  # NaN encodings, never produced
            continue
        got = O.f32_from_e4m3(c)
        assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c])


def test_fp8_entry_scale_and_error_bound():
    rng = np.random.default_rng(2)
    for trial in range(20):
        x = (rng.standard_normal(512) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
        code, scale = O.encode(O.FP8, x)
        amax = np.float32(np.max(np.abs(x)))
        want = O.bf16_from_f32(np.float32(amax / np.float32(448.0)))
        assert scale == want
        s = O.f32_from_bf16(scale)
        dec = O.decode(O.FP8, code, scale, x.size)
        # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals,
        # absolute <= 2^-10 * scale in the subnormal range, plus saturation
        err = np.abs(dec - x.astype(np.float64))
        bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s) + 1e-30
        sat = np.abs(x / s) > 448
        assert np.all(err[~sat] <= bound[~sat])
    code, scale = O.encode(O.FP8, np.zeros(8, np.float32))
    assert scale == 0x3F80 and np.all(code == 0)


def test_gate_softmax_matches_scipy():
    rng = np.random.default_rng(3)
    for n in (4, 16, 128):
        g = rng.standard_normal(n).astype(np.float32)
        ref = scipy.special.softmax(g.astype(np.float64)).astype(np.float32)
        got = O.softmax_f32(g)
        assert np.max(np.abs(got.view(np.int32) - ref.view(np.int32))) <= 1
    one_hot = O.softmax_f32(np.float32([-np.inf, 0.0, -np.inf, -np.inf]))
    assert list(one_hot) == [0.0, 1.0, 0.0, 0.0]
    assert list(O.softmax_f32(np.zeros(4, np.float32))) == [0.25] * 4


# --------------------------------------------------------------------------
# compressor: special cases with known answers and the fp32 chain bound
# --------------------------------------------------------------------------

def one_hot_gates(cfg, hot_csa, hot_hca, hot_idx):
    """logits -inf except one position per head: alpha is exactly one-hot"""
    nl = cfg["n_layers"]
    g_csa = np.full((nl, cfg["heads"], cfg["m"]), -np.inf, np.float32)
    g_hca = np.full((nl, cfg["heads"], cfg["m_prime"]), -np.inf, np.float32)
    g_idx = np.full((nl, cfg["idx_heads"], cfg["m"]), -np.inf, np.float32)
    for l in range(nl):
        for h in range(cfg["heads"]):
            g_csa[l, h, hot_csa[h]] = 0
            g_hca[l, h, hot_hca[h]] = 0
        for g in range(cfg["idx_heads"]):
            g_idx[l, g, hot_idx[g]] = 0
    return g_csa, g_hca, g_idx


@pytest.mark.parametrize("cache", [O.F32, O.BF16])
def test_compressor_one_hot_gate_selects_that_token(cache):
    cfg = small_cfg(cache_dtype=cache, in_dtype=O.BF16 if cache == O.BF16 else O.F32)
    o = oracle_for(cfg, gates=one_hot_gates(cfg, [1, 3], [5, 14], [2, 0]))
    HD, XD = o.HD, o.XD
    rng = np.random.default_rng(4)
    toks = torch.from_numpy(rng.standard_normal(16 * 2 * HD).astype(np.float32)).bfloat16().float().numpy()
    toks = toks.reshape(16, 2, 2, 4)  # [token][K/V][head][dim], bf16-representable
    code, sc = o.compress_kv(0, 1, toks[:4].reshape(4, -1))
    e = o.entry_values(code, sc)  # [2][H][d]
    for h, hot in enumerate([1, 3]):
        assert np.array_equal(e[:, h, :], toks[hot, :, h, :])  # K and V share the gate
    code, sc = o.compress_kv(0, 2, toks.reshape(16, -1))
    e = o.entry_values(code, sc)
    for h, hot in enumerate([5, 14]):
        assert np.array_equal(e[:, h, :], toks[hot, :, h, :])
    keys = toks[:4, 0].reshape(4, XD)
    code, sc = o.compress_idx(0, keys)
    dec = O.decode(cache, code, int(sc[0]), XD).reshape(2, 4)
    assert np.array_equal(dec[0], keys[2].reshape(2, 4)[0])
    assert np.array_equal(dec[1], keys[0].reshape(2, 4)[1])


def test_compressor_equal_gates_is_mean_pooling_and_random_gates_within_bound():
    cfg = small_cfg()
    rng = np.random.default_rng(5)
    zeros = (np.zeros((1, 2, 4), np.float32), np.zeros((1, 2, 16), np.float32), np.zeros((1, 2, 4), np.float32))
    o = oracle_for(cfg, gates=zeros)
    toks = rng.standard_normal((16, 16)).astype(np.float32)
    code, _ = o.compress_kv(0, 1, toks[:4])
    got = code.view(np.float32)
    exact = toks[:4].astype(np.float64).mean(axis=0)
    assert np.all(np.abs(got - exact) <= 4 * U * np.abs(toks[:4]).astype(np.float64).mean(axis=0) + 1e-45)
    code, _ = o.compress_kv(0, 2, toks)
    exact = toks.astype(np.float64).mean(axis=0)
    assert np.all(np.abs(code.view(np.float32) - exact) <= 16 * U * np.abs(toks).mean(axis=0) + 1e-45)
    # random gates: sum_i alpha_i x_i in fp64 with the fp32 alphas, chain error <= m u sum|alpha x|
    g = H.gates(dict(cfg, seed=7))
    o = oracle_for(cfg, gates=g)
    for kind, cnt, gl in ((1, 4, g[0]), (2, 16, g[1])):
        alpha = np.stack([O.softmax_f32(gl[0, h]) for h in range(2)]).astype(np.float64)  # [H][cnt]
        t = rng.standard_normal((cnt, 2, 2, 4)).astype(np.float32)
        code, _ = o.compress_kv(0, kind, t.reshape(cnt, -1))
        got = code.view(np.float32).reshape(2, 2, 4)
        ref = np.einsum("hi,ikhj->khj", alpha, t.astype(np.float64))
        mag = np.einsum("hi,ikhj->khj", np.abs(alpha), np.abs(t.astype(np.float64)))
        assert np.all(np.abs(got - ref) <= cnt * U * mag + 1e-45)
        # a dropped term or a wrong head's gate would exceed this bound
        assert np.max(np.abs(got - ref)) < 1e-5


# --------------------------------------------------------------------------
# bookkeeping: the pages' worked example and closed forms
# --------------------------------------------------------------------------

def append_tokens(o, cfg, reqs, pos0s, counts, wids=None):
    wids = reqs if wids is None else wids
    k, v, x = H.tokens(cfg, wids, pos0s, counts)
    return o.append(reqs, counts, k, v, x)


def tiny_bookkeeping_cfg(**kw):
    return small_cfg(m=4, m_prime=128, n_win=128, heads=1, head_dim=4, idx_heads=1, idx_dim=4, **kw)


def test_golden_l130_example():
    g = golden("l130_example.json")
    cfg = tiny_bookkeeping_cfg()
    o = oracle_for(cfg)
    rc, r = o.alloc_request()
    assert rc == O.OK
    assert append_tokens(o, cfg, [r], [0], [g["length"]]) == O.OK
    rc, info, ids = o.request_info(r)
    assert info["n_csa"] == g["classical_csa_entries"]
    assert info["n_hca"] == g["classical_hca_entries"]
    assert info["n_blocks"] == g["sealed_blocks"] and len(ids) == 1
    assert info["hca_tail"] == g["tail_tokens"] and info["csa_tail"] == g["tail_tokens"]
    # every CSA entry of tokens 1..128 is in the sealed block; none is staged
    for e in range(32):
        rc1, c1, s1 = o.request_entry(0, r, 1, e)
        rc2, c2, s2 = o.block_entry(0, int(ids[0]), 1, e)
        assert rc1 == rc2 == O.OK and np.array_equal(c1, c2)
    assert o.request_entry(0, r, 1, 32)[0] == O.ERR_INVALID_ARG


def test_golden_block_shape_and_decompositions():
    g = golden("block_shape.json")
    tb = golden("tail_bounds.json")
    cfg = tiny_bookkeeping_cfg()
    o = oracle_for(cfg, max_blocks=64, mbpr=64)
    assert o.CB == g["csa_per_block"]
    rc, r = o.alloc_request()
    L = 0
    rng = np.random.default_rng(6)
    seen_csa_tail, seen_hca_tail = set(), set()
    checkpoints = {d[0]: d for d in g["decompositions"]}
    for target in sorted(set(list(checkpoints) + list(rng.integers(0, 1500, 40)))):
        if target < L:
            continue
        assert append_tokens(o, cfg, [r], [L], [target - L]) == O.OK
        L = target
        rc, info, ids = o.request_info(r)
        q, rem = divmod(L, g["block_tokens"])
        assert info["n_blocks"] == q and len(ids) == q
        assert info["n_csa"] == g["csa_per_block"] * q + rem // cfg["m"]
        assert info["n_hca"] == g["hca_per_block"] * q
        assert info["hca_tail"] == rem and info["csa_tail"] == L % cfg["m"]
        assert info["csa_tail"] <= tb["csa_tail_max"] and info["hca_tail"] <= tb["hca_tail_max"]
        seen_csa_tail.add(info["csa_tail"])
        seen_hca_tail.add(info["hca_tail"])
        if L in checkpoints:
            _, qq, rr = checkpoints[L]
            assert (info["n_blocks"], info["hca_tail"]) == (qq, rr)


def test_golden_hca_entries_at_one_million():
    g = golden("hca_1m.json")
    cfg = small_cfg(m=4, m_prime=128, n_win=128, heads=1, head_dim=1, idx_heads=1, idx_dim=1)
    o = oracle_for(cfg, max_requests=1, max_blocks=8192, mbpr=8192)
    rc, r = o.alloc_request()
    n = g["length"]
    ones = np.ones((1, n, 1), np.float32)
    assert o.append([r], [n], ones, ones, ones) == O.OK
    rc, info, ids = o.request_info(r)
    assert info["n_hca"] == g["hca_entries"] and info["n_blocks"] == g["hca_entries"]
    assert info["hca_tail"] == 0 and info["window"] == 128
    assert sorted(ids.tolist()) == list(range(8192))
    assert o.free_block_count() == 0


def test_golden_window_is_whole_blocks_and_state_stays_constant():
    g = golden("window_lcm.json")
    assert g["n_win"] == g["window_blocks"] * g["lcm"]
    cfg = small_cfg(m=4, m_prime=128, n_win=g["n_win"], heads=1, head_dim=1, idx_heads=1, idx_dim=1)
    o = oracle_for(cfg, max_requests=1, max_blocks=512, mbpr=512)
    rc, r = o.alloc_request()
    L = 0
    for total, blocks, tail in sorted(g["demo_totals"]):
        ones = np.ones((1, total - L, 1), np.float32)
        assert o.append([r], [total - L], ones, ones, ones) == O.OK
        L = total
        rc, info, _ = o.request_info(r)
        assert (info["n_blocks"], info["hca_tail"]) == (blocks, tail)
        assert info["window"] == g["n_win"]  # State: fixed window + tail < 128
    # a window that is not a whole number of blocks is refused
    with pytest.raises(ValueError):
        oracle_for(small_cfg(m=4, m_prime=128, n_win=4000))


def test_golden_volume_ratio_of_entry_bytes():
    g = golden("volume_ratio.json")
    o = oracle_for(small_cfg(m=4, m_prime=128, n_win=128, cache_dtype=O.FP8, in_dtype=O.BF16, heads=16,
                             head_dim=128))
    per_token_swa = o.esz          # one window slot per token
    per_token_csa = o.esz / o.m   # one CSA entry per 4 tokens
    per_token_hca = o.esz / o.m_prime
    assert per_token_swa / per_token_hca == g["swa"] and per_token_csa / per_token_hca == g["csa"]


def test_window_holds_exactly_the_last_tokens():
    for cache in (O.F32, O.BF16, O.FP8):
        cfg = small_cfg(cache_dtype=cache, in_dtype=O.F32 if cache == O.F32 else O.BF16)
        o = oracle_for(cfg)
        rc, r = o.alloc_request()
        L = 0
        for n in (5, 1, 30, 3, 17):
            assert append_tokens(o, cfg, [r], [L], [n]) == O.OK
            L += n
            k, v, _ = H.tokens(cfg, [r], [0], [L])
            for p in range(max(0, L - cfg["n_win"]), L):
                rc, code, sc = o.window_token(0, r, p)
                assert rc == O.OK
                ck, sk = O.encode(cache, k[0, p])
                cv, sv = O.encode(cache, v[0, p])
                assert np.array_equal(code, np.concatenate([ck, cv]))
                if cache == O.FP8:
                    assert (sc[0], sc[1]) == (sk, sv)
            # a position that left the window is gone
            if L > cfg["n_win"]:
                assert o.window_token(0, r, L - cfg["n_win"] - 1)[0] == O.ERR_INVALID_ARG


def test_entries_compress_exactly_their_own_token_groups():
    """CSA entry e holds tokens 4e..4e+3 and HCA entry t tokens 128t..128t+127,
    whether sealed or staged (checked through the pure compressor on the
    regenerated tokens; an off-by-one group boundary fails here)."""
    cfg = small_cfg(cache_dtype=O.BF16, in_dtype=O.BF16)
    o = oracle_for(cfg)
    rc, r = o.alloc_request()
    L = 0
    for n in (7, 9, 1, 22, 13):
        assert append_tokens(o, cfg, [r], [L], [n]) == O.OK
        L += n
    k, v, x = H.tokens(cfg, [r], [0], [L])
    kv = np.concatenate([k[0], v[0]], axis=1)  # [L][2*HD]
    rc, info, ids = o.request_info(r)
    for e in range(L // 4):
        c_ref, s_ref = o.compress_kv(0, 1, kv[4 * e:4 * e + 4])
        rc, c, s = o.request_entry(0, r, 1, e)
        assert np.array_equal(c, c_ref)
        x_ref, _ = o.compress_idx(0, x[0, 4 * e:4 * e + 4])
        rc, c, s = o.request_entry(0, r, 3, e)
        assert np.array_equal(c, x_ref)
    for t in range(L // 16):
        c_ref, _ = o.compress_kv(0, 2, kv[16 * t:16 * t + 16])
        rc, c, s = o.block_entry(0, int(ids[t]), 2, 0)
        assert rc == O.OK and np.array_equal(c, c_ref)


# --------------------------------------------------------------------------
# prefix sharing, allocation policy and errors
# --------------------------------------------------------------------------

def test_prefix_sharing_refcounts_and_immutability():
    cfg = small_cfg(cache_dtype=O.BF16, in_dtype=O.BF16)
    o = oracle_for(cfg, max_blocks=8)
    _, a = o.alloc_request()
    _, b = o.alloc_request()
    assert append_tokens(o, cfg, [a], [0], [40]) == O.OK  # 2 sealed blocks of 16
    _, ia, ids_a = o.request_info(a)
    k, v, _ = H.tokens(cfg, [a], [0], [32])
    w = min(32, cfg["n_win"])
    assert o.share_prefix(b, a, 32, k[:, 32 - w:32], v[:, 32 - w:32]) == O.OK
    _, ib, ids_b = o.request_info(b)
    assert ids_b.tolist() == ids_a[:2].tolist() and ib["length"] == 32 and ib["hca_tail"] == 0
    assert all(o.block_refcount(int(i)) == 2 for i in ids_a[:2])
    before = [o.block_entry(0, int(i), 1, 3)[1].copy() for i in ids_a[:2]]
    # b grows on its own: new blocks get new ids, shared blocks do not change
    assert append_tokens(o, cfg, [b], [32], [20], wids=[7]) == O.OK
    _, ib, ids_b2 = o.request_info(b)
    assert ids_b2[:2].tolist() == ids_a[:2].tolist() and ids_b2[2] not in ids_a.tolist()
    after = [o.block_entry(0, int(i), 1, 3)[1] for i in ids_a[:2]]
    assert all(np.array_equal(x, y) for x, y in zip(before, after))
    # refcounts fall to zero only when both have gone
    assert o.free_request(a) == O.OK
    assert all(o.block_refcount(int(i)) == 1 for i in ids_a[:2])
    free_before = o.free_block_count()
    assert o.free_request(b) == O.OK
    assert o.free_block_count() == free_before + 3 and o.free_block_count() == 8
    # smallest free id is reused first
    _, c = o.alloc_request()
    assert append_tokens(o, cfg, [c], [0], [16]) == O.OK
    assert o.request_info(c)[2].tolist() == [0]


def test_share_prefix_refusals():
    cfg = small_cfg()
    o = oracle_for(cfg)
    _, a = o.alloc_request()
    _, b = o.alloc_request()
    append_tokens(o, cfg, [a], [0], [40])
    win = np.zeros((1, 32, 8), np.float32)
    assert o.share_prefix(b, a, 24, win, win) == O.ERR_NOT_SHAREABLE  # not whole blocks
    assert o.share_prefix(b, a, 48, win, win) == O.ERR_NOT_SHAREABLE  # beyond the sealed blocks
    assert o.share_prefix(b, b, 16, win, win) == O.ERR_BAD_REQUEST
    assert o.share_prefix(b, 3, 16, win, win) == O.ERR_BAD_REQUEST
    assert o.share_prefix(b, a, 16, win, win) == O.OK
    assert o.share_prefix(b, a, 16, win, win) == O.ERR_NOT_SHAREABLE  # dst not fresh


def test_errors_leave_state_unchanged():
    cfg = small_cfg()
    o = oracle_for(cfg, max_requests=3, max_blocks=3, mbpr=2)
    _, a = o.alloc_request()
    _, b = o.alloc_request()
    assert append_tokens(o, cfg, [a, b], [0, 0], [15, 15]) == O.OK
    snap = [o.request_info(r)[1] for r in (a, b)]
    # a and b both seal one block: fine; then 2 more seals with 1 free block left
    assert append_tokens(o, cfg, [a, b], [15, 15], [1, 1]) == O.OK
    snap = [o.request_info(r)[1] for r in (a, b)]
    assert append_tokens(o, cfg, [a, b], [16, 16], [16, 16]) == O.ERR_OUT_OF_BLOCKS
    assert [o.request_info(r)[1] for r in (a, b)] == snap
    assert append_tokens(o, cfg, [a], [16], [40]) == O.ERR_CAPACITY  # > 2 blocks for one request
    assert append_tokens(o, cfg, [a, a], [16, 16], [1, 1]) == O.ERR_INVALID_ARG  # duplicate
    assert o.append([2], [1], np.zeros((1, 1, 8)), np.zeros((1, 1, 8)), np.zeros((1, 1, 8))) == O.ERR_BAD_REQUEST
    assert [o.request_info(r)[1] for r in (a, b)] == snap
    _, c = o.alloc_request()
    assert o.alloc_request()[0] == O.ERR_OUT_OF_REQUESTS
    assert o.free_request(c) == O.OK and o.free_request(c) == O.ERR_BAD_REQUEST


# --------------------------------------------------------------------------
# indexer score and top-k
# --------------------------------------------------------------------------

def test_score_special_cases_and_bound():
    cfg = small_cfg(idx_heads=4, idx_dim=64)
    o = oracle_for(cfg)
    rng = np.random.default_rng(8)
    key = rng.standard_normal(256).astype(np.float32)
    code, sc = O.encode(O.F32, key)
    for v0 in (0, 77, 255):
        q = np.zeros(256, np.float32)
        q[v0] = 1.0
        assert o.score(code, sc, q) == key[v0]
    q = rng.standard_normal(256).astype(np.float32)
    ref = float(np.dot(q.astype(np.float64), key.astype(np.float64)))
    assert abs(o.score(code, sc, q) - ref) <= 256 * U * float(np.dot(np.abs(q), np.abs(key)))
    # fp8: the chain runs on the codes, the scale multiplies once at the end
    o8 = oracle_for(dict(cfg, cache_dtype=O.FP8, in_dtype=O.BF16))
    c8, s8 = O.encode(O.FP8, key)
    dec = O.decode(O.FP8, c8, s8, 256)
    ref = float(np.dot(q.astype(np.float64), dec))
    assert abs(o8.score(c8, s8, q) - ref) <= 257 * U * float(np.dot(np.abs(q), np.abs(dec)))


def test_topk_ties_signed_zero_and_limits():
    assert O.topk([1, 3, 3, 2, 3], 2).tolist() == [1, 2]
    assert O.topk([5, 5, 5, 5], 3).tolist() == [0, 1, 2]
    assert O.topk(np.float32([-0.0, 0.0]), 1).tolist() == [0]
    assert O.topk(np.float32([0.0, -0.0]), 1).tolist() == [0]
    assert O.topk([3, 1, 2], 5).tolist() == [0, 1, 2, -1, -1]
    assert O.topk([3, 1, 2], 0).tolist() == []
    rng = np.random.default_rng(9)
    s = rng.standard_normal(5000).astype(np.float32)
    for k in (1, 17, 512, 4999):
        ref = np.sort(np.argsort(-s.astype(np.float64), kind="stable")[:k])
        assert np.array_equal(O.topk(s, k), ref)


def test_stateful_topk_matches_brute_force_over_fp64_scores():
    cfg = small_cfg(idx_heads=4, idx_dim=64, cache_dtype=O.BF16, in_dtype=O.BF16, m_prime=128, n_win=128)
    o = oracle_for(cfg, max_blocks=16, mbpr=16)
    _, r = o.alloc_request()
    append_tokens(o, cfg, [r], [0], [1000])
    q, qi = H.queries(cfg, 0, [r], 0)
    n_c = 250
    entries = [o.request_entry(0, r, 3, e) for e in range(n_c)]
    s64 = np.array([np.dot(qi[0].astype(np.float64), O.decode(O.BF16, c, int(sc[0]), 256)) for _, c, sc in entries])
    for k in (16, 100):
        order = np.argsort(-s64, kind="stable")
        gap = s64[order[k - 1]] - s64[order[k]]
        bound = 2 * 256 * U * np.max(np.abs(s64)) * 8
        assert gap > bound  # the seeded draw separates the k-th score
        rc, out, tk = o.decode_attend(0, [r], q, qi, k)
        assert rc == O.OK and np.array_equal(tk[0], np.sort(order[:k]))


# --------------------------------------------------------------------------
# attention: closed form and textbook special cases
# --------------------------------------------------------------------------

def test_attention_with_zero_keys_is_the_mean_of_values():
    cfg = small_cfg()
    o = oracle_for(cfg)
    rng = np.random.default_rng(10)
    n = 37
    ent = np.concatenate([np.zeros((n, 8), np.float32), rng.standard_normal((n, 8)).astype(np.float32)], axis=1)
    codes = ent.view(np.uint8).reshape(-1)
    rc, out = o.attend_sources(codes, np.zeros((n, 2), np.uint16), rng.standard_normal(8).astype(np.float32))
    assert rc == O.OK
    assert np.allclose(out.reshape(-1), ent[:, 8:].astype(np.float64).mean(axis=0), rtol=0, atol=1e-15)


def sdpa(q, keys, vals):
    """textbook softmax attention per head via torch (float64): q [H][d],
    keys/vals [n][H][d] -> [H][d]"""
    qt = torch.from_numpy(np.asarray(q, np.float64))[:, None, :]        # [H][1][d]
    kt = torch.from_numpy(np.asarray(keys, np.float64)).permute(1, 0, 2)  # [H][n][d]
    vt = torch.from_numpy(np.asarray(vals, np.float64)).permute(1, 0, 2)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0, :].numpy()


@pytest.mark.parametrize("top_k", [10 ** 6, 5])
def test_attention_over_concatenated_sources_is_textbook(top_k):
    """With one-hot gates every CSA / HCA entry is an exact token; with top_k
    covering all entries the result is plain softmax attention over
    [those tokens, the window] (spec pin); with a small top_k it is the
    same over the selected subset."""
    cfg = small_cfg(heads=2, head_dim=4, m=4, m_prime=16, n_win=32)
    hot_c, hot_h = [2, 2], [9, 9]
    o = oracle_for(cfg, gates=one_hot_gates(cfg, hot_c, hot_h, [0, 0]))
    _, r = o.alloc_request()
    L = 75
    append_tokens(o, cfg, [r], [0], [L])
    k, v, _ = H.tokens(cfg, [r], [0], [L])
    q, qi = H.queries(cfg, 0, [r], 3)
    rc, out, tk = o.decode_attend(0, [r], q, qi, top_k)
    assert rc == O.OK
    n_c = L // 4
    sel = np.arange(n_c) if top_k >= n_c else tk[0]
    src = [4 * e + hot_c[0] for e in sel] + [16 * t + hot_h[0] for t in range(L // 16)] + \
          list(range(L - cfg["n_win"], L))
    keys = k[0, src].reshape(-1, 2, 4)
    vals = v[0, src].reshape(-1, 2, 4)
    ref = sdpa(q[0].reshape(2, 4), keys, vals)
    assert np.allclose(out[0], ref, rtol=1e-12, atol=1e-12)


def test_swa_only_layer_is_sliding_window_attention():
    cfg = small_cfg(n_layers=2, layer_kinds=[O.SWA_ONLY, O.CSA_HCA], n_win=16, m_prime=16)
    o = oracle_for(cfg)
    _, r = o.alloc_request()
    L = 50
    append_tokens(o, cfg, [r], [0], [L])
    k, v, _ = H.tokens(cfg, [r], [0], [L])
    q, qi = H.queries(cfg, 0, [r], 0)
    rc, out, _ = o.decode_attend(0, [r], q, qi, 4)
    assert rc == O.OK
    ref = sdpa(q[0].reshape(2, 4), k[0, L - 16:].reshape(-1, 2, 4), v[0, L - 16:].reshape(-1, 2, 4))
    assert np.allclose(out[0], ref, rtol=1e-12, atol=1e-12)
    # the SWA-only layer never forms entries, but blocks still seal (one id spans all layers)
    _, info, ids = o.request_info(r)
    assert info["n_blocks"] == 3 and o.request_entry(0, r, 1, 0)[0] == O.ERR_INVALID_ARG


# --------------------------------------------------------------------------
# FP4 (e2m1) indexer entries
# --------------------------------------------------------------------------
def _e2m1_value(code):
    """Value of a 4-bit e2m1 code from its bit layout: sign, 2 exponent bits
    (bias 1), 1 mantissa bit; exponent 0 is subnormal (0.m x 2^0)."""
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
    return -mag if s else mag


def test_e2m1_codes_decode_to_the_format_values():
    assert [_e2m1_value(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for c in range(16):
        v = O.f32_from_e2m1(c)
        assert v == _e2m1_value(c) and math.copysign(1, v) == (-1 if c & 8 else 1)


def test_e2m1_rounds_to_nearest_even_and_saturates():
    from fractions import Fraction
    mags = [Fraction(_e2m1_value(c)) for c in range(8)]

    def expect(x):
        s = 8 if math.copysign(1, x) < 0 else 0
        a = Fraction(abs(x))
        if a >= 6:
            return s | 7
        d = [abs(a - v) for v in mags]
        best = min(d)
        ties = [c for c in range(8) if d[c] == best]
        return s | (ties[0] if len(ties) == 1 else [c for c in ties if c & 1 == 0][0])

    xs = [0.0, -0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 1e9, -0.25, -5.0, -1e-30, 0.2499, 0.2501,
          4.999, 5.001]
    rng = np.random.default_rng(21)
    xs += list(rng.uniform(-8, 8, 2000).astype(np.float32)) + list((rng.standard_normal(500) * 1e-3).astype(np.float32))
    for x in xs:
        x = float(np.float32(x))
        assert O.e2m1_from_f32(x) == expect(x), x


def test_fp4_entry_scale_packing_and_error_bound():
    rng = np.random.default_rng(22)
    for trial in range(20):
        x = (rng.standard_normal(256) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        code, sc = O.encode(O.FP4, x)
        assert code.size == 128
        amax = np.float32(np.max(np.abs(x)))
        assert sc == torch.tensor(float(amax / np.float32(6.0)), dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
        s = float(torch.tensor([sc], dtype=torch.int16).view(torch.bfloat16).float().item())
        for i in range(256):
            nib = (int(code[i // 2]) >> (4 * (i & 1))) & 15
            assert nib == O.e2m1_from_f32(float(np.float32(x[i] / np.float32(s))))
        dec = O.decode(O.FP4, code, sc, 256)
        assert np.all(np.abs(dec - x) <= 0.25 * np.maximum(np.abs(x), s) + 1e-30)
    code, sc = O.encode(O.FP4, np.zeros(32, np.float32))
    assert sc == 0x3F80 and not code.any()


def test_fp4_indexer_score_is_the_fixed_chain_times_the_scale():
    cfg = small_cfg(idx_heads=4, idx_dim=64, in_dtype=O.BF16, cache_dtype=O.FP8, idx_fp4=1)
    o = oracle_for(cfg)
    assert o.xsz == 128
    rng = np.random.default_rng(23)
    keys = rng.standard_normal((4, 256)).astype(np.float32)
    code, sc = o.compress_idx(0, keys)
    s = np.float32(torch.tensor([int(sc[0])], dtype=torch.int16).view(torch.bfloat16).float().item())
    q = torch.tensor(rng.standard_normal(256), dtype=torch.bfloat16).float().numpy()
    acc = np.float32(0.0)
    for v in range(256):
        val = np.float32(_e2m1_value((int(code[v // 2]) >> (4 * (v & 1))) & 15))
        acc = np.float32(acc + np.float32(q[v] * val))  # the product of bf16 and e2m1 values is exact in fp32
    assert o.score(code, sc, q) == np.float32(acc * s)
