"""CPU tests of the C-ABI library: it loads, exports every declared symbol,
validates configurations, lays out the arena sanely, and its host bookkeeping
(block ids, refcounts, tails, errors) matches the oracle bit for bit.  No
kernel runs here (pools are created with KVPOOL_FLAG_NO_DEVICE)."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle as O
from heterogeneous_compressed_kv_gb300 import kvpool as K
from tests import harness as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvpool.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvpool_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(K.EXPORTS)
    L = K.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", K.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (kvpool_\w+)", out))
    assert set(names) <= exported


def cfg_of(w, **kw):
    g = H.gates(w)
    d = dict(m=w["m"], m_prime=w["m_prime"], n_win=w["n_win"], heads=w["heads"], head_dim=w["head_dim"],
             idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"], cache_dtype=w["cache_dtype"],
             layer_kinds=w["layer_kinds"], max_requests=8, max_blocks=64, max_blocks_per_request=32, max_batch=8,
             max_top_k=64, gate_csa=g[0], gate_hca=g[1], gate_idx=g[2], flags=K.FLAG_NO_DEVICE)
    d.update(kw)
    return K.PoolConfig(**d)


def base_workload(**kw):
    w = dict(m=4, m_prime=128, n_win=128, heads=4, head_dim=64, idx_heads=1, idx_dim=32, in_dtype=K.F32,
             cache_dtype=K.F32, n_layers=1, layer_kinds=[K.CSA_HCA], seed=5)
    w.update(kw)
    return w


@pytest.mark.parametrize("bad", [dict(m=3), dict(m=5, m_prime=128), dict(n_win=100), dict(n_win=64),
                                 dict(head_dim=96), dict(cache_dtype=7), dict(in_dtype=2), dict(max_batch=0),
                                 dict(heads=1), dict(idx_dim=3), dict(layer_kinds=[9]),
                                 dict(idx_fp4=1, idx_dim=16), dict(idx_fp4=2)])
def test_invalid_configs_are_refused(bad):
    w = base_workload()
    wk = {k: v for k, v in bad.items() if k in w}
    ck = {k: v for k, v in bad.items() if k not in w}
    if "layer_kinds" in bad:
        wk.pop("layer_kinds", None)
        ck["layer_kinds"] = bad["layer_kinds"]
    cfg = cfg_of(base_workload(**wk), **ck)
    assert K.required_bytes(cfg) == 0
    with pytest.raises(K.KvpoolError):
        K.Pool(cfg)


def test_indexer_blocks_must_fit_the_score_kernels_shared_memory():
    """One block's indexer keys are staged whole in shared memory: 32 fp32
    entries of 32 x 64 values (256 KiB) cannot be, so the config is refused;
    the same keys in bf16 (128 KiB) take one score warp and are accepted, as
    are 4 x 64 fp32 keys (32 KiB per block, four warps)."""
    big = dict(heads=16, head_dim=64, idx_heads=32, idx_dim=64)
    assert K.required_bytes(cfg_of(base_workload(**big))) == 0
    with pytest.raises(K.KvpoolError):
        K.Pool(cfg_of(base_workload(**big)))
    assert K.required_bytes(cfg_of(base_workload(cache_dtype=K.BF16, in_dtype=K.BF16, **big))) > 0
    assert K.required_bytes(cfg_of(base_workload(heads=16, head_dim=128, idx_heads=4, idx_dim=64))) > 0


def test_fp4_indexer_layout():
    w = base_workload(cache_dtype=K.BF16, in_dtype=K.BF16, heads=16, head_dim=128, idx_heads=4, idx_dim=64)
    p = K.Pool(cfg_of(w, idx_fp4=1))
    lo, d = p.layout(), p.layout(0)
    assert lo["idx_entry_bytes"] == 128
    assert d["idx_scale_offset"] == 32 * 128 and d["idx_block_bytes"] == 32 * 128 + 64


@pytest.mark.parametrize("cache", [K.F32, K.BF16, K.FP8_E4M3])
def test_layout_is_aligned_and_disjoint(cache):
    w = base_workload(cache_dtype=cache, in_dtype=K.BF16 if cache != K.F32 else K.F32, heads=16, head_dim=128,
                      idx_heads=4, idx_dim=64, n_layers=4, layer_kinds=[K.SWA_ONLY, K.CSA, K.HCA, K.CSA_HCA])
    cfg = cfg_of(w)
    total = K.required_bytes(cfg)
    p = K.Pool(cfg)
    lo = p.layout()
    assert lo["total_bytes"] == total and lo["csa_per_block"] == 32
    vs = {K.F32: 4, K.BF16: 2, K.FP8_E4M3: 1}[cache]
    assert lo["entry_bytes"] == 2 * 2048 * vs + (16 if cache == K.FP8_E4M3 else 0)
    assert lo["entry_bytes"] % 16 == 0 and lo["idx_entry_bytes"] % 16 == 0
    spans = [(lo["table_offset"], lo["table_offset"] + 4 * 8 * 32), (lo["error_offset"], lo["error_offset"] + 4)]
    for l in range(4):
        d = p.layout(l)
        nb = cfg.max_blocks + cfg.max_requests
        kind = d["kind"]
        for part in ("csa", "idx", "hca"):
            present = d[f"{part}_offset"] >= 0
            assert present == (kind in ((K.CSA, K.CSA_HCA) if part != "hca" else (K.HCA, K.CSA_HCA)))
            if present:
                assert d[f"{part}_offset"] % 256 == 0 and d[f"{part}_block_bytes"] % 16 == 0
                spans.append((d[f"{part}_offset"], d[f"{part}_offset"] + nb * d[f"{part}_block_bytes"]))
            else:
                assert d[f"{part}_block_bytes"] == 0
        if kind in (K.CSA, K.CSA_HCA):
            assert d["csa_block_bytes"] == 32 * lo["entry_bytes"]
            assert d["idx_block_bytes"] >= 32 * lo["idx_entry_bytes"]
            assert (d["idx_scale_offset"] == 32 * lo["idx_entry_bytes"]) == (cache == K.FP8_E4M3)
        if kind in (K.HCA, K.CSA_HCA):
            assert d["hca_block_bytes"] == lo["entry_bytes"]
        for key in ("ring_offset", "acc_offset"):
            assert d[key] % 256 == 0
        assert d["ring_request_bytes"] % 256 == 0
        spans.append((d["ring_offset"], d["ring_offset"] + 8 * d["ring_request_bytes"]))
        spans.append((d["acc_offset"], d["acc_offset"] + 8 * d["acc_request_bytes"]))
    spans = sorted(s for s in spans if s[1] > s[0])
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= total


def both(w, max_requests=6, max_blocks=24, mbpr=6):
    o = H.make_oracle(w, max_requests, max_blocks, mbpr)
    p = K.Pool(cfg_of(w, max_requests=max_requests, max_blocks=max_blocks, max_blocks_per_request=mbpr,
                      max_batch=max_requests))
    return o, p


def same_state(o, p, reqs):
    for r in reqs:
        rc1, i1, ids1 = o.request_info(r)
        rc2, i2, ids2 = p.request_info(r)
        assert rc1 == rc2
        if rc1 == 0:
            assert i1 == i2 and ids1.tolist() == ids2.tolist()
    for b in range(24):
        assert o.block_refcount(b) == p.block_refcount(b)
    assert o.free_block_count() == p.free_block_count()


def test_host_bookkeeping_matches_oracle_under_random_traffic():
    w = base_workload(heads=4, head_dim=64, idx_heads=1, idx_dim=16, m_prime=16, n_win=32)
    o, p = both(w)
    rng = np.random.default_rng(12)
    live = []
    HD, XD = 256, 16
    for step in range(300):
        op = rng.integers(0, 10)
        if op < 2:
            rc1, r1 = o.alloc_request()
            try:
                r2 = p.alloc_request()
                rc2 = 0
            except K.KvpoolError as e:
                rc2, r2 = e.code, None
            assert rc1 == rc2
            if rc1 == 0:
                assert r1 == r2
                live.append(r1)
        elif op < 3 and live:
            r = live.pop(rng.integers(0, len(live)))
            assert o.free_request(r) == 0
            p.free_request(r)
        elif op < 4 and len(live) >= 2:
            src, dst = rng.choice(live, 2, replace=False)
            n_tok = int(rng.integers(0, 4)) * 16
            win = np.zeros((1, min(max(n_tok, 1), 32), HD), np.float32)
            rc1 = o.share_prefix(int(dst), int(src), n_tok, win, win)
            rc2 = p.share_prefix(int(dst), int(src), n_tok, None, None, stream=0, check=False)
            assert rc1 == rc2
        elif op < 5 and len(live) >= 2:  # a prefix image of src restored into dst
            src, dst = (int(x) for x in rng.choice(live, 2, replace=False))
            n_tok = int(rng.integers(0, 4)) * 16
            flags = int(rng.integers(0, 2))
            rc1, img = o.export_prefix(src, n_tok, flags, cap=1 << 22)
            hdr = np.zeros(1 << 22, np.uint8)
            rc2 = p.export_prefix(src, n_tok, flags, out=hdr, stream=0, check=False)
            assert rc1 == rc2
            if rc1 == 0:
                assert hdr[:64].tobytes() == img[:64].tobytes()  # the library's header is the oracle's
                win = np.zeros((1, min(n_tok, 32), HD), np.float32)
                rc1 = o.import_prefix(dst, img, win, win)
                rc2 = p.import_prefix(dst, img, stream=0, check=False)
                assert rc1 == rc2
        elif live:
            k = int(rng.integers(1, min(4, len(live)) + 1))
            reqs = [int(x) for x in rng.choice(live, k, replace=False)]
            if rng.random() < 0.1:
                reqs.append(reqs[0])  # duplicate -> refused by both
            counts = [int(x) for x in rng.integers(0, 40, len(reqs))]
            T = sum(counts)
            z = np.zeros((1, T, HD), np.float32)
            rc1 = o.append(reqs, counts, z, z, np.zeros((1, T, XD), np.float32))
            rc2 = p.append(reqs, counts, None, None, None, stream=0, check=False)
            assert rc1 == rc2
        same_state(o, p, range(6))


def test_error_codes_match_oracle():
    w = base_workload(m_prime=16, n_win=16, heads=4, head_dim=64, idx_dim=16)
    o, p = both(w, max_requests=3, max_blocks=3, mbpr=2)
    r = [p.alloc_request() for _ in range(3)]
    assert [o.alloc_request()[1] for _ in range(3)] == r
    with pytest.raises(K.KvpoolError) as e:
        p.alloc_request()
    assert e.value.code == o.alloc_request()[0] == K.ERR_OUT_OF_REQUESTS
    z = lambda T: np.zeros((1, T, 256), np.float32)
    zi = lambda T: np.zeros((1, T, 16), np.float32)
    for reqs, counts in [([0, 1], [16, 16]), ([0, 1, 2], [16, 16, 16]), ([0], [40]), ([0, 0], [1, 1]),
                         ([5], [1]), ([0], [-1]), ([2], [32])]:
        T = sum(max(c, 0) for c in counts)
        rc1 = o.append(reqs, counts, z(T), z(T), zi(T))
        rc2 = p.append(reqs, counts, None, None, None, stream=0, check=False)
        assert rc1 == rc2, (reqs, counts, rc1, rc2)
        same_state(o, p, range(3))
    win = np.zeros((1, 16, 256), np.float32)
    for dst, src, n in [(1, 0, 16), (2, 0, 8), (2, 0, 48), (2, 2, 16), (2, 7, 16), (2, 0, 0)]:
        assert o.share_prefix(dst, src, n, win, win) == p.share_prefix(dst, src, n, None, None, stream=0,
                                                                       check=False)
        same_state(o, p, range(3))
    for r_ in (0, 1, 2):
        assert o.free_request(r_) == p.L.kvpool_free_request(p.h, r_)
    assert o.free_request(1) == p.L.kvpool_free_request(p.h, 1) == K.ERR_BAD_REQUEST
    same_state(o, p, range(3))


@pytest.mark.parametrize("kw", [dict(), dict(cache_dtype=K.BF16, in_dtype=K.BF16),
                                dict(cache_dtype=K.FP8_E4M3, in_dtype=K.BF16, idx_dim=32),
                                dict(cache_dtype=K.FP8_E4M3, in_dtype=K.BF16, idx_fp4=1, idx_dim=32),
                                dict(n_layers=3, layer_kinds=[K.SWA_ONLY, K.CSA, K.HCA], n_win=256),
                                dict(idx_per_token=1),
                                dict(cache_dtype=K.FP8_E4M3, in_dtype=K.BF16, idx_dim=32, idx_per_token=1),
                                dict(cache_dtype=K.FP8_E4M3, in_dtype=K.BF16, idx_fp4=1, idx_dim=32, idx_per_token=1)])
def test_image_header_and_sizes_match_oracle(kw):
    """The library's config fingerprint, image sizes and image header equal
    the oracle's (both written from the documented layout, independently),
    with per-entry and per-token indexer keys."""
    fp4 = kw.pop("idx_fp4", 0)
    pt = kw.pop("idx_per_token", 0)
    w = base_workload(**kw)
    w["idx_fp4"] = fp4
    w["idx_per_token"] = pt
    o = H.make_oracle(w, 4, 16, 8)
    p = K.Pool(cfg_of(w, max_requests=4, max_blocks=16, max_blocks_per_request=8, idx_fp4=fp4, idx_per_token=pt))
    if pt:  # the block's indexer part is m runs of csa_per_block keys
        d = p.layout(0)
        run = d["csa_per_block"] * d["idx_entry_bytes"] + (64 if w["cache_dtype"] == K.FP8_E4M3 else 0)
        assert d["idx_block_bytes"] == w["m"] * run
    assert p.fingerprint() == o.fingerprint()
    for n in (0, 64, 128, 384, 1024):
        for f in (0, K.IMAGE_WINDOW):
            assert p.image_bytes(n, f) == o.image_bytes(n, f)
    r = p.alloc_request()
    assert o.alloc_request()[1] == r
    k, v, x = H.tokens(w, [r], [0], [300])
    assert o.append([r], [300], k, v, x) == 0
    p.append([r], [300], None, None, None, stream=0)
    for n, f in ((256, 0), (128, 0)):
        rc, img = o.export_prefix(r, n, f)
        hdr = np.zeros(img.size, np.uint8)
        p.export_prefix(r, n, f, out=hdr, stream=0)
        assert hdr[:64].tobytes() == img[:64].tobytes()
    for n, f, code in ((256, K.IMAGE_WINDOW, K.ERR_NOT_SHAREABLE), (320, 0, K.ERR_NOT_SHAREABLE),
                       (100, 0, K.ERR_NOT_SHAREABLE), (128, 2, K.ERR_INVALID_ARG)):
        hdr = np.zeros(1 << 20, np.uint8)
        assert p.export_prefix(r, n, f, out=hdr, stream=0, check=False) == code
    small = np.zeros(64, np.uint8)
    assert p.export_prefix(r, 128, 0, out=small, stream=0, check=False) == K.ERR_INVALID_ARG  # capacity


def test_image_import_refusals_match_oracle():
    w = base_workload(m_prime=16, n_win=16, heads=4, head_dim=64, idx_dim=16)
    o, p = both(w, max_requests=4, max_blocks=6, mbpr=3)
    r = [p.alloc_request() for _ in range(4)]
    assert [o.alloc_request()[1] for _ in range(4)] == r
    z = lambda T: np.zeros((1, T, 256), np.float32)
    zi = lambda T: np.zeros((1, T, 16), np.float32)
    assert o.append([0], [48], z(48), z(48), zi(48)) == 0
    p.append([0], [48], None, None, None, stream=0)
    rc, img = o.export_prefix(0, 48, K.IMAGE_WINDOW)
    win = z(16)
    for bad_at in (0, 4, 8, 16, 24, 48):  # magic, version, fingerprint, n_tokens, n_blocks, total
        bad = img.copy()
        bad[bad_at] ^= 1
        assert o.import_prefix(1, bad, win, win) == p.import_prefix(1, bad, stream=0, check=False) == \
            K.ERR_BAD_IMAGE
    assert o.import_prefix(1, img[:-16], win, win) == p.import_prefix(1, img[:-16], stream=0, check=False) == \
        K.ERR_BAD_IMAGE
    assert o.import_prefix(0, img, win, win) == p.import_prefix(0, img, stream=0, check=False) == \
        K.ERR_NOT_SHAREABLE
    assert o.import_prefix(1, img, win, win) == p.import_prefix(1, img, stream=0, check=False) == 0
    same_state(o, p, range(4))
    assert o.import_prefix(2, img, win, win) == p.import_prefix(2, img, stream=0, check=False) == \
        K.ERR_OUT_OF_BLOCKS
    same_state(o, p, range(4))
    o2, p2 = both(w, max_requests=2, max_blocks=6, mbpr=2)
    assert o2.alloc_request()[1] == p2.alloc_request()
    assert o2.import_prefix(0, img, win, win) == p2.import_prefix(0, img, stream=0, check=False) == \
        K.ERR_CAPACITY


def test_hisparse_bookkeeping_matches_oracle_under_random_traffic():
    """GPU and host slots of sealed blocks (smallest free at seal, restore,
    offload and fetch; returned when a block is freed) and every refusal
    equal the oracle's."""
    w = base_workload(heads=4, head_dim=64, idx_heads=1, idx_dim=16, m_prime=16, n_win=32)
    w.update(csa_hot_slots=14, csa_host_slots=12)
    o = H.make_oracle(w, 6, 24, 8)
    p = K.Pool(cfg_of(w, max_requests=6, max_blocks=24, max_blocks_per_request=8, max_batch=6, csa_hot_slots=14,
                      csa_host_slots=12))
    rng = np.random.default_rng(21)
    live = []
    HD = 256
    for step in range(400):
        op = rng.integers(0, 12)
        if op < 2:
            rc1, r1 = o.alloc_request()
            try:
                rc2, r2 = 0, p.alloc_request()
            except K.KvpoolError as e:
                rc2, r2 = e.code, None
            assert rc1 == rc2
            if rc1 == 0:
                assert r1 == r2
                live.append(r1)
        elif op < 3 and live:
            r = live.pop(rng.integers(0, len(live)))
            assert o.free_request(r) == 0
            p.free_request(r)
        elif op < 4 and len(live) >= 2:
            src, dst = (int(x) for x in rng.choice(live, 2, replace=False))
            n_tok = int(rng.integers(0, 4)) * 16
            rc1, img = o.export_prefix(src, n_tok, 0, cap=1 << 22)
            if rc1 == 0:
                win = np.zeros((1, min(n_tok, 32), HD), np.float32)
                assert o.import_prefix(dst, img, win, win) == p.import_prefix(dst, img, stream=0, check=False)
        elif op < 6:  # offload or fetch some live blocks (sometimes refused)
            ids = [b for b in range(24) if o.block_location(b)[0] == 0]
            if ids:
                pick = [int(x) for x in rng.choice(ids, min(len(ids), int(rng.integers(1, 5))), replace=False)]
                if rng.random() < 0.1:
                    pick.append(pick[0])  # repeated -> refused by both
                if op == 4:
                    assert o.offload(pick) == p.offload(pick, stream=0, check=False)
                else:
                    assert o.fetch(pick) == p.fetch(pick, stream=0, check=False)
        elif live:
            k = int(rng.integers(1, min(3, len(live)) + 1))
            reqs = [int(x) for x in rng.choice(live, k, replace=False)]
            counts = [int(x) for x in rng.integers(0, 40, len(reqs))]
            T = sum(counts)
            z = np.zeros((1, T, HD), np.float32)
            assert o.append(reqs, counts, z, z, np.zeros((1, T, 16), np.float32)) == \
                p.append(reqs, counts, None, None, None, stream=0, check=False)
        for b in range(24):
            rc1, l1, _ = o.block_location(b)
            rc2, l2 = p.block_location(b)
            assert rc1 == rc2 and (rc1 != 0 or l1 == l2), (step, b, rc1, rc2, l1, l2)
        assert o.free_block_count() == p.free_block_count()


def test_hisparse_refusals():
    w = base_workload(m_prime=16, n_win=16, heads=4, head_dim=64, idx_dim=16)
    for hot, host in ((-1, 0), (0, 4), (25, 0)):
        cfg = cfg_of(w, max_blocks=24, csa_hot_slots=hot, csa_host_slots=host)
        assert K.required_bytes(cfg) == 0
    p = K.Pool(cfg_of(w, max_blocks=24))
    assert p.offload([0], stream=0, check=False) == K.ERR_INVALID_ARG  # HiSparse off
    assert p.set_host_pool(np.zeros(64, np.uint8), check=False) == K.ERR_INVALID_ARG
    p = K.Pool(cfg_of(w, max_blocks=24, csa_hot_slots=8, csa_host_slots=4))
    lay = p.layout(0)
    assert p.host_slot_bytes() == lay["csa_block_bytes"] == 4 * 2048  # 4 CSA entries of 2 x 256 fp32
    assert lay["csa_staging_base"] == 8 and lay["csa_hot_slots"] == 8
    assert lay["host_slot_bytes"] == lay["csa_block_bytes"] and lay["csa_host_offset"] == 0
    assert p.set_host_pool(np.zeros(16, np.uint8), check=False) == K.ERR_INVALID_ARG  # too small


def test_topk_static_wrapper_refuses_tensors_the_kernels_cannot_take():
    # the binding checks shapes, types and devices before calling the library
    import torch
    s = torch.zeros((2, 8), dtype=torch.float32)  # host memory
    out = torch.zeros((2, 3), dtype=torch.int32)
    with pytest.raises(ValueError):
        K.topk_static(s, 3, out)
    with pytest.raises(ValueError):
        K.topk_static(torch.zeros(8, dtype=torch.float32), 3, out)  # not 2-D
    with pytest.raises(ValueError):
        K.topk_static(s.double(), 3, out)
