"""Pins of the oracle's prefix images: the sealed blocks of a request prefix
serialized to host memory and restored into another request, with or
without the SWA window ("Ch 12 Inference framework: heterogeneous KV
scheduling" s3 disk-resident KV and s3.1 SWA policies; "V4 disk prefix
cache": Full / Periodic checkpointing / Zero SWA).

The checks come from outside the image code: published FNV-1a test vectors,
the byte layout recomputed here from the config, the oracle's separate entry
and window accessors, and the invariant the pages' policies rest on: a
restored request (plus, for a checkpoint, the replayed gap) is the same
request as the one that never left.
"""
import struct

import numpy as np
import pytest

import oracle as O
from tests import harness as H
from tests.test_oracle_pins import append_tokens, oracle_for, small_cfg


def test_fnv1a64_published_vectors():
    # the FNV authors' test vectors for FNV-1a, 64 bit
    assert O.fnv1a64(b"") == 0xCBF29CE484222325
    assert O.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert O.fnv1a64(b"foobar") == 0x85944171F73967E8


def _record(cfg, gates):
    """The canonical config record, assembled here from the documented field list."""
    g_csa, g_hca, g_idx = (np.asarray(g, np.float32) for g in gates)
    b = struct.pack("<11i", cfg["m"], cfg["m_prime"], cfg["n_win"], cfg["heads"], cfg["head_dim"],
                    cfg["idx_heads"], cfg["idx_dim"], cfg["in_dtype"], cfg["cache_dtype"], cfg.get("idx_fp4", 0),
                    cfg["n_layers"])
    for l, k in enumerate(cfg["layer_kinds"]):
        b += struct.pack("<i", k)
        if k in (O.CSA, O.CSA_HCA):
            b += g_csa[l].astype("<f4").tobytes() + g_idx[l].astype("<f4").tobytes()
        if k in (O.HCA, O.CSA_HCA):
            b += g_hca[l].astype("<f4").tobytes()
    return b


@pytest.mark.parametrize("kinds", [[O.CSA_HCA], [O.SWA_ONLY, O.CSA, O.HCA]])
def test_fingerprint_is_fnv1a_of_the_config_record(kinds):
    cfg = small_cfg(n_layers=len(kinds), layer_kinds=kinds, cache_dtype=O.FP8, in_dtype=O.BF16, idx_dim=8)
    gates = H.gates(cfg)
    o = oracle_for(cfg)
    assert o.fingerprint() == O.fnv1a64(_record(cfg, gates))
    # capacities do not enter it; a gate logit or the indexer format does
    assert oracle_for(cfg, max_requests=7, max_blocks=99, mbpr=33).fingerprint() == o.fingerprint()
    g2 = [g.copy() for g in gates]
    g2[1][-1, 0, 0] += 1.0 if kinds[-1] in (O.HCA, O.CSA_HCA) else 0.0
    g2[0][-1, 0, 0] += 0.0 if kinds[-1] in (O.HCA, O.CSA_HCA) else 1.0
    assert oracle_for(cfg, gates=g2).fingerprint() != o.fingerprint()
    assert oracle_for(dict(cfg, idx_fp4=1, idx_dim=16)).fingerprint() != o.fingerprint()


def _sizes(cfg):
    HD, XD = cfg["heads"] * cfg["head_dim"], cfg["idx_heads"] * cfg["idx_dim"]
    vs = {O.F32: 4, O.BF16: 2, O.FP8: 1}[cfg["cache_dtype"]]
    E = 2 * HD * vs + (16 if cfg["cache_dtype"] == O.FP8 else 0)
    CB = cfg["m_prime"] // cfg["m"]
    idx_dtype = O.FP4 if cfg.get("idx_fp4") else cfg["cache_dtype"]
    xs = XD // 2 if idx_dtype == O.FP4 else XD * {O.F32: 4, O.BF16: 2, O.FP8: 1}[idx_dtype]
    X = CB * xs + ((2 * CB + 15) // 16 * 16 if idx_dtype in (O.FP8, O.FP4) else 0)
    return E, X, CB, xs


CASES = [
    dict(cache_dtype=O.F32, in_dtype=O.F32),
    dict(cache_dtype=O.BF16, in_dtype=O.BF16),
    dict(cache_dtype=O.FP8, in_dtype=O.BF16, idx_dim=8),
    dict(cache_dtype=O.FP8, in_dtype=O.BF16, idx_fp4=1, idx_dim=16),
    dict(cache_dtype=O.BF16, in_dtype=O.BF16, n_layers=3, layer_kinds=[O.SWA_ONLY, O.CSA, O.HCA]),
]


def _name(c):
    return "-".join(f"{k}{v}" for k, v in c.items() if k != "layer_kinds")


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_image_layout_matches_the_entry_accessors(case):
    """Every byte of an image is where the documented layout puts it: checked
    against the oracle's block-entry and window accessors."""
    cfg = small_cfg(**case)
    o = oracle_for(cfg)
    _, a = o.alloc_request()
    L = 80  # 5 sealed blocks of 16
    assert append_tokens(o, cfg, [a], [0], [L]) == O.OK
    _, info, ids = o.request_info(a)
    E, X, CB, xs = _sizes(cfg)
    nb, w = L // 16, min(L, cfg["n_win"])
    for flags in (0, O.IMAGE_WINDOW):
        rc, img = o.export_prefix(a, L, flags)
        assert rc == O.OK
        per_block = sum((CB * E + X if k in (O.CSA, O.CSA_HCA) else 0) + (E if k in (O.HCA, O.CSA_HCA) else 0)
                        for k in cfg["layer_kinds"])
        wb = w * E * cfg["n_layers"] if flags else 0
        total = 64 + nb * per_block + wb
        assert img.size == total == o.image_bytes(L, flags)
        magic, ver, fp, n_tok, nbh, wh, bb, wbh, tot, zero = struct.unpack("<IIQqiiQQQQ", img[:64].tobytes())
        assert (magic, ver, fp, n_tok, nbh, wh) == (0x4950564B, 1, o.fingerprint(), L, nb, w if flags else 0)
        assert (bb, wbh, tot, zero) == (nb * per_block, wb, total, 0)

        def rec(code, sc):
            r = code.tobytes()
            if cfg["cache_dtype"] == O.FP8:
                r += struct.pack("<HH", int(sc[0]), int(sc[1])) + bytes(12)
            return r

        off = 64
        for l, k in enumerate(cfg["layer_kinds"]):
            if k in (O.CSA, O.CSA_HCA):
                for b in range(nb):
                    for e in range(CB):
                        rc, c, s = o.block_entry(l, int(ids[b]), 1, e)
                        assert img[off:off + E].tobytes() == rec(c, s)
                        off += E
                for b in range(nb):
                    part = img[off:off + X]
                    for e in range(CB):
                        rc, c, s = o.block_entry(l, int(ids[b]), 3, e)
                        got = bytes(part[(j // 16 * CB + e) * 16 + j % 16] for j in range(xs))
                        assert got == c.tobytes()
                        if X > CB * xs:
                            assert part[CB * xs + 2 * e:CB * xs + 2 * e + 2].tobytes() == struct.pack("<H", int(s[0]))
                    assert not part[CB * xs + 2 * CB:].any() if X > CB * xs else True
                    off += X
            if k in (O.HCA, O.CSA_HCA):
                for b in range(nb):
                    rc, c, s = o.block_entry(l, int(ids[b]), 2, 0)
                    assert img[off:off + E].tobytes() == rec(c, s)
                    off += E
        if flags:
            for l in range(cfg["n_layers"]):
                for pos in range(L - w, L):
                    rc, c, s = o.window_token(l, a, pos)
                    assert rc == O.OK and img[off:off + E].tobytes() == rec(c, s)
                    off += E
        assert off == total


def _request_state(o, cfg, r):
    """Everything observable about a request: info, every entry, the window."""
    _, info, _ = o.request_info(r)
    st = [tuple(sorted(info.items()))]
    for l, k in enumerate(cfg["layer_kinds"]):
        if k in (O.CSA, O.CSA_HCA):
            for e in range(info["n_csa"]):
                for kind in (1, 3):
                    rc, c, s = o.request_entry(l, r, kind, e)
                    st.append((l, kind, e, c.tobytes(), s.tobytes()))
        for pos in range(info["length"] - info["window"], info["length"]):
            rc, c, s = o.window_token(l, r, pos)
            st.append((l, "w", pos, c.tobytes(), s.tobytes()))
    return st


def _outputs(o, cfg, r, wid, step, top_k=6):
    outs = []
    for l in range(cfg["n_layers"]):
        q, qi = H.queries(cfg, l, [wid], step)
        rc, out, tk = o.decode_attend(l, [r], q, qi, top_k)
        assert rc == O.OK
        outs.append((out.copy(), tk.copy()))
    return outs


def _same_outputs(a, b):
    return all(np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1]) for x, y in zip(a, b))


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_restored_prefix_is_the_same_request(case):
    """Restore (window from the image) into another pool whose free ids differ:
    the restored request equals the original, entry for entry and output
    for output, and stays equal while both grow on the same tokens."""
    cfg = small_cfg(**case)
    A = oracle_for(cfg)
    _, a = A.alloc_request()
    assert append_tokens(A, cfg, [a], [0], [96]) == O.OK
    rc, img = A.export_prefix(a, 96, O.IMAGE_WINDOW)
    assert rc == O.OK
    B = oracle_for(cfg, max_blocks=40)
    _, other = B.alloc_request()
    assert append_tokens(B, cfg, [other], [0], [50], wids=[9]) == O.OK  # occupies ids 0..2
    _, b = B.alloc_request()
    assert B.import_prefix(b, img) == O.OK
    _, ib, ids_b = B.request_info(b)
    assert ids_b.tolist() == list(range(3, 9))  # smallest free ids, in image order
    assert all(B.block_refcount(int(i)) == 1 for i in ids_b)
    assert _request_state(A, cfg, a) == _request_state(B, cfg, b)
    assert _same_outputs(_outputs(A, cfg, a, a, 0), _outputs(B, cfg, b, a, 0))
    # both grow on request a's tokens (a partial block, then across a seal)
    for pos, n in ((96, 7), (103, 30)):
        assert append_tokens(A, cfg, [a], [pos], [n]) == O.OK
        assert append_tokens(B, cfg, [b], [pos], [n], wids=[a]) == O.OK
        assert _request_state(A, cfg, a) == _request_state(B, cfg, b)
        assert _same_outputs(_outputs(A, cfg, a, a, pos), _outputs(B, cfg, b, a, pos))
    # the restored blocks are the pool's own: freeing returns them
    free0 = B.free_block_count()
    assert B.free_request(b) == O.OK and B.free_block_count() == free0 + 8


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_zero_swa_restore_equals_full_restore_and_share_prefix(case):
    """Zero SWA ([P4]): the image holds no window and the caller gives the
    recomputed window tokens; the request equals the Full restore and the
    in-pool share_prefix of the same prefix."""
    cfg = small_cfg(**case)
    o = oracle_for(cfg, max_blocks=64)
    _, a = o.alloc_request()
    assert append_tokens(o, cfg, [a], [0], [70]) == O.OK
    P = 64
    rc, zero = o.export_prefix(a, P, 0)
    assert rc == O.OK
    assert o.export_prefix(a, P, O.IMAGE_WINDOW)[0] == O.ERR_NOT_SHAREABLE  # the window exists at L only
    w = min(P, cfg["n_win"])
    k, v, _ = H.tokens(cfg, [a], [P - w], [w])
    _, b = o.alloc_request()
    _, c = o.alloc_request()
    assert o.import_prefix(b, zero) == O.ERR_INVALID_ARG  # Zero SWA needs the window
    assert o.import_prefix(b, zero, k, v) == O.OK
    assert o.share_prefix(c, a, P, k, v) == O.OK
    sb, sc = _request_state(o, cfg, b), _request_state(o, cfg, c)
    assert sb == sc
    assert _same_outputs(_outputs(o, cfg, b, a, 3), _outputs(o, cfg, c, a, 3))
    # Full: a request whose length is P exports its window; restoring it equals b
    _, d = o.alloc_request()
    assert append_tokens(o, cfg, [d], [0], [P], wids=[a]) == O.OK
    rc, full = o.export_prefix(d, P, O.IMAGE_WINDOW)
    assert rc == O.OK and full.size == zero.size + w * _sizes(cfg)[0] * cfg["n_layers"]
    assert full[64 + 32:64 + 40].tobytes() == zero[64 + 32:64 + 40].tobytes()  # same block section size
    assert full[64:].tobytes()[:zero.size - 64] == zero[64:].tobytes()  # same blocks
    assert o.free_request(b) == O.OK
    _, e = o.alloc_request()
    assert o.import_prefix(e, full) == O.OK
    assert _request_state(o, cfg, e) == sc


@pytest.mark.parametrize("case", CASES[1:3], ids=_name)
def test_periodic_checkpoint_restore_and_replay_is_continuous(case):
    """Periodic checkpointing ([P3] s3.1, [P4]): a checkpoint every p tokens
    (blocks + window); after a restore the gap since the checkpoint is
    recomputed by replaying its tokens.  The result equals the request that
    ran continuously."""
    cfg = small_cfg(**case)
    p = 32  # checkpoint period (a multiple of the block length 16)
    o = oracle_for(cfg, max_blocks=64)
    _, a = o.alloc_request()
    ckpt, ckpt_at, L = None, None, 0
    for n in (13, 20, 9, 31, 5):  # appends of a serving loop
        # the policy: an append that reaches a multiple of p is split there
        # and the checkpoint (blocks + window) taken at that length
        while n > 0:
            step = min(n, (L // p + 1) * p - L)
            assert append_tokens(o, cfg, [a], [L], [step]) == O.OK
            L, n = L + step, n - step
            if L % p == 0:
                rc, ckpt = o.export_prefix(a, L, O.IMAGE_WINDOW)
                assert rc == O.OK
                ckpt_at = L
    assert ckpt_at == 64 and L == 78
    _, b = o.alloc_request()
    assert o.import_prefix(b, ckpt) == O.OK
    assert append_tokens(o, cfg, [b], [ckpt_at], [L - ckpt_at], wids=[a]) == O.OK  # replay the gap
    assert _request_state(o, cfg, a)[1:] == _request_state(o, cfg, b)[1:]
    assert o.request_info(a)[1] == o.request_info(b)[1]
    assert _same_outputs(_outputs(o, cfg, a, a, 5), _outputs(o, cfg, b, a, 5))


def test_image_refusals_leave_the_pool_unchanged():
    cfg = small_cfg(cache_dtype=O.BF16, in_dtype=O.BF16)
    o = oracle_for(cfg, max_blocks=8, mbpr=4)
    _, a = o.alloc_request()
    assert append_tokens(o, cfg, [a], [0], [70]) == O.OK  # 4 sealed blocks
    assert o.export_prefix(a, 24, 0)[0] == O.ERR_NOT_SHAREABLE  # not whole blocks
    assert o.export_prefix(a, 80, 0)[0] == O.ERR_NOT_SHAREABLE  # beyond the sealed blocks
    assert o.export_prefix(3, 16, 0)[0] == O.ERR_BAD_REQUEST
    assert o.export_prefix(a, 64, 0, cap=100)[0] == O.ERR_INVALID_ARG
    assert o.export_prefix(a, 64, 2)[0] == O.ERR_INVALID_ARG  # unknown flag
    rc, img = o.export_prefix(a, 64, 0)
    win = np.zeros((1, 32, 8), np.float32)
    _, c = o.alloc_request()
    assert append_tokens(o, cfg, [c], [0], [16], wids=[5]) == O.OK  # 3 blocks stay free
    _, b = o.alloc_request()
    free0 = o.free_block_count()
    snap = o.request_info(b)[1]
    bad = img.copy()
    bad[0] ^= 1
    assert o.import_prefix(b, bad, win, win) == O.ERR_BAD_IMAGE  # magic
    bad = img.copy()
    bad[8] ^= 1
    assert o.import_prefix(b, bad, win, win) == O.ERR_BAD_IMAGE  # fingerprint
    assert o.import_prefix(b, img[:-1], win, win) == O.ERR_BAD_IMAGE  # truncated
    other = oracle_for(dict(cfg, seed=12))
    _, x = other.alloc_request()
    assert other.import_prefix(x, img, win, win) == O.ERR_BAD_IMAGE  # other gates
    assert o.import_prefix(b, img, win, win) == O.ERR_OUT_OF_BLOCKS  # 4 needed, 3 free
    assert o.free_block_count() == free0 and o.request_info(b)[1] == snap
    assert o.import_prefix(a, img, win, win) == O.ERR_NOT_SHAREABLE  # not fresh
    # keys that are not whole 16-byte chunks have no image layout
    odd = oracle_for(small_cfg(cache_dtype=O.FP8, in_dtype=O.BF16))
    _, z = odd.alloc_request()
    assert append_tokens(odd, small_cfg(cache_dtype=O.FP8, in_dtype=O.BF16), [z], [0], [16]) == O.OK
    assert odd.image_bytes(16) == -1 and odd.export_prefix(z, 16, 0, cap=1 << 16)[0] == O.ERR_INVALID_ARG
    small = oracle_for(cfg, max_blocks=8, mbpr=2)
    _, y = small.alloc_request()
    assert small.import_prefix(y, img, win, win) == O.ERR_CAPACITY
