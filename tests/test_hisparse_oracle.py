"""Pins of the oracle's HiSparse placement ("V4 KV Layout" ESS / HiSparse
table: inactive C4 entries of the Classical pool move off the GPU; "Why does
V4 split pools?" s1 and s3.2: only full, immutable blocks move, the SWA
window stays resident).

Checked against brute force written here: the activity stamps against the
top-k index sets the oracle returns, the slot allocators against the
smallest-free rule on a scripted sequence, the inactive set against its
definition, and placement against the invariant that it never changes a
value (an offloading pool and a plain one give the same outputs and entries).
"""
import numpy as np
import pytest

import oracle as O
from tests import harness as H
from tests.test_oracle_pins import append_tokens, small_cfg


def pair(**kw):
    cfg = small_cfg(cache_dtype=O.BF16, in_dtype=O.BF16, **kw)
    plain = H.make_oracle(cfg, 4, 32, 16)
    hs = H.make_oracle(dict(cfg, csa_hot_slots=10, csa_host_slots=32), 4, 32, 16)
    return cfg, plain, hs


def test_config_refusals():
    cfg = small_cfg()
    with pytest.raises(ValueError):
        H.make_oracle(dict(cfg, csa_hot_slots=0, csa_host_slots=4), 2, 8, 8)  # host slots need HiSparse
    with pytest.raises(ValueError):
        H.make_oracle(dict(cfg, csa_hot_slots=-1), 2, 8, 8)
    o = H.make_oracle(cfg, 2, 8, 8)
    _, a = o.alloc_request()
    assert append_tokens(o, cfg, [a], [0], [40]) == O.OK
    assert o.block_location(0)[1:] == (0, 0)  # without HiSparse a block's entries stay with it
    assert o.offload([0]) == O.ERR_INVALID_ARG and o.fetch([0]) == O.ERR_INVALID_ARG


def test_slot_allocators_take_the_smallest_free_slot():
    cfg = small_cfg(cache_dtype=O.BF16, in_dtype=O.BF16)
    o = H.make_oracle(dict(cfg, csa_hot_slots=4, csa_host_slots=3), 4, 16, 8)
    _, a = o.alloc_request()
    _, b = o.alloc_request()
    assert append_tokens(o, cfg, [a], [0], [64]) == O.OK  # blocks 0-3 -> hot 0-3
    assert [o.block_location(i)[1] for i in range(4)] == [0, 1, 2, 3]
    info = o.request_info(a)[1]
    assert append_tokens(o, cfg, [b], [0], [16], wids=[1]) == O.ERR_OUT_OF_BLOCKS  # no hot slot
    assert o.request_info(a)[1] == info and o.free_block_count() == 12
    assert o.offload([2, 0]) == O.OK  # host slots 0, 1 in the given order
    assert [o.block_location(i)[1] for i in range(4)] == [-2, 1, -1, 3]
    assert append_tokens(o, cfg, [b], [0], [40], wids=[1]) == O.OK  # blocks 4, 5 -> hot 0, 2
    assert [o.block_location(i)[1] for i in (4, 5)] == [0, 2]
    assert o.fetch([0]) == O.ERR_OUT_OF_BLOCKS  # every hot slot is taken
    assert o.offload([1, 3, 4]) == O.ERR_OUT_OF_BLOCKS  # only one host slot left
    assert o.offload([1, 1]) == O.ERR_INVALID_ARG  # repeated
    assert o.offload([0]) == O.ERR_INVALID_ARG  # already offloaded
    assert o.offload([9]) == O.ERR_INVALID_ARG  # free block
    assert o.fetch([1]) == O.ERR_INVALID_ARG  # resident
    assert [o.block_location(i)[1] for i in range(6)] == [-2, 1, -1, 3, 0, 2]
    assert o.offload([5]) == O.OK and o.block_location(5)[1] == -3
    assert o.fetch([0]) == O.OK and o.block_location(0)[1] == 2  # the slot block 5 left
    assert o.free_request(a) == O.OK  # blocks 0-3: hot 2, 1, 3 and host 0 return
    assert o.fetch([5]) == O.OK and o.block_location(5)[1] == 1
    _, c = o.alloc_request()
    assert append_tokens(o, cfg, [c], [0], [32], wids=[2]) == O.OK  # ids 0, 1 -> hot 2, 3
    assert [o.block_location(i)[1] for i in (0, 1)] == [2, 3]


def _expected_stamps(o, cfg, reqs, tk, stamps, epoch):
    CB = cfg["m_prime"] // cfg["m"]
    for r, row in zip(reqs, tk):
        ids = o.request_info(r)[2]
        for e in row:
            if e >= 0 and e // CB < len(ids):
                stamps[int(ids[e // CB])] = epoch


def test_activity_stamps_are_the_blocks_of_the_selected_entries():
    cfg = small_cfg(cache_dtype=O.BF16, in_dtype=O.BF16, n_layers=3, layer_kinds=[O.CSA, O.HCA, O.CSA_HCA])
    o = H.make_oracle(dict(cfg, csa_hot_slots=30, csa_host_slots=8), 4, 32, 16)
    reqs = [o.alloc_request()[1] for _ in range(3)]
    assert append_tokens(o, cfg, reqs, [0, 0, 0], [70, 150, 33]) == O.OK
    stamps = {}
    for r in reqs:  # sealing stamps the epoch of the time: 0
        for b in o.request_info(r)[2]:
            stamps[int(b)] = 0
    L = [70, 150, 33]
    for step in range(9):
        layer = step % 3
        q, qi = H.queries(cfg, layer, reqs, step)
        rc, out, tk = o.decode_attend(layer, reqs, q, qi, 5)
        assert rc == O.OK and o.epoch() == step + 1
        if cfg["layer_kinds"][layer] != O.HCA:  # HCA layers read every HCA entry: no CSA selection
            _expected_stamps(o, cfg, reqs, tk, stamps, step + 1)
        if step == 4:
            assert append_tokens(o, cfg, reqs, L, [1, 20, 40]) == O.OK  # seals stamp epoch 5
            for r, l0, n in zip(reqs, L, [1, 20, 40]):
                ids = o.request_info(r)[2]
                for s in range(l0 // 16, (l0 + n) // 16):
                    stamps[int(ids[s])] = 5
            L = [a + b for a, b in zip(L, [1, 20, 40])]
        got = {b: o.block_location(b)[2] for b in stamps}
        assert got == stamps
    # the inactive set: resident blocks idle for at least `idle` epochs
    for idle in (0, 1, 3, 5, 20):
        want = sorted(b for b, t in stamps.items() if o.epoch() - t >= idle)
        assert o.inactive_blocks(idle).tolist() == want
    off = o.inactive_blocks(4)[:3].tolist()
    assert o.offload(off) == O.OK
    assert all(b not in o.inactive_blocks(0).tolist() for b in off)  # offloaded blocks are not listed
    assert o.fetch(off[:1]) == O.OK and o.block_location(off[0])[2] == o.epoch()  # a fetch stamps


def test_placement_never_changes_a_value():
    """A pool that offloads every resident block between steps and fetches
    one back gives exactly the outputs, top-k sets and entries of a pool
    without HiSparse."""
    cfg, plain, hs = pair()
    reqs = [plain.alloc_request()[1] for _ in range(3)]
    assert [hs.alloc_request()[1] for _ in range(3)] == reqs
    L = [0, 0, 0]
    rng = np.random.default_rng(4)
    for step in range(8):
        n = [int(x) for x in rng.integers(1, 30, 3)]
        for o in (plain, hs):
            assert append_tokens(o, cfg, reqs, L, n) == O.OK
        L = [a + b for a, b in zip(L, n)]
        q, qi = H.queries(cfg, 0, reqs, step)
        r1 = plain.decode_attend(0, reqs, q, qi, 6)
        r2 = hs.decode_attend(0, reqs, q, qi, 6)
        assert r1[0] == r2[0] == O.OK
        assert np.array_equal(r1[1], r2[1]) and np.array_equal(r1[2], r2[2])
        assert hs.offload(hs.inactive_blocks(0).tolist()) == O.OK  # every resident block
        back = [b for b in range(32) if hs.block_location(b)[0] == O.OK and hs.block_location(b)[1] < 0][:1]
        assert hs.fetch(back) == O.OK
    for r in reqs:
        info = plain.request_info(r)[1]
        assert info == hs.request_info(r)[1]
        for e in range(info["n_csa"]):
            for kind in (1, 3):
                assert np.array_equal(plain.request_entry(0, r, kind, e)[1], hs.request_entry(0, r, kind, e)[1])
    assert any(hs.block_location(b)[0] == O.OK and hs.block_location(b)[1] < 0 for b in range(32))


def test_images_and_sharing_with_offloaded_blocks():
    """An image does not depend on where the CSA entries are; a restore into
    a HiSparse pool needs hot slots for its blocks; shared blocks move once."""
    cfg, plain, hs = pair()
    a = plain.alloc_request()[1]
    assert hs.alloc_request()[1] == a
    for o in (plain, hs):
        assert append_tokens(o, cfg, [a], [0], [96]) == O.OK  # 6 blocks
    assert hs.offload([1, 3, 4]) == O.OK
    i1, i2 = plain.export_prefix(a, 96, O.IMAGE_WINDOW), hs.export_prefix(a, 96, O.IMAGE_WINDOW)
    assert i1[0] == i2[0] == O.OK and i1[1].size > 0
    # the fingerprint covers the layout, not the placement capacities
    assert np.array_equal(i1[1], i2[1])
    b = hs.alloc_request()[1]
    assert hs.share_prefix(b, a, 64, *H.tokens(cfg, [a], [32], [32])[:2]) == O.OK
    assert [hs.block_location(x)[1] for x in range(4)] == [0, -1, 2, -2]
    assert hs.free_request(a) == O.OK  # blocks 0-3 stay (shared), 4-5 return their slots
    assert hs.block_location(4)[0] == O.ERR_INVALID_ARG
    c = hs.alloc_request()[1]
    assert hs.import_prefix(c, i1[1]) == O.OK  # 6 blocks -> the free hot slots 1, 3..7
    ids = hs.request_info(c)[2].tolist()
    assert [hs.block_location(x)[1] for x in ids] == [1, 3, 4, 5, 6, 7]
    d = hs.alloc_request()[1]
    assert hs.import_prefix(d, i1[1]) == O.ERR_OUT_OF_BLOCKS  # 2 hot slots left for 6 blocks
