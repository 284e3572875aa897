"""Parity of prefix images on the GPU ("Ch 12 Inference framework:
heterogeneous KV scheduling" s3, s3.1; "V4 disk prefix cache"): the image
the CUDA path writes into page-locked host memory is byte-identical to the
oracle's; an image restored on the GPU (the oracle's or the GPU's own) gives
the oracle's request state bit for bit; a restored checkpoint grows exactly
like the request it was taken from, on the GPU bit for bit; Zero SWA takes
the caller's recomputed window."""
import numpy as np
import pytest
import torch

import oracle as O
from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import compare_request_state
from tests.test_gpu_parity import append_both, attend_both, make_pair

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_f32": dict(W.TINY, seed=31),
    "bf16": dict(W.DECODE_BATCH, seed=32),
    "fp8": dict(W.LONG_CONTEXT, seed=33),
    "fp8_fp4_indexer": dict(W.LONG_CONTEXT, seed=34, idx_fp4=1),
    "mixed_kinds": dict(W.MIXED_SERVING, n_win=256, seed=35),
}


def pinned(arr):
    t = torch.empty(arr.size, dtype=torch.uint8, pin_memory=True)
    t.numpy()[:] = arr
    return t


def gpu_image(g, slot, n, flags):
    img = g.pool.export_prefix(slot, n, flags)
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    return img.numpy()[:g.pool.image_bytes(n, flags)].copy()


def zero_swa_window(g, wid, n):
    w = min(n, g.w["n_win"])
    k, v, _ = H.tokens(g.w, [wid], [n - w], [w])
    gk, gv, _ = g.tokens([wid], [n - w], [w])
    return (k, v), (gk, gv)


@pytest.mark.parametrize("name", list(CASES))
def test_images_match_the_oracle_and_restore_bit_exactly(name):
    w = CASES[name]
    mp = w["m_prime"]
    o, g = make_pair(w, 8, 48, 12, 8, 128)
    s = [g.pool.alloc_request() for _ in range(3)]
    assert [o.alloc_request()[1] for _ in range(3)] == s
    # fragment the free ids: s0 seals 3 blocks, s1 2, s0 leaves, s2 takes 0-2 then 5-6
    append_both(o, g, [s[0], s[1]], [0, 1], [0, 0], [3 * mp + 5, 2 * mp + 9])
    o.free_request(s[0])
    g.pool.free_request(s[0])
    append_both(o, g, [s[2]], [2], [0], [5 * mp + 37])
    assert o.request_info(s[2])[2].tolist() == [0, 1, 2, 5, 6]
    # a checkpoint needs the length on a block boundary: s1 grows to 3 blocks exactly
    append_both(o, g, [s[1]], [1], [2 * mp + 9], [mp - 9])
    for slot, n, flags in ((s[2], 5 * mp, 0), (s[2], 2 * mp, 0), (s[1], 3 * mp, K.IMAGE_WINDOW)):
        rc, ref = o.export_prefix(slot, n, flags)
        assert rc == 0
        got = gpu_image(g, slot, n, flags)
        assert got.size == ref.size
        if not np.array_equal(got, ref):
            bad = np.nonzero(got != ref)[0]
            pytest.fail(f"image of {n} tokens differs at {bad.size} bytes, first {bad[:8].tolist()}")

    # restore: the oracle's Zero SWA image of s2 and the GPU's checkpoint of s1
    (k, v), (gk, gv) = zero_swa_window(g, 2, 5 * mp)
    rc, zimg = o.export_prefix(s[2], 5 * mp, 0)
    ckpt = gpu_image(g, s[1], 3 * mp, K.IMAGE_WINDOW)
    r = [g.pool.alloc_request() for _ in range(2)]
    assert [o.alloc_request()[1] for _ in range(2)] == r
    assert o.import_prefix(r[0], zimg, k, v) == 0
    g.pool.import_prefix(r[0], pinned(zimg), gk, gv)
    assert o.import_prefix(r[1], ckpt) == 0
    g.pool.import_prefix(r[1], pinned(ckpt))
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    for x in r:
        compare_request_state(g, o, x)
    # everyone grows on its source's tokens, across a seal, then decodes
    append_both(o, g, [s[1], s[2], r[0], r[1]], [1, 2, 2, 1], [3 * mp, 5 * mp + 37, 5 * mp, 3 * mp],
                [mp + 3, 1, mp + 40, mp + 3])
    for x in (s[1], r[0], r[1]):
        compare_request_state(g, o, x)
    for layer in range(g.nl):
        attend_both(o, g, layer, [s[1], r[1], r[0]], [1, 1, 2], 0, 128)
        # the restored checkpoint and its source are the same request: same bits
        out, tk = g.attend(layer, [s[1], r[1]], [1, 1], 1, 128)
        assert torch.equal(out[0], out[1]) and torch.equal(tk[0], tk[1])


def test_fragmented_ids_need_several_copy_launches():
    """70 blocks on alternate ids: export and import each take several
    launches (at most 64 copies and 64 table runs per launch)."""
    w = dict(W.DECODE_BATCH, seed=36)
    mp = w["m_prime"]
    o, g = make_pair(w, 4, 160, 80, 4, 128)
    a, b = g.pool.alloc_request(), g.pool.alloc_request()
    assert [o.alloc_request()[1] for _ in range(2)] == [a, b]
    for i in range(70):  # a seals even ids, b odd ids
        append_both(o, g, [a, b], [0, 1], [i * mp, i * mp], [mp, mp])
    assert o.request_info(a)[2].tolist() == list(range(0, 140, 2))
    n = 70 * mp
    rc, ref = o.export_prefix(a, n, K.IMAGE_WINDOW)
    got = gpu_image(g, a, n, K.IMAGE_WINDOW)
    assert np.array_equal(got, ref)
    o.free_request(b)
    g.pool.free_request(b)
    c = g.pool.alloc_request()
    assert o.alloc_request()[1] == c
    assert o.import_prefix(c, ref) == 0
    g.pool.import_prefix(c, pinned(got))
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    assert g.pool.request_info(c)[2].tolist() == list(range(1, 140, 2))
    compare_request_state(g, o, c, sample=64, rng=np.random.default_rng(0))
    append_both(o, g, [a, c], [0, 0], [n, n], [3, 3])
    attend_both(o, g, 0, [a, c], [0, 0], 0, 128)


def test_indexer_scale_padding_is_zero_in_the_image():
    """With m'/m = 4 CSA entries per block the 8 bytes of fp8 indexer
    scales are padded to 16: the export writes the padding as zeros whatever
    the arena holds there (append and export only)."""
    w = dict(W.TINY, m_prime=16, n_win=32, in_dtype=K.BF16, cache_dtype=K.FP8_E4M3, heads=4, head_dim=64,
             idx_heads=1, idx_dim=32, seed=37)
    o, g = make_pair(w, 2, 16, 8, 2, 16)
    d = g.pool.layout(0)
    assert d["idx_block_bytes"] - d["idx_scale_offset"] == 16  # 8 bytes of scales + 8 of padding
    n_ids = 16 + 2  # blocks + staging blocks
    g.arena[d["idx_offset"]:d["idx_offset"] + n_ids * d["idx_block_bytes"]].fill_(0xA5)  # never written there
    a = g.pool.alloc_request()
    assert o.alloc_request()[1] == a
    append_both(o, g, [a], [0], [0], [80])
    rc, ref = o.export_prefix(a, 80, K.IMAGE_WINDOW)
    got = gpu_image(g, a, 80, K.IMAGE_WINDOW)
    assert np.array_equal(got, ref)


def test_image_refusals_on_the_device():
    w = dict(W.DECODE_BATCH, seed=38)
    o, g = make_pair(w, 3, 8, 8, 3, 128)
    a = g.pool.alloc_request()
    g.append([a], [0], [0], [256])
    img = np.zeros(g.pool.image_bytes(256, 0), np.uint8)  # pageable host memory
    assert g.pool.export_prefix(a, 256, 0, out=img, check=False) == K.ERR_INVALID_ARG
    pin = g.pool.export_prefix(a, 256, 0)
    torch.cuda.synchronize()
    b = g.pool.alloc_request()
    assert g.pool.import_prefix(b, pin, check=False) == K.ERR_INVALID_ARG  # Zero SWA image needs a window
    gk, gv, _ = g.tokens([0], [128], [128])
    assert g.pool.import_prefix(b, pin[1:], gk, gv, check=False) in (K.ERR_BAD_IMAGE, K.ERR_INVALID_ARG)
    assert g.pool.free_block_count() == 6
    g.pool.import_prefix(b, pin, gk, gv)
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0 and g.pool.free_block_count() == 4
