"""HiSparse on the GPU ("V4 KV Layout" ESS / HiSparse table: inactive C4
entries move off the GPU): with sealed blocks' CSA entries offloaded to
page-locked host slots, decode outputs and top-k sets are bit-identical to a
pool that keeps everything resident (the attention reads offloaded entries
from host memory), and match the oracle within the cache dtype's tolerance;
locations, activity stamps and inactive sets equal the oracle's; prefix
images of requests with offloaded blocks are the oracle's."""
import numpy as np
import pytest
import torch

from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import GpuCase, check_out, compare_request_state

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": dict(W.DECODE_BATCH, seed=41),
    "fp8": dict(W.LONG_CONTEXT, seed=42),
    "fp8_fp4_indexer": dict(W.LONG_CONTEXT, seed=43, idx_fp4=1),
    "mixed_kinds": dict(W.MIXED_SERVING, n_win=256, seed=44),
}


def locations_match(o, g, max_blocks):
    for b in range(max_blocks):
        rc1, l1, _ = o.block_location(b)
        rc2, l2 = g.pool.block_location(b)
        assert rc1 == rc2 and (rc1 != 0 or l1 == l2), (b, rc1, rc2, l1, l2)


@pytest.mark.parametrize("name", list(CASES))
def test_offloaded_blocks_give_bit_identical_outputs(name):
    w = CASES[name]
    mp = w["m_prime"]
    hs = dict(w, csa_hot_slots=14, csa_host_slots=24)
    o = H.make_oracle(hs, 6, 32, 12)
    g = GpuCase(hs, 6, 32, 12, 6, 256)  # HiSparse pool
    ref = GpuCase(w, 6, 32, 12, 6, 256)  # everything resident
    slots = [g.pool.alloc_request() for _ in range(4)]
    assert [o.alloc_request()[1] for _ in range(4)] == slots == [ref.pool.alloc_request() for _ in range(4)]
    L = [0] * 4
    rng = np.random.default_rng(7)
    for rnd in range(6):
        counts = [int(x) for x in rng.integers(1, 2 * mp, 4)] if rnd < 4 else [1, 1, 1, 1]
        k, v, x = H.tokens(w, slots, L, counts)
        assert o.append(slots, counts, k, v, x) == 0
        g.append(slots, slots, L, counts)
        ref.append(slots, slots, L, counts)
        L = [a + b for a, b in zip(L, counts)]
        for layer in range(g.nl):
            q, qi = H.queries(w, layer, slots, rnd)
            rc, out_ref, tk_ref = o.decode_attend(layer, slots, q, qi, 256)
            assert rc == 0
            out_g, tk_g = g.attend(layer, slots, slots, rnd, 256)
            out_r, tk_r = ref.attend(layer, slots, slots, rnd, 256)
            assert g.pool.check_device() == 0 and ref.pool.check_device() == 0
            assert torch.equal(out_g, out_r) and torch.equal(tk_g, tk_r), "placement changed a value"
            assert np.array_equal(tk_g.cpu().numpy(), tk_ref)
            check_out(out_g.cpu().numpy().reshape(out_ref.shape), out_ref, w["cache_dtype"])
        # activity stamps of every live block equal the oracle's
        live = [b for b in range(32) if o.block_location(b)[0] == 0]
        assert g.pool.epoch() == o.epoch()
        assert g.pool.block_activity(live).tolist() == [o.block_location(b)[2] for b in live]
        for idle in (0, 1, 2):
            assert g.pool.inactive_blocks(idle).tolist() == o.inactive_blocks(idle).tolist()
        # offload every resident block but one, bring one back
        res = o.inactive_blocks(0).tolist()[1:]
        room = 24 - sum(1 for b in live if o.block_location(b)[1] < 0)
        res = res[:room]
        assert o.offload(res) == 0
        g.pool.offload(res)
        back = [b for b in live if o.block_location(b)[1] < 0][:1]
        assert o.fetch(back) == 0
        g.pool.fetch(back)
        locations_match(o, g, 32)
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    assert any(o.block_location(b)[1] < 0 for b in range(32) if o.block_location(b)[0] == 0)
    for s_ in slots:
        compare_request_state(g, o, s_)
    # images of requests with offloaded blocks: the oracle's bytes; restored
    # into the HiSparse pool they take GPU slots and stamps like the oracle's
    n = (L[0] // mp) * mp
    assert n > 0
    rc, ref_img = o.export_prefix(slots[0], n, 0)
    img = g.pool.export_prefix(slots[0], n, 0)
    torch.cuda.synchronize()
    assert np.array_equal(img.numpy()[:ref_img.size], ref_img)
    for s_ in slots[1:]:
        assert o.free_request(s_) == 0
        g.pool.free_request(s_)
    r = g.pool.alloc_request()
    assert o.alloc_request()[1] == r
    wl = min(n, w["n_win"])
    k, v, _ = H.tokens(w, [slots[0]], [n - wl], [wl])
    gk, gv, _ = g.tokens([slots[0]], [n - wl], [wl])
    assert o.import_prefix(r, ref_img, k, v) == 0
    g.pool.import_prefix(r, img, gk, gv)
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    locations_match(o, g, 32)
    ids = o.request_info(r)[2].tolist()
    assert g.pool.block_activity(ids).tolist() == [o.block_location(b)[2] for b in ids]
    compare_request_state(g, o, r)
    for layer in range(g.nl):
        q, qi = H.queries(w, layer, [slots[0], slots[0]], 99)  # both rows: the source's query
        rc, out_ref, tk_ref = o.decode_attend(layer, [slots[0], r], q, qi, 256)
        out_g, tk_g = g.attend(layer, [slots[0], r], [slots[0], slots[0]], 99, 256)
        assert g.pool.check_device() == 0
        assert np.array_equal(tk_g.cpu().numpy(), tk_ref)
        check_out(out_g.cpu().numpy().reshape(out_ref.shape), out_ref, w["cache_dtype"])


def test_host_slot_bytes_span_every_csa_layer():
    w = dict(W.MIXED_SERVING, n_win=256, seed=45, csa_hot_slots=4, csa_host_slots=4)
    g = GpuCase(w, 2, 8, 8, 2, 64)
    per = [g.pool.layout(l) for l in range(4)]
    csa = [d for d, k in zip(per, w["layer_kinds"]) if k in (K.CSA, K.CSA_HCA)]
    assert g.pool.host_slot_bytes() == sum(d["csa_block_bytes"] for d in csa)
    assert [d["csa_host_offset"] for d in csa] == [0, csa[0]["csa_block_bytes"]]
    assert [d["csa_host_offset"] for d, k in zip(per, w["layer_kinds"]) if k not in (K.CSA, K.CSA_HCA)] == [-1, -1]
