"""Parity of per-token indexer keys on the GPU.

Source: "V4 KV Layout: Classical + State dual pool": the State cache table
keeps one K-only indexer key per token, and a block holds 128 of them.  An
entry's score combines its m tokens' scores with the entry's indexer gates.

What is checked against the oracle:
- Every stored key, staged or sealed, is byte-exact.  Some of them are staged
  by earlier calls and copied in at the seal.
- Top-k sets are bit-exact.
- Outputs are within the cache dtype's tolerance.
- Prefix images are byte-identical and restore bit for bit.
"""
import numpy as np
import pytest
import torch

from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import compare_request_state
from tests.test_gpu_parity import append_both, attend_both, make_pair

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_f32_one_head": dict(W.TINY, seed=71, idx_per_token=1),
    "tiny_f32_two_heads": dict(W.TINY, idx_heads=2, idx_dim=32, seed=72, idx_per_token=1),
    "bf16": dict(W.DECODE_BATCH, seed=73, idx_per_token=1),
    "fp8": dict(W.LONG_CONTEXT, seed=74, idx_per_token=1),
    "fp8_fp4_keys": dict(W.LONG_CONTEXT, seed=75, idx_fp4=1, idx_per_token=1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_per_token_keys_scores_and_outputs_match_the_oracle(name):
    w = CASES[name]
    mp = w["m_prime"]
    o, g = make_pair(w, 4, 40, 12, 4, 256)
    slots = [g.pool.alloc_request() for _ in range(3)]
    assert [o.alloc_request()[1] for _ in range(3)] == slots
    L = [0, 0, 0]
    rng = np.random.default_rng(5)
    for rnd in range(5):
        # ragged calls: odd counts stage keys across calls; some calls seal
        counts = [int(x) for x in rng.integers(1, 2 * mp + 30, 3)] if rnd < 3 else [1, 3, 2]
        append_both(o, g, slots, slots, L, counts)
        L = [a + b for a, b in zip(L, counts)]
        for s_ in slots:
            compare_request_state(g, o, s_)
        for top_k in (16, 256):
            attend_both(o, g, 0, slots, slots, rnd * 10 + top_k, top_k)
    assert g.pool.check_device() == 0


@pytest.mark.parametrize("name", ["bf16", "fp8_fp4_keys"])
def test_per_token_prefix_images_match_the_oracle_and_restore(name):
    w = CASES[name]
    mp = w["m_prime"]
    o, g = make_pair(w, 4, 40, 12, 4, 256)
    a = g.pool.alloc_request()
    assert o.alloc_request()[1] == a
    append_both(o, g, [a], [0], [0], [3 * mp + 17])
    n = 3 * mp
    rc, ref = o.export_prefix(a, n, 0)
    assert rc == 0
    img = g.pool.export_prefix(a, n, 0)
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    assert np.array_equal(img.numpy()[:ref.size], ref)
    b = g.pool.alloc_request()
    assert o.alloc_request()[1] == b
    wl = min(n, w["n_win"])
    k, v, _ = H.tokens(w, [0], [n - wl], [wl])
    gk, gv, _ = g.tokens([0], [n - wl], [wl])
    assert o.import_prefix(b, ref, k, v) == 0
    g.pool.import_prefix(b, img, gk, gv)
    torch.cuda.synchronize()
    assert g.pool.check_device() == 0
    compare_request_state(g, o, b)
    append_both(o, g, [b], [0], [n], [17])
    attend_both(o, g, 0, [a, b], [0, 0], 3, 64)
