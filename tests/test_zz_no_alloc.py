"""The allocation-free top-k entry point (kvpool_topk_static) against the
regular path.  Some callers cannot allocate device memory (a plugin that only
gets its input and output buffers from a framework that owns every
allocation, a serving loop whose memory is budgeted once at start-up);
kvpool_topk_static serves them from a static device array.  Its
selection must equal what kvpool_decode_attend returns as top-k for the same
indexer scores -- exactly, as every top-k comparison in these tests -- on two
calls in a row (the second call reuses the array the first one left behind).
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import GpuCase

pytestmark = pytest.mark.gpu


def test_static_topk_matches_decode_attend_topk_twice():
    w = dict(W.DECODE_BATCH, seed=31)
    o = H.make_oracle(w, 4, 64, 16)
    g = GpuCase(w, 4, 64, 16, 4, 512)
    slots = [g.pool.alloc_request() for _ in range(3)]
    assert [o.alloc_request()[1] for _ in range(3)] == slots
    L = 1500  # same length: 375 CSA entries per request
    k, v, x = H.tokens(w, slots, [0] * 3, [L] * 3)
    assert o.append(slots, [L] * 3, k, v, x) == 0
    g.append(slots, slots, [0] * 3, [L] * 3)
    for call, top_k in enumerate((100, 100, 375, 7)):
        # regular path: top-k from decode_attend
        out, tk_ref = g.attend(0, slots, slots, call, top_k)
        tk_ref = tk_ref.cpu().numpy()
        # the same indexer scores (the oracle's fp32 chain, identical to the GPU's)
        _, qi = H.queries(w, 0, slots, call)
        scores = np.stack([o.request_scores(0, s, qi[j], L // 4)[1] for j, s in enumerate(slots)])
        d_scores = torch.from_numpy(scores).cuda()
        got = torch.full((3, top_k), -7, dtype=torch.int32, device="cuda")
        assert K.topk_static(d_scores, top_k, got) == 0
        assert K.topk_static_check() == (0, 0), "the kernels flagged an error"
        assert np.array_equal(got.cpu().numpy(), tk_ref), f"call {call}: static top-k differs"


def test_static_topk_refuses_oversized_and_pads():
    big = torch.zeros((2, 4 << 20), dtype=torch.float32, device="cuda")
    out = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    assert K.topk_static(big, 8, out) == K.ERR_INVALID_ARG
    s = torch.tensor([[3.0, -0.0, 0.0, 3.0]], device="cuda")
    out = torch.zeros((1, 6), dtype=torch.int32, device="cuda")
    assert K.topk_static(s, 6, out) == 0
    assert out.cpu().tolist() == [[0, 1, 2, 3, -1, -1]]
    out = torch.zeros((1, 3), dtype=torch.int32, device="cuda")
    assert K.topk_static(s, 3, out) == 0
    assert out.cpu().tolist() == [[0, 1, 3]]  # 3, 3, then the first of the equal zeros


def _scores(kind, rows, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal((rows, n)).astype(np.float32)
    if kind == "ties":  # few distinct values: the k-th largest is shared by thousands of keys
        return rng.integers(-3, 7, (rows, n)).astype(np.float32)
    if kind == "signed_zeros":  # +0 and -0 are one value; the order among them is the index order
        s = rng.choice(np.array([0.0, -0.0, 1.5, -2.0], np.float32), (rows, n))
        return s.astype(np.float32)
    if kind == "equal":
        return np.full((rows, n), 0.25, np.float32)
    if kind == "narrow":  # positive values in one octave: most keys share the top radix digits
        return (1.0 + rng.random((rows, n))).astype(np.float32)
    raise ValueError(kind)


# candidate counts on both sides of the select paths' limits: one CTA per row
# (<= 4096), 4096-key chunks with a last-CTA threshold (up to 16 chunks), one
# thread-block cluster per row with its keys in shared memory (beyond), each
# with a ragged last chunk
@pytest.mark.parametrize("n, top_k, kind", [
    (4096, 512, "normal"),
    (4097, 512, "ties"),
    (40000, 2048, "narrow"),
    (65536, 2048, "normal"),
    (65537, 2048, "ties"),
    (65537, 1, "normal"),
    (100003, 2048, "signed_zeros"),
    (100003, 777, "equal"),
    (262145, 2048, "narrow"),
    (262145, 2048, "ties"),
    (300001, 300001, "normal"),
    (300001, 300000, "ties"),
    (491520, 2048, "narrow"),     # the largest rows a cluster takes (30,720 keys per CTA)
    (491521, 2048, "narrow"),     # one more: 4096-key chunks
    (1048576, 2048, "normal"),    # the largest row: 256 chunks
    (1, 5, "normal"),             # fewer columns than top_k: all of them, then -1
    (0, 3, "normal"),             # no columns: -1 only
])
def test_static_topk_matches_the_oracle_across_select_paths(n, top_k, kind):
    """Every row's selection equals the oracle's top-k (largest scores,
    the lowest indices first among equal ones, ascending order, -1 padding)
    bit for bit, on two calls in a row."""
    import oracle as O
    rows = 4 if n <= 100003 else (2 if n <= 300001 else 1)
    s = _scores(kind, rows, n, seed=n + top_k)
    d = torch.from_numpy(s).cuda()
    ref = np.stack([O.topk(s[r], top_k) for r in range(rows)])
    for call in range(2):
        got = torch.full((rows, top_k), -7, dtype=torch.int32, device="cuda")
        assert K.topk_static(d, top_k, got) == 0
        assert K.topk_static_check() == (0, 0), "the kernels flagged an error"
        g = got.cpu().numpy()
        for r in range(rows):
            if not np.array_equal(g[r], ref[r]):
                bad = np.nonzero(g[r] != ref[r])[0]
                pytest.fail(f"call {call} row {r}: {bad.size} positions differ, first {bad[:6].tolist()}")
