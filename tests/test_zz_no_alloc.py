"""The allocation-free top-k entry point (kvpool_topk_static) against the
regular path.  Some callers cannot allocate device memory (a stream being
captured into a CUDA graph, a plugin that only gets its input and output
buffers); kvpool_topk_static serves them from a static device array.  Its
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
        torch.cuda.synchronize()
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
