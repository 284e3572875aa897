"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the
same seeded inputs: block tables, counts, tails, every stored entry and window
token and the top-k index sets bit-exact; attention outputs within the
tolerance of the cache dtype (fp32 1e-4 / rel-L2 1e-5, bf16 2e-2 / 5e-3,
fp8 6e-2)."""
import numpy as np
import pytest
import torch

from heterogeneous_compressed_kv_gb300 import gen
from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import GpuCase, check_out, compare_request_state

pytestmark = pytest.mark.gpu


def make_pair(w, max_requests, max_blocks, mbpr, max_batch, max_top_k, gates=None):
    o = H.make_oracle(w, max_requests, max_blocks, mbpr, gate_override=gates)
    g = GpuCase(w, max_requests, max_blocks, mbpr, max_batch, max_top_k, gates=gates)
    return o, g


def append_both(o, g, slots, wids, pos0s, counts):
    k, v, x = H.tokens(g.w, wids, pos0s, counts)
    rc1 = o.append(slots, counts, k, v, x)
    rc2 = g.append(slots, wids, pos0s, counts, check=False)
    assert rc1 == rc2 == 0, (rc1, rc2, g.pool.last_error())


def attend_both(o, g, layer, slots, wids, step, top_k):
    q, qi = H.queries(g.w, layer, wids, step)
    rc, ref, tk_ref = o.decode_attend(layer, slots, q, qi, top_k)
    assert rc == 0
    out, tk = g.attend(layer, slots, wids, step, top_k)
    assert g.pool.check_device() == 0
    tk = tk.cpu().numpy()
    assert np.array_equal(tk, tk_ref), "top-k index sets differ"
    return check_out(out.cpu().numpy().reshape(ref.shape), ref, g.w["cache_dtype"])


def test_generator_device_matches_host():
    runs = [(gen.stream_id(gen.K, 0, 3), 17, 1000, 0), (gen.stream_id(gen.V, 2, 9), 5, 777, 1000)]
    for dt, tdt in ((gen.OUT_F32, torch.float32), (gen.OUT_BF16, torch.bfloat16)):
        host = gen.fill_host(1777, dt, 42, runs)
        dev = torch.empty(1777, dtype=tdt, device="cuda")
        gen.fill_device(dev.data_ptr(), dt, 42, runs, torch.cuda.current_stream().cuda_stream)
        got = dev.cpu().view(torch.int32 if dt == gen.OUT_F32 else torch.int16).numpy()
        assert np.array_equal(got.view(host.dtype), host)


def test_tiny_fp32_inputs_with_fp4_indexer():
    """fp32 inputs and cache with FP4 indexer entries: the query is not exact
    in f16, so the scores take the plain fp32 chain."""
    w = dict(W.TINY, idx_fp4=1, seed=31)
    o, g = make_pair(w, 2, 8, 4, 2, 64)
    r = g.pool.alloc_request()
    assert o.alloc_request() == (0, r)
    append_both(o, g, [r], [0], [0], [300])
    compare_request_state(g, o, r)
    for step in range(3):
        append_both(o, g, [r], [0], [300 + step], [1])
        attend_both(o, g, 0, [r], [0], step, w["top_k"])


def test_tiny_prefix_130_then_8_decode_steps():
    """Tiny workload: 1 layer, 1 request, prefix L=130 in one append (one
    sealed block, 32 CSA + 1 HCA, 2-token tail), then 8 x (append 1, attend)
    with top_k = 16 and with top_k covering every entry."""
    w = W.TINY
    o, g = make_pair(w, 2, 8, 4, 2, 64)
    r = g.pool.alloc_request()
    assert o.alloc_request() == (0, r)
    append_both(o, g, [r], [0], [0], [130])
    compare_request_state(g, o, r)
    rc, info, ids = g.pool.request_info(r)
    assert (info["n_csa"], info["n_hca"], info["hca_tail"], len(ids)) == (32, 1, 2, 1)
    for step in range(w["decode_steps"]):
        L = 130 + step
        append_both(o, g, [r], [0], [L], [1])
        compare_request_state(g, o, r)
        attend_both(o, g, 0, [r], [0], step, w["top_k"])
        attend_both(o, g, 0, [r], [0], step, 64)


@pytest.mark.parametrize("cache,idx_fp4,per_token", [(K.BF16, 0, 0), (K.FP8_E4M3, 0, 0), (K.FP8_E4M3, 1, 0),
                                                    (K.BF16, 0, 1)])
def test_long_units_split_over_ctas(cache, idx_fp4, per_token):
    """Prefill chunks of one request, the launches too small to fill the
    GPU: each long unit's HCA chain runs in one CTA and its CSA groups and
    window tokens in several others.  130 tokens, then 2,000 (the first unit
    starts inside a CSA group, the last ends inside one), then 2,048 more,
    then decode steps; every stored entry, accumulator-derived entry and
    window token bit-exact, attention within tolerance."""
    w = dict(W.DECODE_BATCH, cache_dtype=cache, seed=28, idx_fp4=idx_fp4, idx_per_token=per_token)
    o, g = make_pair(w, 2, 48, 40, 2, 256)
    r = g.pool.alloc_request()
    assert o.alloc_request()[1] == r
    L = 0
    for n in (130, 2000, 2048):
        append_both(o, g, [r], [r], [L], [n])
        L += n
        compare_request_state(g, o, r)
    for step in range(3):
        append_both(o, g, [r], [r], [L], [1])
        L += 1
        attend_both(o, g, 0, [r], [r], step, 256)
    compare_request_state(g, o, r)


@pytest.mark.parametrize("cache", [K.BF16, K.FP8_E4M3])
def test_split_units_with_mixed_layer_kinds(cache):
    """Split units across layers of every kind ([SWA-only, CSA, HCA, CSA],
    window 512): one request's appends of 600 and 640 tokens are few units
    for 4 layers x 2 slices, so each long unit runs as an HCA CTA and CSA
    CTAs; in a layer without HCA the HCA CTA has nothing but the seal copies,
    in one without CSA the CSA CTAs only write the window."""
    w = dict(W.MIXED_SERVING, n_win=512, seed=29, cache_dtype=cache)
    o, g = make_pair(w, 2, 40, 16, 2, 256)
    r = g.pool.alloc_request()
    assert o.alloc_request()[1] == r
    L = 0
    for n in (130, 600, 640):
        append_both(o, g, [r], [r], [L], [n])
        L += n
        compare_request_state(g, o, r)
    for step in range(2):
        append_both(o, g, [r], [r], [L], [1])
        L += 1
        for layer in range(4):
            attend_both(o, g, layer, [r], [r], step, 256)
    compare_request_state(g, o, r)


@pytest.mark.parametrize("cache,idx_fp4", [(K.BF16, 0), (K.FP8_E4M3, 0), (K.FP8_E4M3, 1), (K.BF16, 1)])
def test_batched_ragged_appends_and_decode(cache, idx_fp4):
    """Decode-batch shapes (16 heads x 128, indexer 4 x 64) with ragged,
    unaligned multi-request appends (blocks sealed mid-call, a call spanning
    three segments with a partial start and end), then decode steps; the
    indexer entries in the cache dtype or in FP4."""
    w = dict(W.DECODE_BATCH, cache_dtype=cache, seed=21, idx_fp4=idx_fp4)
    o, g = make_pair(w, 6, 64, 16, 6, 128)
    slots = [g.pool.alloc_request() for _ in range(5)]
    assert [o.alloc_request()[1] for _ in range(5)] == slots
    L = [0] * 5
    rng = np.random.default_rng(3)
    for rnd in range(4):
        counts = [int(x) for x in rng.integers(0, 400, 5)]
        if rnd == 1:
            counts[2] = 300  # spans three segments
        append_both(o, g, slots, slots, L, counts)
        L = [a + b for a, b in zip(L, counts)]
    for s in slots:
        compare_request_state(g, o, s)
    for step in range(3):
        append_both(o, g, slots, slots, L, [1] * 5)
        L = [a + 1 for a in L]
        attend_both(o, g, 0, slots, slots, step, 128)
    for s in slots:
        compare_request_state(g, o, s)


@pytest.mark.parametrize("in_dtype,cache,heads,head_dim", [
    (K.F32, K.BF16, 8, 64), (K.BF16, K.BF16, 8, 64), (K.F32, K.BF16, 16, 128),
    (K.F32, K.FP8_E4M3, 8, 64), (K.BF16, K.FP8_E4M3, 8, 64), (K.F32, K.F32, 16, 128)])
def test_attention_consumer_layouts(in_dtype, cache, heads, head_dim):
    """Every mapping of the attention consumers' dims: bf16 caches take two
    runs of 8 dims half a head apart, fp8 and fp32 caches 16 contiguous dims;
    64- and 128-dim heads (4 and 8 threads per head); fp32 and bf16 inputs."""
    w = dict(W.DECODE_BATCH, in_dtype=in_dtype, cache_dtype=cache, heads=heads, head_dim=head_dim, seed=33)
    o, g = make_pair(w, 3, 32, 16, 3, 64)
    slots = [g.pool.alloc_request() for _ in range(3)]
    assert [o.alloc_request()[1] for _ in range(3)] == slots
    L = [0] * 3
    for counts in ([300, 77, 513], [200, 400, 3]):
        append_both(o, g, slots, slots, L, counts)
        L = [a + b for a, b in zip(L, counts)]
    for step in range(2):
        append_both(o, g, slots, slots, L, [1] * 3)
        L = [a + 1 for a in L]
        attend_both(o, g, 0, slots, slots, step, 64)
    for sl in slots:
        compare_request_state(g, o, sl)


def test_prefix_sharing_with_recomputed_window():
    """Chunked-prefill shapes: request 0 appends 2048-token chunks; requests
    1 and 2 share its first 1024 tokens (8 sealed blocks) with the window
    recomputed by the caller, then all grow on their own."""
    w = dict(W.CHUNKED_PREFILL, seed=22)
    o, g = make_pair(w, 4, 64, 16, 4, 128)
    s = [g.pool.alloc_request() for _ in range(3)]
    assert [o.alloc_request()[1] for _ in range(3)] == s
    append_both(o, g, [s[0]], [0], [0], [512])
    append_both(o, g, [s[0]], [0], [512], [700])
    n = 1024
    wlen = min(n, w["n_win"])
    k, v, _ = H.tokens(w, [0], [n - wlen], [wlen])
    gk, gv, _ = g.tokens([0], [n - wlen], [wlen])
    for dst in (s[1], s[2]):
        assert o.share_prefix(dst, s[0], n, k, v) == 0
        g.pool.share_prefix(dst, s[0], n, gk, gv)
    for b in o.request_info(s[0])[2][:8]:
        assert g.pool.block_refcount(int(b)) == o.block_refcount(int(b)) == 3
    # requests 1 and 2 continue with their own tokens (workload ids 1, 2)
    append_both(o, g, [s[1], s[2], s[0]], [1, 2, 0], [n, n, 1212], [300, 17, 5])
    for x in s:
        compare_request_state(g, o, x)
    attend_both(o, g, 0, s, [0, 1, 2], 0, 128)
    # the shared blocks are immutable: free the owner, the sharers still read them
    o.free_request(s[0])
    g.pool.free_request(s[0])
    attend_both(o, g, 0, [s[1], s[2]], [1, 2], 1, 128)


def test_edge_cases_small_lengths_and_top_k_limits():
    w = dict(W.DECODE_BATCH, seed=23)
    o, g = make_pair(w, 8, 32, 8, 8, 600)
    slots = [g.pool.alloc_request() for _ in range(6)]
    [o.alloc_request() for _ in range(6)]
    lens = [1, 3, 4, 127, 128, 129]
    append_both(o, g, slots, slots, [0] * 6, lens)
    for x in slots:
        compare_request_state(g, o, x)
    for top_k in (0, 1, 31, 32, 33, 600):
        attend_both(o, g, 0, slots, slots, top_k, top_k)


def test_equal_scores_select_lowest_indices():
    """q_idx = 0 makes every indexer score +0 (or -0): the top-k must be the
    k lowest entry indices (ties broken by lower index; -0 == +0)."""
    w = dict(W.DECODE_BATCH, seed=24)
    o, g = make_pair(w, 2, 32, 16, 2, 256)
    r = g.pool.alloc_request()
    o.alloc_request()
    append_both(o, g, [r], [0], [0], [1500])
    q, _ = H.queries(w, 0, [0], 0)
    qi = np.zeros((1, g.XD), np.float32)
    rc, ref, tk_ref = o.decode_attend(0, [r], q, qi, 100)
    assert tk_ref[0].tolist() == list(range(100))
    gq, _ = g.queries(0, [0], 0)
    gqi = torch.zeros((1, g.XD), dtype=g.tdtype, device="cuda")
    out = torch.empty((1, g.HD), dtype=torch.float32, device="cuda")
    tk = torch.empty((1, 100), dtype=torch.int32, device="cuda")
    g.pool.decode_attend(0, [r], gq, gqi, 100, out, tk)
    assert tk.cpu().numpy()[0].tolist() == list(range(100))
    check_out(out.cpu().numpy().reshape(ref.shape), ref, w["cache_dtype"])


def test_select_paths_in_one_launch():
    """One decode launch whose requests take different select shapes: 67,500
    candidates (17 chunks of 4096 keys), 5,000 (2 chunks), 75 (a chunk with
    a ragged tail), 0 (k = 0, padding only); top-k sets bit-exact,
    outputs within fp32 tolerance; then the same with every indexer score
    equal (q_idx = 0: the k lowest indices), which puts all 67,500 keys on
    the threshold."""
    w = dict(W.TINY, seed=26)
    lens = [270003, 20001, 300, 2]
    mp_ = w["m_prime"]
    o, g = make_pair(w, 4, sum(L // mp_ + 1 for L in lens) + 4, lens[0] // mp_ + 4, 4, 4096)
    slots = [g.pool.alloc_request() for _ in lens]
    assert [o.alloc_request()[1] for _ in lens] == slots
    pos = [0] * len(lens)
    while True:
        cnt = [min(16384, L - p) for L, p in zip(lens, pos)]
        if sum(cnt) == 0:
            break
        live = [j for j, c in enumerate(cnt) if c > 0]
        append_both(o, g, [slots[j] for j in live], live, [pos[j] for j in live], [cnt[j] for j in live])
        pos = [p + c for p, c in zip(pos, cnt)]
    wids = list(range(len(lens)))
    for step, top_k in enumerate((64, 2048, 4096)):
        attend_both(o, g, 0, slots, wids, step, top_k)
    attend_both(o, g, 0, [slots[0], slots[3]], [0, 3], 7, 300)
    q, _ = H.queries(w, 0, [0], 0)
    qi = np.zeros((1, g.XD), np.float32)
    rc, ref, tk_ref = o.decode_attend(0, [slots[0]], q, qi, 1000)
    assert tk_ref[0].tolist() == list(range(1000))
    gq, _ = g.queries(0, [0], 0)
    gqi = torch.zeros((1, g.XD), dtype=g.tdtype, device="cuda")
    out = torch.empty((1, g.HD), dtype=torch.float32, device="cuda")
    tk = torch.empty((1, 1000), dtype=torch.int32, device="cuda")
    g.pool.decode_attend(0, [slots[0]], gq, gqi, 1000, out, tk)
    assert g.pool.check_device() == 0
    assert tk.cpu().numpy()[0].tolist() == list(range(1000))
    check_out(out.cpu().numpy().reshape(ref.shape), ref, w["cache_dtype"])


def test_mixed_layer_kinds_with_churn():
    """Mixed-serving shapes at reduced scale: layers [SWA-only, CSA, HCA,
    CSA], window 512, requests finishing and arriving between steps."""
    w = dict(W.MIXED_SERVING, n_win=512, seed=25)
    o, g = make_pair(w, 10, 96, 16, 10, 256)
    rng = np.random.default_rng(5)
    live = {}
    wid = 0
    for _ in range(6):
        s = g.pool.alloc_request()
        assert o.alloc_request()[1] == s
        live[s] = [wid, 0]
        wid += 1
    for step in range(4):
        # arrivals' prefill + everyone's decode token in one append
        slots = sorted(live)
        counts = [int(rng.integers(200, 900)) if live[s_][1] == 0 else 1 for s_ in slots]
        append_both(o, g, slots, [live[s_][0] for s_ in slots], [live[s_][1] for s_ in slots], counts)
        for s_, c in zip(slots, counts):
            live[s_][1] += c
        for layer in range(4):
            attend_both(o, g, layer, slots, [live[s_][0] for s_ in slots], step, 256)
        # churn: one finishes, one arrives
        gone = slots[int(rng.integers(0, len(slots)))]
        o.free_request(gone)
        g.pool.free_request(gone)
        del live[gone]
        s = g.pool.alloc_request()
        assert o.alloc_request()[1] == s
        live[s] = [wid, 0]
        wid += 1
    for s_ in sorted(live):
        if live[s_][1] > 0:
            compare_request_state(g, o, s_)


def test_bounded_wait_is_reported_and_the_pool_stays_usable():
    """Failure detection without a fault: a kernel waits on a barrier that
    nothing completes; its wait gives up after the 1 s limit and sets the
    wait flag, which kvpool_check_device reports; the context, the pool and
    the error word are usable afterwards."""
    import time
    w = dict(W.DECODE_BATCH, seed=26)
    o, g = make_pair(w, 2, 8, 4, 2, 64)
    r = g.pool.alloc_request()
    assert o.alloc_request()[1] == r
    append_both(o, g, [r], [0], [0], [200])
    t0 = time.time()
    g.pool.wait_selftest()
    with pytest.raises(K.KvpoolError) as e:
        g.pool.check_device()
    assert e.value.code == K.ERR_DEVICE_CHECK and "flags 0x1" in str(e.value)
    assert time.time() - t0 >= 0.9
    assert g.pool.check_device() == 0  # read and cleared
    append_both(o, g, [r], [r], [200], [1])
    attend_both(o, g, 0, [r], [r], 0, 64)


def test_profiling_events_and_count_only_agree():
    """The two profiling modes account the same launches: two pools with the
    same history run the same decode step, one recording events and one
    counting without events; launch counts and algorithmic bytes agree for
    every kernel kind, the count-only mode measures no time and records no
    timeline, and the outputs are the same bits."""
    w = dict(W.DECODE_BATCH, seed=27)
    cases = [GpuCase(w, 3, 32, 8, 3, 128) for _ in range(2)]
    totals, outs = [], []
    for g, (kinds, count) in zip(cases, ((None, False), ([], True))):
        slots = [g.pool.alloc_request() for _ in range(3)]
        g.append(slots, slots, [0, 0, 0], [700, 300, 1100])
        g.pool.profile_enable(True, kinds=kinds, count=count)
        g.append(slots, slots, [700, 300, 1100], [1, 1, 1])
        out, tk = g.attend(0, slots, slots, 0, 128)
        assert g.pool.check_device() == 0
        totals.append([g.pool.profile_read(k) for k in range(len(K.KERNEL_NAMES))])
        if count:
            assert g.pool.profile_timeline() == []
        g.pool.profile_enable(False)
        outs.append((out.cpu().numpy(), tk.cpu().numpy()))
    ev, ct = totals
    for k, name in enumerate(K.KERNEL_NAMES):
        assert ev[k][1:] == ct[k][1:], (name, ev[k], ct[k])
        assert ct[k][0] == 0.0, name
    for name in ("append", "score", "select", "attend", "combine"):
        e = ev[K.KERNEL_NAMES.index(name)]
        assert e[0] > 0 and e[1] > 0, (name, e)
        # the select's keys are scratch that stays in L2: no algorithmic bytes
        assert (e[2] == 0) == (name == "select"), (name, e)
    assert np.array_equal(outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][0].view(np.uint8), outs[1][0].view(np.uint8))
