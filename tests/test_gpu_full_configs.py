"""Parity at the workloads' full sizes, in the launch configuration bench.py
times.  Where the oracle can follow the whole run in seconds it does (decode
batch, chunked prefill); at 1M-token context it checks sampled outputs it can
compute one by one and properties that hold at any size (long context)."""
import struct

import numpy as np
import pytest
import torch

from heterogeneous_compressed_kv_gb300 import gen
from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import GpuCase, check_out, compare_request_state

pytestmark = pytest.mark.gpu


def _pair(w, max_requests, max_blocks, mbpr, max_batch, max_top_k):
    o = H.make_oracle(w, max_requests, max_blocks, mbpr)
    g = GpuCase(w, max_requests, max_blocks, mbpr, max_batch, max_top_k)
    return o, g


def _append(o, g, slots, wids, pos0s, counts):
    k, v, x = H.tokens(g.w, wids, pos0s, counts)
    assert o.append(slots, counts, k, v, x) == 0
    assert g.append(slots, wids, pos0s, counts, check=False) == 0, g.pool.last_error()


def _attend(o, g, slots, wids, step, top_k):
    q, qi = H.queries(g.w, 0, wids, step)
    rc, ref, tk_ref = o.decode_attend(0, slots, q, qi, top_k)
    assert rc == 0
    out, tk = g.attend(0, slots, wids, step, top_k)
    assert g.pool.check_device() == 0
    assert np.array_equal(tk.cpu().numpy(), tk_ref), f"top-k index sets differ at step {step}"
    return check_out(out.cpu().numpy().reshape(ref.shape), ref, g.w["cache_dtype"])


def test_decode_batch_full():
    """32 requests with lengths U[1, 8192] (seed 1), bf16, top_k 512: prefill
    in 2048-token chunks, then 100 decode steps of one token per request;
    top-k sets and outputs compared every 10th step, the stored state of
    every request (sampled entries) at the end."""
    w = W.DECODE_BATCH
    B = w["n_requests"]
    lens = [int(x) for x in W.uniform_lengths(w["seed"], B, w["len_lo"], w["len_hi"])]
    steps = w["decode_steps"]
    mbpr = (max(lens) + steps) // w["m_prime"] + 2
    max_blocks = sum((L + steps) // w["m_prime"] + 1 for L in lens)
    o, g = _pair(w, B, max_blocks, mbpr, B, w["top_k"])
    slots = [g.pool.alloc_request() for _ in range(B)]
    assert [o.alloc_request()[1] for _ in range(B)] == slots
    wids = list(range(B))
    pos = [0] * B
    while True:
        cnt = [min(2048, L - p) for L, p in zip(lens, pos)]
        if sum(cnt) == 0:
            break
        _append(o, g, slots, wids, pos, cnt)
        pos = [p + c for p, c in zip(pos, cnt)]
    for step in range(steps):
        _append(o, g, slots, wids, pos, [1] * B)
        pos = [p + 1 for p in pos]
        if step % 10 == 0 or step == steps - 1:
            _attend(o, g, slots, wids, step, w["top_k"])
    rng = np.random.default_rng(0)
    for s in slots:
        compare_request_state(g, o, s, sample=24, rng=rng)


def test_chunked_prefill_full():
    """4 requests x 32768 tokens in 2048-token chunks; the first 16384 tokens
    are request 0's, shared by requests 1-3 through refcounted blocks (their
    windows recomputed by the caller); every request then appends its own
    16384 tokens in 2048-token chunks, batched.  Tables, refcounts and every
    stored entry bit-exact; then decode steps at top_k 512."""
    w = W.CHUNKED_PREFILL
    B, T, C, S = w["n_requests"], w["tokens"], w["chunk"], w["shared"]
    mp = w["m_prime"]
    mbpr = T // mp + 4
    o, g = _pair(w, B, S // mp + B * ((T - S) // mp + 2), mbpr, B, w["top_k"])
    slots = [g.pool.alloc_request() for _ in range(B)]
    assert [o.alloc_request()[1] for _ in range(B)] == slots
    for p0 in range(0, S, C):
        _append(o, g, [slots[0]], [0], [p0], [C])
    wlen = min(S, w["n_win"])
    k, v, _ = H.tokens(w, [0], [S - wlen], [wlen])
    gk, gv, _ = g.tokens([0], [S - wlen], [wlen])
    for dst in slots[1:]:
        assert o.share_prefix(dst, slots[0], S, k, v) == 0
        g.pool.share_prefix(dst, slots[0], S, gk, gv)
    for b in o.request_info(slots[0])[2]:
        assert g.pool.block_refcount(int(b)) == o.block_refcount(int(b)) == B
    wids = list(range(B))
    for p0 in range(S, T, C):
        _append(o, g, slots, wids, [p0] * B, [C] * B)
    assert g.pool.free_block_count() == o.free_block_count()
    for s in slots:
        compare_request_state(g, o, s)
    pos = [T] * B
    for step in range(4):
        _append(o, g, slots, wids, pos, [1] * B)
        pos = [p + 1 for p in pos]
        _attend(o, g, slots, wids, step, w["top_k"])


def _spawn_pool():
    import multiprocessing as mp
    import os
    return mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))


@pytest.mark.parametrize("idx_fp4, per_token", [(0, 0), (1, 0), (0, 1)], ids=["fp8", "fp4", "fp8_per_token"])
def test_long_context_full_sampled(idx_fp4, per_token):
    """8 requests x 1,048,576 tokens, fp8 cache, top_k 2048, in bench.py's
    pool configuration and prefill order (2048-token chunks, every request per
    call), then one decode step.  For one request the oracle recomputes, one
    piece at a time in worker processes, all 262,144 indexer scores (top-k set
    compared bit for bit), all 8,192 HCA entries, the selected CSA entries and
    the window, and the attention output (fp8 tolerance); sampled CSA,
    indexer and HCA entries and the window are compared byte for byte with
    the arena; block tables follow the smallest-free policy.  Indexer entries
    in fp8 (the workload) or FP4, or one fp8 key per token."""
    from tests import oracle_pool as OP
    w = dict(W.LONG_CONTEXT, idx_fp4=idx_fp4, idx_per_token=per_token)
    B, Lc, C, mp_, top_k = w["n_requests"], w["length"], w["chunk"], w["m_prime"], w["top_k"]
    extra = 8
    g = GpuCase(w, B, B * ((Lc + extra) // mp_ + 1), (Lc + extra) // mp_ + 2, B, top_k)
    o = OP._oracle(w)
    slots = [g.pool.alloc_request() for _ in range(B)]
    wids = list(range(B))
    for p0 in range(0, Lc, C):
        assert g.append(slots, wids, [p0] * B, [C] * B, check=False) == 0
    assert g.append(slots, wids, [Lc] * B, [1] * B, check=False) == 0
    out, tk = g.attend(0, slots, wids, 0, top_k)
    assert g.pool.check_device() == 0
    out, tk = out.cpu().numpy(), tk.cpu().numpy()
    L = Lc + 1
    n_csa, n_hca = L // w["m"], L // mp_
    # block ids: chunk c seals 16 blocks per request, requests in batch order
    per = C // mp_
    for r, s in enumerate(slots):
        rc, info, ids = g.pool.request_info(s)
        assert info["length"] == L and info["n_csa"] == n_csa and info["n_hca"] == n_hca
        expect = [c * B * per + r * per + j for c in range(Lc // C) for j in range(per)]
        assert ids.tolist() == expect
    import oracle as O
    pool = _spawn_pool()
    try:
        n_w = pool._processes
        # two requests' outputs against the oracle (both bounds of check_out)
        for r in (2, 5):
            s, wid = slots[r], wids[r]
            q, qi = H.queries(w, 0, [wid], 0)
            cuts = np.linspace(0, n_csa, 4 * n_w + 1).astype(int)
            parts = pool.starmap(OP.idx_scores, [(w, wid, qi[0], int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])])
            scores = np.concatenate(parts)
            hcuts = np.linspace(0, n_hca, 4 * n_w + 1).astype(int)
            hparts = pool.starmap(OP.kv_entries,
                                  [(w, wid, 2, list(range(int(a), int(b)))) for a, b in zip(hcuts[:-1], hcuts[1:])])
            sel = O.topk(scores, top_k)
            assert np.array_equal(tk[r], sel), f"request {r}: top-k index set differs from the oracle's"
            hca_codes = np.concatenate([p[0] for p in hparts])
            hca_scales = np.concatenate([p[1] for p in hparts])
            csa_codes, csa_scales = OP.kv_entries(w, wid, 1, sel.tolist())
            win_codes, win_scales = OP.window_entries(w, wid, L - w["n_win"], w["n_win"])
            codes = np.concatenate([csa_codes, hca_codes, win_codes])
            scales = np.concatenate([csa_scales, hca_scales, win_scales])
            rc, ref = o.attend_sources(codes, scales, q[0])
            assert rc == 0
            err, rel = check_out(out[r].reshape(ref.shape), ref, w["cache_dtype"])
            print(f"long context request {r}: max-abs {err:.3e}, rel-L2 {rel:.3e}")
    finally:
        pool.close()
        pool.join()
    # the rest checks request 5's stored bytes (hca_codes etc. are its own)
    _, ids = g.pool.request_info(s)[1:]
    # stored bytes: sampled CSA / indexer / HCA entries and the whole window
    rng = np.random.default_rng(1)
    es = sorted(set(rng.integers(0, n_csa, 48).tolist()) | {0, n_csa - 1})
    cc, csc = OP.kv_entries(w, wid, 1, es)
    ie = None if per_token else OP.idx_entries(w, wid, es)
    for j, e in enumerate(es):
        c, sc = g.csa_entry(0, s, e, ids)
        assert np.array_equal(c, cc[j]) and np.array_equal(sc, csc[j]), f"CSA entry {e}"
        if ie is not None:
            c, sc = g.idx_entry(0, s, e, ids)
            assert np.array_equal(c, ie[j][0]) and sc[0] == ie[j][1][0], f"indexer entry {e}"
    if per_token:  # sampled tokens' own keys, including the staged tail
        ts = sorted(set(rng.integers(0, L, 48).tolist()) | {0, L - 1})
        for t, (kc, ks) in zip(ts, OP.token_keys(w, wid, ts)):
            c, sc = g.idx_entry(0, s, t, ids)
            assert np.array_equal(c, kc) and sc[0] == ks, f"indexer key of token {t}"
    for t in sorted(set(rng.integers(0, n_hca, 16).tolist()) | {n_hca - 1}):
        c, sc = g.hca_entry(0, int(ids[t]))
        assert np.array_equal(c, hca_codes[t]) and np.array_equal(sc, hca_scales[t]), f"HCA entry {t}"
    for t, pos in enumerate(range(L - w["n_win"], L)):
        c, sc = g.window_token(0, s, pos)
        assert np.array_equal(c, win_codes[t]) and np.array_equal(sc, win_scales[t]), f"window token {pos}"
    if idx_fp4 or per_token:
        return
    # the request's 1,048,576-token prefix as an image (Zero SWA): sampled
    # entries where the image layout puts them; then restored in its place,
    # grown by the same token and decoded again: the same bits as before
    n = (L // mp_) * mp_
    nb = n // mp_
    img = g.pool.export_prefix(s, n, 0)
    torch.cuda.synchronize()
    raw = img.numpy()
    magic, ver, fp, n_tok, nbh, wh = struct.unpack("<IIQqii", raw[:32].tobytes())
    assert (magic, ver, fp, n_tok, nbh, wh) == (0x4950564B, 1, o.fingerprint(), n, nb, 0)
    lay = g.pool.layout(0)
    E, CBk, X = lay["entry_bytes"], lay["csa_per_block"], lay["idx_block_bytes"]
    HDb = 2 * w["heads"] * w["head_dim"]
    for j, e in enumerate(es):
        b, t = divmod(e, CBk)
        if b >= nb:
            continue
        off = 64 + (b * CBk + t) * E
        assert np.array_equal(raw[off:off + HDb], cc[j]), f"image CSA entry {e}"
        assert raw[off + HDb:off + HDb + 4].tobytes() == csc[j].astype("<u2").tobytes()
        part = raw[64 + nb * CBk * E + b * X:64 + nb * CBk * E + (b + 1) * X]
        key = bytes(part[(k // 16 * CBk + t) * 16 + k % 16] for k in range(lay["idx_entry_bytes"]))
        assert key == ie[j][0].tobytes(), f"image indexer entry {e}"
    for t in sorted(set(rng.integers(0, nb, 16).tolist()) | {nb - 1}):
        off = 64 + nb * (CBk * E + X) + t * E
        assert np.array_equal(raw[off:off + HDb], hca_codes[t]), f"image HCA entry {t}"
    before = g.attend(0, slots, wids, 1, top_k)
    g.pool.free_request(s)
    assert g.pool.alloc_request() == s
    wl = w["n_win"]
    gk, gv, _ = g.tokens([wid], [n - wl], [wl])
    g.pool.import_prefix(s, img, gk, gv)
    assert g.pool.request_info(s)[2].tolist() == ids[:nb].tolist()  # its own ids back: the smallest free
    assert g.append([s], [wid], [Lc], [1], check=False) == 0
    after = g.attend(0, slots, wids, 1, top_k)
    assert g.pool.check_device() == 0
    assert torch.equal(before[0], after[0]) and torch.equal(before[1], after[1]), "restored request differs"


def _mixed_schedule(w, steps):
    """The serving schedule on the host: departures and arrivals (slot,
    workload id, length) per step and the peak number of sealed blocks.
    Lengths are lognormal (median 4096, capped); slots are taken lowest first;
    step 0 has no churn."""
    B, n_ch, mp_ = w["n_requests"], W.churn_count(w), w["m_prime"]
    lens = [int(x) for x in W.lognormal_lengths(w["seed"], B, w["len_median"], w["len_sigma"], w["len_cap"])]
    cur = {s: L for s, L in enumerate(lens)}
    free, wid, plan, peak = [], B, [], 0
    for step in range(steps):
        gone, arrivals = [], []
        if step > 0:
            order = sorted(cur)
            gone = [order[j] for j in W.churn_picks(w["seed"], step, len(order), n_ch)]
            for s in gone:
                del cur[s]
            free = sorted(free + gone)
            for L in W.lognormal_lengths(w["seed"], n_ch, w["len_median"], w["len_sigma"], w["len_cap"],
                                         index0=B + (step - 1) * n_ch):
                s = free.pop(0)
                arrivals.append((s, wid, int(L)))
                cur[s] = int(L)
                wid += 1
        for s in cur:
            cur[s] += 1
        plan.append((gone, arrivals))
        peak = max(peak, sum(L // mp_ for L in cur.values()))
    return lens, plan, peak


@pytest.mark.parametrize("hisparse", [False, True], ids=["resident", "hisparse"])
def test_mixed_serving_full_sampled(hisparse):
    """256 requests, lognormal lengths (median 4096, capped at 131072), four
    layers [SWA-only, CSA, HCA, CSA], window 4096, top_k 1024; from the second
    step on, 10% of the requests finish and as many arrive (their prefill
    appended in 2048-token chunks) before every live request decodes one token
    and attends in every layer, for 200 steps.  Block tables are checked against
    the smallest-free policy replayed on the host (ids reused after
    departures); for three requests (the longest live one and the two last
    arrivals) the oracle recomputes every layer's attention output of the
    last step from the generator's tokens, with the CSA layers' top-k sets
    compared bit for bit, and sampled stored CSA entries byte for byte.
    With HiSparse, every tenth step the blocks idle for 3 or more decode
    calls move their CSA entries to host slots (up to 2,048 of them) and a
    few come back: the same checks hold, the attention reading offloaded
    entries from host memory."""
    from tests import oracle_pool as OP
    import oracle as O
    w = W.MIXED_SERVING
    steps, C, mp_, top_k, n_win = w["decode_steps"], w["chunk"], w["m_prime"], w["top_k"], w["n_win"]
    lens, plan, peak = _mixed_schedule(w, steps)
    B = w["n_requests"]
    gw = dict(w, csa_hot_slots=peak + 64, csa_host_slots=2048) if hisparse else w
    g = GpuCase(gw, B, peak + 64, (w["len_cap"] + steps) // mp_ + 2, B, top_k)
    assert [g.pool.alloc_request() for _ in range(B)] == list(range(B))
    import heapq
    live = {s: [s, 0] for s in range(B)}  # slot -> [workload id, length]
    free_ids = list(range(peak + 64))  # a heap
    table = {s: [] for s in live}

    def append(slots, counts):
        assert g.append(slots, [live[s][0] for s in slots], [live[s][1] for s in slots], counts, check=False) == 0
        # replay: smallest free id at each seal, requests in batch order, then positions
        for s, c in zip(slots, counts):
            for _ in range((live[s][1] + c) // mp_ - live[s][1] // mp_):
                table[s].append(heapq.heappop(free_ids))
            live[s][1] += c

    def prefill(slots, targets):
        while True:
            cnt = [min(C, t - live[s][1]) for s, t in zip(slots, targets)]
            if sum(cnt) == 0:
                return
            append(slots, cnt)

    prefill(list(range(B)), lens)
    last = {}
    moved = 0
    for step, (gone, arrivals) in enumerate(plan):
        for s in gone:
            g.pool.free_request(s)
            for b in table.pop(s):
                heapq.heappush(free_ids, b)
            del live[s]
        for s, wid, _ in arrivals:
            assert g.pool.alloc_request() == s
            live[s] = [wid, 0]
            table[s] = []
        if arrivals:
            prefill([a[0] for a in arrivals], [a[2] for a in arrivals])
        slots = sorted(live)
        append(slots, [1] * len(slots))
        for layer in range(4):
            out, tk = g.attend(layer, slots, [live[s][0] for s in slots], step, top_k)
            if step == steps - 1:
                last[layer] = (slots, out.cpu().numpy(), tk.cpu().numpy())
        assert g.pool.check_device() == 0
        if hisparse and step % 10 == 5:
            room = 2048 - sum(1 for ids in table.values() for b in ids if g.pool.block_location(b)[1] < 0)
            idle = g.pool.inactive_blocks(3).tolist()[:room]
            g.pool.offload(idle)
            moved += len(idle)
            back = [b for ids in table.values() for b in ids if g.pool.block_location(b)[1] < 0][:8]
            g.pool.fetch(back)
            assert g.pool.check_device() == 0
    for s in sorted(live):
        rc, info, ids = g.pool.request_info(s)
        assert info["length"] == live[s][1]
        assert ids.tolist() == table[s], f"block table of slot {s}"
    assert g.pool.free_block_count() == len(free_ids)
    assert moved > 0 or not hisparse
    # the oracle's last step for three requests
    slots = last[0][0]
    first = max(slots, key=lambda s: live[s][1])
    late = sorted((s for s in slots if s != first), key=lambda s: -live[s][0])[:2]
    o = OP._oracle(w)
    pool = _spawn_pool()
    try:
        n_w = pool._processes
        for s in [first] + late:
            wid_s, L = live[s]
            i = slots.index(s)
            for layer, kind in enumerate(w["layer_kinds"]):
                q, qi = H.queries(w, layer, [wid_s], steps - 1)
                wc, ws = OP.window_entries(w, wid_s, max(0, L - n_win), min(L, n_win), layer)
                codes, scales = [wc], [ws]
                if kind == W.CSA:
                    n_csa = L // w["m"]
                    cuts = np.linspace(0, n_csa, 2 * n_w + 1).astype(int)
                    sc = np.concatenate(pool.starmap(OP.idx_scores, [(w, wid_s, qi[0], int(a), int(b), layer)
                                                                     for a, b in zip(cuts[:-1], cuts[1:])]))
                    sel = O.topk(sc, top_k)
                    assert np.array_equal(last[layer][2][i], sel), f"top-k of slot {s}, layer {layer}"
                    cc, cs = OP.kv_entries(w, wid_s, 1, sel[sel >= 0].tolist(), layer)
                    codes.insert(0, cc)
                    scales.insert(0, cs)
                elif kind == W.HCA:
                    cuts = np.linspace(0, L // mp_, 2 * n_w + 1).astype(int)
                    hp = pool.starmap(OP.kv_entries, [(w, wid_s, 2, list(range(int(a), int(b))), layer)
                                                      for a, b in zip(cuts[:-1], cuts[1:])])
                    codes.insert(0, np.concatenate([p[0] for p in hp]))
                    scales.insert(0, np.concatenate([p[1] for p in hp]))
                rc, ref = o.attend_sources(np.concatenate(codes), np.concatenate(scales), q[0])
                assert rc == 0
                check_out(last[layer][1][i].reshape(ref.shape), ref, w["cache_dtype"])
            # sampled stored CSA entries of the two CSA layers
            _, ids = g.pool.request_info(s)[1:]
            n_csa = L // w["m"]
            es = sorted(set(np.random.default_rng(s).integers(0, n_csa, 8).tolist())) if n_csa else []
            for layer in (1, 3):
                cc, cs = OP.kv_entries(w, wid_s, 1, es, layer)
                for j, e in enumerate(es):
                    c, sc_ = g.csa_entry(layer, s, e, ids)
                    assert np.array_equal(c, cc[j]) and np.array_equal(sc_, cs[j]), f"CSA entry {e}, layer {layer}"
    finally:
        pool.close()
        pool.join()
