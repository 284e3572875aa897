"""Benchmark of the decode-step hot path of the two-pool KV cache on GB300.

A step = append one new token to every request (window write, CSA / indexer
/ HCA compression, block seals) + decode attention of the layer (indexer
scores, top-k select, three-source split-K attention, merge), through the
kvpool C ABI.  Default workload: the long-context configuration (8 requests
at 1,048,576 tokens: 262,144 CSA and 8,192 HCA entries each, fp8 e4m3 cache
with bf16 scales, 16 heads x 128, indexer 4 x 64, window 128, top_k 2048).

Prints one JSON line (rank 0).  With torchrun (N > 1) every rank serves its
own 8 requests on its own GPU (weak scaling, no data-path collective; the
process group only carries the timing barrier and the max over ranks).

  python bench.py [--steps K] [--warmup W]
                  [--config long_context|decode_batch|chunked_prefill|mixed_serving]
                  [--idx-fp4 | --idx-per-token] [--hisparse F] [--prefix-image]
  python bench.py --impl reference   # the CPU oracle on the same workload

The CPU oracle's bounded sample (cpu_baseline) runs in processes spawned
before the first CUDA call that start working only once the GPU timing is
done.  Decode workloads whose timed window would grow the mean context by
more than 1% (the decode batch) rebuild their requests at the post-warm-up
lengths, untimed, before every window.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode steps/sec (tokens/s) and achieved HBM GB/s vs 8 TB/s per config"
NOMINAL_HBM_GBS = 8000.0
# steps per timed window and warm-up steps when not given: a decode step is
# ~0.07-0.2 ms, a chunked-prefill step (the whole protocol) a few ms, a
# mixed-serving step (4 layers, 256 requests, arrivals prefilled) tens of ms
DEFAULT_STEPS = {"long_context": (1000, 10), "decode_batch": (1000, 10), "chunked_prefill": (20, 3),
                 "mixed_serving": (20, 3)}
MIN_TIMED_S = 0.5         # timed windows repeat until this much time has been timed
MAX_TIMED_STEPS = 10000   # ... or this many steps


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def workload(name, idx_fp4=False, idx_per_token=False):
    """The workload recipe; idx_fp4 stores the indexer entries in FP4 (e2m1 +
    one bf16 scale) instead of the cache dtype; idx_per_token keeps one
    indexer key per token instead of one per CSA entry."""
    from heterogeneous_compressed_kv_gb300.gen import workloads as W
    if name == "long_context":
        w = dict(W.LONG_CONTEXT)
        w["lengths"] = [w["length"]] * w["n_requests"]
    elif name == "decode_batch":
        w = dict(W.DECODE_BATCH)
        w["lengths"] = W.uniform_lengths(w["seed"], w["n_requests"], w["len_lo"], w["len_hi"]).tolist()
        w["chunk"] = 2048
    elif name == "chunked_prefill":
        w = dict(W.CHUNKED_PREFILL)
    elif name == "mixed_serving":
        w = dict(W.MIXED_SERVING)
    else:
        raise SystemExit(f"unknown config {name}")
    w["idx_fp4"] = 1 if idx_fp4 else 0
    w["idx_per_token"] = 1 if idx_per_token else 0
    return w


def dtype_label(w):
    """The arithmetic the GPU path computes in for this workload."""
    if w["cache_dtype"] == 2:  # fp8 e4m3 cache with bf16 scales
        q = ("q.k on e4m3 tensor-core MMAs (bf16 query as two exact e4m3 pieces)" if w["in_dtype"] == 1
             else "q.k as f16 x f16 products")
        return (f"e4m3 cache + bf16 scales; {q}; p.V as f16 x f16 products; fp32 accumulation and softmax; "
                "indexer scores fp32 chains of f16 x f16 products")
    if w["cache_dtype"] == 1:
        return "bf16 cache; bf16 x bf16 products (exact in fp32); fp32 accumulation and softmax"
    return "f32"


def gates(w):
    from heterogeneous_compressed_kv_gb300 import gen
    nl = w["n_layers"]
    return (gen.gate_logits(w["seed"], gen.GATE_CSA, nl, w["heads"], w["m"]),
            gen.gate_logits(w["seed"], gen.GATE_HCA, nl, w["heads"], w["m_prime"]),
            gen.gate_logits(w["seed"], gen.GATE_IDX, nl, w["idx_heads"], w["m"]))


# ---------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference); no CUDA in here
# ---------------------------------------------------------------------------
# The cpu_baseline processes are spawned before the first CUDA call but hold
# until the GPU measurements are done (the gate), so that they do not compete
# with the host thread that enqueues the GPU work.
_GATE = None


def _gate_init(gate):
    global _GATE
    _GATE = gate


def _gate_wait():
    if _GATE is not None:
        _GATE.wait()


def oracle_pool(n_workers, gated):
    """A spawned pool of n_workers processes, and the gate that releases them
    (already open when not gated)."""
    ctx = mp.get_context("spawn")
    gate = ctx.Event()
    if not gated:
        gate.set()
    return ctx.Pool(n_workers, initializer=_gate_init, initargs=(gate,)), gate


def _oracle_worker(args):
    """Prefill one workload request into the oracle (untimed), then time
    `steps` decode steps (append 1 token + decode_attend) of it."""
    name, idx_fp4, wid, steps, warm, idx_per_token = args
    _gate_wait()
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle as O
    from heterogeneous_compressed_kv_gb300 import gen
    w = workload(name, idx_fp4, idx_per_token)
    L0 = int(w["lengths"][wid])
    total = L0 + warm + steps + 1
    g = gates(w)
    o = O.Oracle(m=w["m"], m_prime=w["m_prime"], n_win=w["n_win"], heads=w["heads"], head_dim=w["head_dim"],
                 idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"],
                 cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"], max_requests=1,
                 max_blocks=total // w["m_prime"] + 1, max_blocks_per_request=total // w["m_prime"] + 1,
                 gate_csa=g[0], gate_hca=g[1], gate_idx=g[2], idx_fp4=w["idx_fp4"],
                 idx_per_token=w["idx_per_token"])
    _, r = o.alloc_request()
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    dt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16

    def vals(n, runs):
        x = gen.fill_host(n, dt, w["seed"], runs)
        return x if dt == gen.OUT_F32 else gen.bf16_bits_to_f32(x)

    def toks(p0, n):
        k = vals(n * HD, gen.token_runs(gen.K, 0, [wid], [p0], [n], HD)).reshape(1, n, HD)
        v = vals(n * HD, gen.token_runs(gen.V, 0, [wid], [p0], [n], HD)).reshape(1, n, HD)
        x = vals(n * XD, gen.token_runs(gen.IDXK, 0, [wid], [p0], [n], XD)).reshape(1, n, XD)
        return k, v, x

    t_setup = time.perf_counter()
    p = 0
    while p < L0:
        n = min(16384, L0 - p)
        assert o.append([r], [n], *toks(p, n)) == 0
        p += n
    t_setup = time.perf_counter() - t_setup

    def step(s):
        assert o.append([r], [1], *toks(L0 + s, 1)) == 0
        q = vals(HD, gen.token_runs(gen.Q, 0, [wid], [s], [1], HD))
        qi = vals(XD, gen.token_runs(gen.QIDX, 0, [wid], [s], [1], XD))
        rc, out, tk = o.decode_attend(0, [r], q.reshape(1, HD), qi.reshape(1, XD), w["top_k"])
        assert rc == 0

    for s in range(warm):
        step(s)
    t0 = time.perf_counter()
    for s in range(warm, warm + steps):
        step(s)
    return time.perf_counter() - t0, t_setup


def start_oracle(name, n_workers, steps, warm, idx_fp4=False, idx_per_token=False, gated=False):
    """Spawned before any CUDA call: one oracle process per sampled request
    (held by the gate until it is opened when gated)."""
    pool, gate = oracle_pool(n_workers, gated)
    res = pool.map_async(_oracle_worker, [(name, idx_fp4, i, steps, warm, idx_per_token) for i in range(n_workers)])
    return pool, res, gate


def oracle_workers(w):
    cores = os.cpu_count() or 1
    return max(1, min(w["n_requests"], cores - 1 if cores > 2 else 1))


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on this workload.  One
    step = one decode step (append 1 token + attend) of each sampled request,
    the requests running in parallel processes on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args.config, args.idx_fp4, args.idx_per_token)
    if args.config in ("chunked_prefill", "mixed_serving"):
        run_reference_protocol(args, w)
        return
    n = oracle_workers(w)
    pool, res, _ = start_oracle(args.config, n, args.steps, args.warmup, args.idx_fp4, args.idx_per_token)
    out = res.get()
    pool.close()
    t = max(o[0] for o in out)
    tokens = n * args.steps
    value = tokens / t
    line = dict(impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * t / args.steps, higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64 attention / f32 compressor and scores",
                data="synthetic", config=config_block(w, args),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=n, kind="oracle",
                                  sample=f"{n} of {w['n_requests']} requests (one process each) at their full "
                                         f"context; setup (oracle prefill) {max(o[1] for o in out):.0f} s untimed"),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line))


def run_reference_protocol(args, w):
    """--impl reference for chunked prefill (the whole protocol per step, one
    process; at most 3 timed steps, each ~1-2 s of oracle work) and mixed
    serving (decode steps of all 4 layers for sampled requests, one process
    each)."""
    ctx = mp.get_context("spawn")
    if args.config == "chunked_prefill":
        steps = min(args.steps, 3)
        with ctx.Pool(1) as pool:
            t = pool.map(_c3_oracle_worker, [(steps, min(args.warmup, 1))])[0]
        n, tokens = 1, (w["shared"] + w["n_requests"] * (w["tokens"] - w["shared"])) * steps
        metric, sample = METRIC + " (chunked prefill: appended tokens/s)", \
            f"{steps} runs of the whole protocol in one process; inputs drawn untimed"
    else:
        n = max(1, min(8, (os.cpu_count() or 2) - 1))
        steps = min(args.steps, 3)
        with ctx.Pool(n) as pool:
            t = max(pool.map(_c5_oracle_worker, [(i, steps) for i in range(n)]))
        tokens = n * steps
        metric, sample = METRIC + " (mixed serving: decode tokens/s)", \
            f"{n} of {w['n_requests']} requests at their initial lengths, {steps} decode steps of all 4 layers each, " \
            f"one process per request; prefill untimed"
    value = tokens / t
    line = dict(impl="reference", metric=metric, value=value, unit="tokens/s", n_gpus=args.gpus, steps=steps,
                warmup=args.warmup, ms_per_step=1e3 * t / steps, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64 attention / f32 compressor and scores", data="synthetic",
                config=config_block(w, args),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=n, kind="oracle", sample=sample),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line))


def config_block(w, args):
    c = dict(workload=w["name"], requests=w["n_requests"], heads=w["heads"], head_dim=w["head_dim"],
             indexer=f"{w['idx_heads']}x{w['idx_dim']}", m=w["m"], m_prime=w["m_prime"], n_win=w["n_win"],
             top_k=w["top_k"], in_dtype={0: "f32", 1: "bf16"}[w["in_dtype"]],
             cache_dtype={0: "f32", 1: "bf16", 2: "fp8_e4m3+bf16_scale"}[w["cache_dtype"]])
    if w.get("idx_fp4"):
        c["indexer_dtype"] = "fp4_e2m1+bf16_scale"
    if w.get("idx_per_token"):
        c["indexer_keys"] = "one per token (128 per block)"
    if getattr(args, "hisparse", 0) > 0:
        c["hisparse_offloaded"] = args.hisparse
    if w["name"] == "long_context":
        c["context"] = w["length"]
    elif w["name"] == "decode_batch":
        c["lengths"] = f"uniform[{w['len_lo']},{w['len_hi']}] seed {w['seed']}"
    elif w["name"] == "chunked_prefill":
        c.update(tokens_per_request=w["tokens"], chunk=w["chunk"], shared_prefix=w["shared"],
                 protocol="request 0: 8 chunks; 3 prefix shares; 8 rounds of 4 x 2048")
    elif w["name"] == "mixed_serving":
        c.update(layers="SWA-only, CSA, HCA, CSA",
                 lengths=f"lognormal(median {w['len_median']}, sigma {w['len_sigma']}) capped {w['len_cap']}",
                 churn=f"{w['churn']:.0%} of the requests finish and arrive per step")
    return c


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if not self.p:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=mx, reasons=sorted(reasons), samples=len(sm))


# ---------------------------------------------------------------------------
# replicas: one pool per rank, no data-path collective
# ---------------------------------------------------------------------------
def rank_env():
    """(world size, rank, local rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_wids(rank, n_requests):
    """Workload ids of this rank's requests: every rank serves its own."""
    return [rank * n_requests + i for i in range(n_requests)]


def max_over_ranks(x, world):
    """The largest value of x over the ranks (the timing of the slowest)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def traffic_record(kernel, source):
    """DRAM bytes per launch of `kernel` ("workload/kernel") from a committed
    ncu summary, only if the kernel source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    r = rec.get(kernel)
    if not r:
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()[:16]
    return r["bytes_per_launch"] if r.get("source_sha") == sha else None


# ---------------------------------------------------------------------------
# prefix images (the host-memory prefix store): export and restore bandwidth
# ---------------------------------------------------------------------------
def run_prefix_image(args):
    """Export (HBM -> page-locked host memory) and restore (host -> HBM) of one
    long-context request's sealed blocks and window as a prefix image, each
    call between CUDA events on the launching stream.  The copy engines' rate
    for the same bytes over the same link (pinned cudaMemcpyAsync) is measured
    beside them as the roofline denominator; the image is far larger than L2."""
    import torch
    from heterogeneous_compressed_kv_gb300 import gen
    from heterogeneous_compressed_kv_gb300 import kvpool as K

    w = workload("long_context", args.idx_fp4)
    L = args.context or w["length"]
    mp_ = w["m_prime"]
    L = L // mp_ * mp_
    K_, W_ = args.steps, args.warmup
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    g = gates(w)
    nb = L // mp_
    cfg = K.PoolConfig(m=w["m"], m_prime=mp_, n_win=w["n_win"], heads=w["heads"], head_dim=w["head_dim"],
                       idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"],
                       cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"], max_requests=2,
                       max_blocks=2 * nb + 2, max_blocks_per_request=nb + 1, max_batch=2, max_top_k=w["top_k"],
                       gate_csa=g[0], gate_hca=g[1], gate_idx=g[2], idx_fp4=w["idx_fp4"])
    arena = torch.empty(K.required_bytes(cfg), dtype=torch.uint8, device=dev)
    pool = K.Pool(cfg, arena, stream)
    a = pool.alloc_request()
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    tdt = torch.float32 if w["in_dtype"] == 0 else torch.bfloat16
    gdt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16
    chunk = w["chunk"]
    kb = torch.empty((1, chunk, HD), dtype=tdt, device=dev)
    vb, xb = torch.empty_like(kb), torch.empty((1, chunk, XD), dtype=tdt, device=dev)
    pool.profile_enable(True, kinds=[K.KERNEL_APPEND])
    for p0 in range(0, L, chunk):  # the prefill a restore replaces (its append kernels timed)
        c = min(chunk, L - p0)
        gen.fill_device(kb.data_ptr(), gdt, w["seed"], gen.token_runs(gen.K, 0, [0], [p0], [c], HD), sp)
        gen.fill_device(vb.data_ptr(), gdt, w["seed"], gen.token_runs(gen.V, 0, [0], [p0], [c], HD), sp)
        gen.fill_device(xb.data_ptr(), gdt, w["seed"], gen.token_runs(gen.IDXK, 0, [0], [p0], [c], XD), sp)
        pool.append([a], [c], kb, vb, xb, stream=sp)
    torch.cuda.synchronize()
    prefill_ms, prefill_launches, _ = pool.profile_read(K.KERNEL_APPEND)
    del kb, vb, xb
    pool.check_device(sp)

    n_bytes = pool.image_bytes(L, K.IMAGE_WINDOW)
    img = torch.empty(n_bytes, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(n_bytes, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    t_exp, t_imp, t_h2d, t_d2h = [], [], [], []
    clocks = Clocks(0)
    pool.profile_enable(True, kinds=[K.KERNEL_IMAGE])
    for it in range(W_ + K_):
        if it == W_:
            clocks.start()
        ev[0].record(stream)
        pool.export_prefix(a, L, K.IMAGE_WINDOW, out=img, stream=sp)
        ev[1].record(stream)
        torch.cuda.synchronize()  # the host reads the header when restoring
        b = pool.alloc_request()
        ev[2].record(stream)
        pool.import_prefix(b, img, stream=sp)
        ev[3].record(stream)
        torch.cuda.synchronize()
        if it >= W_:
            t_exp.append(ev[0].elapsed_time(ev[1]))
            t_imp.append(ev[2].elapsed_time(ev[3]))
        info_a, info_b = pool.request_info(a)[1], pool.request_info(b)[1]
        assert info_a == info_b, (info_a, info_b)
        pool.free_request(b)
    clk = clocks.stop()
    img_ms, img_launches, _ = pool.profile_read(K.KERNEL_IMAGE)
    pool.profile_enable(False)
    pool.check_device(sp)
    for it in range(W_ + K_):  # the copy engines on the same bytes and link
        ev[0].record(stream)
        dbuf.copy_(img, non_blocking=True)
        ev[1].record(stream)
        img.copy_(dbuf, non_blocking=True)
        ev[2].record(stream)
        torch.cuda.synchronize()
        if it >= W_:
            t_h2d.append(ev[0].elapsed_time(ev[1]))
            t_d2h.append(ev[1].elapsed_time(ev[2]))

    med = lambda x: float(sorted(x)[len(x) // 2])
    gbs = lambda ms: n_bytes / (ms / 1e3) / 1e9
    imp, exp_, h2d, d2h = med(t_imp), med(t_exp), med(t_h2d), med(t_d2h)
    line = dict(metric="prefix image restore bandwidth (page-locked host -> HBM)", value=gbs(imp), unit="GB/s",
                n_gpus=1, steps=K_, warmup=W_, ms_per_step=imp, higher_is_better=True, scaling="none",
                vs_baseline=None, dtype="u8", data="synthetic (seeded counter generator; no dataset)",
                config=dict(workload=f"long_context prefix image: 1 request x {L:,} tokens, "
                                     f"{'FP4' if w['idx_fp4'] else 'fp8'} indexer keys, with the SWA window",
                            image_bytes=n_bytes, blocks=nb,
                            l2="image larger than L2"),
                roofline=dict(kernel="image_copy", bound="host link", achieved=gbs(imp), peak=gbs(h2d), unit="GB/s",
                              frac=h2d / imp, traffic=None,
                              peak_source="copy engines: pinned host -> device cudaMemcpyAsync of the same bytes, "
                                          "measured in this run"),
                export=dict(ms=exp_, gbs=gbs(exp_), copy_engine_gbs=gbs(d2h), frac=d2h / exp_),
                prefill=dict(ms=prefill_ms, launches=prefill_launches,
                             note="append kernels of the same tokens (the work a restore skips; no model forward)"),
                kernel_ms_per_call=img_ms / max(1, 2 * (W_ + K_)), gpu_launches=img_launches, clocks=clk)
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# chunked prefill: appended tokens/s of the shared-prefix prefill protocol
# ---------------------------------------------------------------------------
def _oracle_of(w, max_requests, max_blocks, mbpr):
    import oracle as O
    g = gates(w)
    return O.Oracle(m=w["m"], m_prime=w["m_prime"], n_win=w["n_win"], heads=w["heads"], head_dim=w["head_dim"],
                    idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"],
                    cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"], max_requests=max_requests,
                    max_blocks=max_blocks, max_blocks_per_request=mbpr, gate_csa=g[0], gate_hca=g[1],
                    gate_idx=g[2], idx_fp4=w.get("idx_fp4", 0), idx_per_token=w.get("idx_per_token", 0))


def _host_tokens(w, wids, pos0s, counts, layers=None):
    """K, V, indexer keys [n_layers][sum counts][width] as fp32 values of the
    input dtype, for workload requests `wids` at [pos0, pos0 + count)."""
    import numpy as np
    from heterogeneous_compressed_kv_gb300 import gen
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    dt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16_F32
    T = int(sum(counts))
    layers = range(w["n_layers"]) if layers is None else layers
    out = []
    for kind, width in ((gen.K, HD), (gen.V, HD), (gen.IDXK, XD)):
        a = np.empty((len(layers), T, width), np.float32)
        for j, l in enumerate(layers):
            gen.fill_host(T * width, dt, w["seed"], gen.token_runs(kind, l, wids, pos0s, counts, width),
                          a[j].reshape(-1))
        out.append(a)
    return out


def _c3_oracle_worker(args):
    """The chunked-prefill protocol on the CPU oracle: inputs drawn untimed,
    then `steps` timed runs of the protocol (each: 4 requests allocated, 16 +
    8 appends and 3 prefix shares, all freed)."""
    steps, warm = args
    _gate_wait()
    sys.path.insert(0, ROOT)
    import numpy as np
    w = workload("chunked_prefill")
    B, T, C, S, mp_, W = w["n_requests"], w["tokens"], w["chunk"], w["shared"], w["m_prime"], w["n_win"]
    o = _oracle_of(w, B, S // mp_ + B * ((T - S) // mp_ + 2), T // mp_ + 4)
    first = _host_tokens(w, [0], [0], [S])
    rounds = [_host_tokens(w, list(range(B)), [S + r * C] * B, [C] * B) for r in range((T - S) // C)]
    win = (np.ascontiguousarray(first[0][:, S - W:S]), np.ascontiguousarray(first[1][:, S - W:S]))

    def step():
        slots = [o.alloc_request()[1] for _ in range(B)]
        for c in range(S // C):
            sl = slice(c * C, (c + 1) * C)
            assert o.append([slots[0]], [C], first[0][:, sl], first[1][:, sl], first[2][:, sl]) == 0
        for d in slots[1:]:
            assert o.share_prefix(d, slots[0], S, win[0], win[1]) == 0
        for k, v, x in rounds:
            assert o.append(slots, [C] * B, k, v, x) == 0
        for r in slots:
            o.free_request(r)

    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    return time.perf_counter() - t0


def run_chunked_prefill(args):
    """Chunked prefill with a shared prefix ("Ch 12 Inference framework:
    heterogeneous KV scheduling" s2.2: the Block cache shared by refcount):
    request 0 appends 16,384 tokens in 2,048-token chunks, requests 1-3 share
    those 128 sealed blocks (their windows recomputed by the caller), then
    8 rounds append 2,048 tokens to each of the 4 requests in one call.  One
    step = the whole protocol (81,920 appended tokens, 3 shares; the
    requests are freed at the end, host bookkeeping only); value = appended
    tokens/s with every input resident in HBM."""
    import numpy as np
    world, rank, local = rank_env()
    w = workload("chunked_prefill")
    B, T, C, S, mp_, W = w["n_requests"], w["tokens"], w["chunk"], w["shared"], w["m_prime"], w["n_win"]
    R = (T - S) // C
    tokens_per_step = S + B * (T - S)
    K_, W_ = args.steps, args.warmup
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpool, gate = oracle_pool(1, gated=True)
        cpu = (cpool, cpool.map_async(_c3_oracle_worker, [(1, 0)]), gate)

    import torch
    import torch.distributed as dist
    from heterogeneous_compressed_kv_gb300 import gen
    from heterogeneous_compressed_kv_gb300 import kvpool as K

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("gloo", rank=rank, world_size=world)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    g = gates(w)
    cfg = K.PoolConfig(m=w["m"], m_prime=mp_, n_win=W, heads=w["heads"], head_dim=w["head_dim"],
                       idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"],
                       cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"], max_requests=B,
                       max_blocks=S // mp_ + B * ((T - S) // mp_ + 2), max_blocks_per_request=T // mp_ + 4,
                       max_batch=B, max_top_k=w["top_k"], gate_csa=g[0], gate_hca=g[1], gate_idx=g[2])
    arena = torch.empty(K.required_bytes(cfg), dtype=torch.uint8, device=dev)
    pool = K.Pool(cfg, arena, stream)
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    tdt = torch.float32 if w["in_dtype"] == 0 else torch.bfloat16
    gdt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16
    wids = [rank * B + i for i in range(B)]
    # every input of a step in one device buffer: request 0's shared half, then
    # each round's 4 x 2048 tokens (K, V, indexer keys of each call adjacent)
    row = 2 * HD + XD
    calls = [([wids[0]], [0], [S])] + [(wids, [S + r * C] * B, [C] * B) for r in range(R)]
    offs, n_el = [], 0
    for _, _, cnt in calls:
        offs.append(n_el)
        n_el += sum(cnt) * row
    din = torch.empty(n_el, dtype=tdt, device=dev)

    def views(buf):
        out = []
        for (wd, p0, cnt), o0 in zip(calls, offs):
            n = sum(cnt)
            k = buf[o0:o0 + n * HD].view(1, n, HD)
            v = buf[o0 + n * HD:o0 + 2 * n * HD].view(1, n, HD)
            x = buf[o0 + 2 * n * HD:o0 + n * row].view(1, n, XD)
            out.append((k, v, x))
        return out

    for (wd, p0, cnt), (k, v, x) in zip(calls, views(din)):
        gen.fill_device(k.data_ptr(), gdt, w["seed"], gen.token_runs(gen.K, 0, wd, p0, cnt, HD), sp)
        gen.fill_device(v.data_ptr(), gdt, w["seed"], gen.token_runs(gen.V, 0, wd, p0, cnt, HD), sp)
        gen.fill_device(x.data_ptr(), gdt, w["seed"], gen.token_runs(gen.IDXK, 0, wd, p0, cnt, XD), sp)
    torch.cuda.synchronize()

    def step(vs):
        slots = [pool.alloc_request() for _ in range(B)]
        k0, v0, x0 = vs[0]
        for c in range(S // C):
            pool.append([slots[0]], [C], k0[:, c * C:(c + 1) * C], v0[:, c * C:(c + 1) * C],
                        x0[:, c * C:(c + 1) * C], stream=sp)
        for d in slots[1:]:  # the recomputed window: request 0's last W tokens of the prefix
            pool.share_prefix(d, slots[0], S, k0[:, S - W:S], v0[:, S - W:S], stream=sp)
        for k, v, x in vs[1:]:
            pool.append(slots, [C] * B, k, v, x, stream=sp)
        for sl in slots:
            pool.free_request(sl)

    dv = views(din)
    pool.profile_enable(True)
    for _ in range(W_):
        step(dv)
    torch.cuda.synchronize()
    pool.check_device(sp)
    max_windows = max(1, MAX_TIMED_STEPS // K_)
    clocks = Clocks(local)
    pool.profile_enable(True, kinds=[K.KERNEL_APPEND])
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    windows = []
    clocks.start()
    time.sleep(0.05)
    while True:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(K_):
            step(dv)
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        windows.append(max_over_ranks(ev0.elapsed_time(ev1), world))
        if sum(windows) >= 1e3 * MIN_TIMED_S or len(windows) >= max_windows:
            break
    clk = clocks.stop()
    ms = statistics.median(windows)
    a_ms, a_n, a_b = pool.profile_read(K.KERNEL_APPEND)
    n_steps_timed = len(windows) * K_
    pool.profile_enable(False)
    pool.check_device(sp)

    # end to end: each step's inputs copied from one pinned host buffer, the
    # device error word read back
    hin = din.cpu().pin_memory()
    lay = pool.layout()
    err_view = arena[lay["error_offset"]:lay["error_offset"] + 4]
    hout = torch.empty(4, dtype=torch.uint8).pin_memory()
    e2e_windows = []
    for _ in range(W_):
        din.copy_(hin, non_blocking=True)
        step(dv)
        hout.copy_(err_view, non_blocking=True)
    torch.cuda.synchronize()
    while True:
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(K_):
            din.copy_(hin, non_blocking=True)
            step(dv)
            hout.copy_(err_view, non_blocking=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        e2e_windows.append(max_over_ranks(ev0.elapsed_time(ev1), world))
        if sum(e2e_windows) >= 1e3 * MIN_TIMED_S / 2 or len(e2e_windows) >= max_windows:
            break
    pool.check_device(sp)
    e2e_ms = statistics.median(e2e_windows)
    if cpu is not None:  # the GPU measurements are done: release the oracle baseline
        cpu[-1].set()
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    step_bytes = a_b / n_steps_timed
    achieved = (a_b / a_n) / (a_ms / a_n / 1e3) / 1e9 if a_ms > 0 else None
    value = tokens_per_step * K_ * world / (ms / 1e3)
    line = dict(metric=METRIC + " (chunked prefill: appended tokens/s)", value=value, unit="tokens/s",
                n_gpus=world, steps=K_, warmup=W_, ms_per_step=ms / K_, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype=dtype_label(w), data="synthetic (seeded counter generator; no dataset)",
                config=dict(config_block(w, args), parallelism=f"replicas x{world} (requests per GPU fixed)",
                            l2=f"inputs larger than L2: {n_el * (4 if tdt == torch.float32 else 2) / 1e6:.0f} MB "
                               f"of tokens per step"),
                appended_tokens_per_step=tokens_per_step,
                hbm_gbs=step_bytes / (ms / K_ / 1e3) / 1e9,
                hbm_frac_of_8tbs=step_bytes / (ms / K_ / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                hbm_frac_of_measured=step_bytes / (ms / K_ / 1e3) / 1e9 / hbm_peak,
                roofline=dict(kernel="append", bound="hbm", achieved=achieved, peak=hbm_peak, unit="GB/s",
                              frac=(achieved / hbm_peak) if achieved else None,
                              traffic=traffic_record("chunked_prefill/append",
                                                     "heterogeneous_compressed_kv_gb300/csrc/kvpool_append.cu"),
                              peak_source=peak_kind, bytes_per_launch=a_b / a_n if a_n else None,
                              ms_per_launch=a_ms / a_n if a_n else None),
                e2e=dict(value=tokens_per_step * K_ * world / (e2e_ms / 1e3), unit="tokens/s",
                         h2d_bytes_per_step=hin.numel() * hin.element_size(), d2h_bytes_per_step=4),
                timed_windows=dict(count=len(windows), steps_each=K_, reported="median window",
                                   ms_per_step_min=min(windows) / K_, ms_per_step_median=ms / K_,
                                   ms_per_step_max=max(windows) / K_),
                gpu_launches=round(a_n / n_steps_timed * K_), clocks=clk)
    if cpu is not None:
        cpool, cres, _ = cpu
        try:
            t = cres.get(timeout=900)[0]
            line["cpu_baseline"] = dict(value=tokens_per_step / t, unit="tokens/s", cores=1, kind="oracle",
                                        sample=f"one run of the whole protocol ({tokens_per_step} appended tokens) "
                                               f"in one process; inputs drawn untimed")
        except Exception as e:  # noqa: BLE001
            line["cpu_baseline"] = dict(value=None, unit="tokens/s", cores=1, kind="oracle",
                                        sample=f"not completed: {type(e).__name__}")
        cpool.terminate()
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# mixed serving: 4 layers of different kinds, 256 requests, 10% churn per step
# ---------------------------------------------------------------------------
def _c5_oracle_worker(args):
    """One mixed-serving request on the CPU oracle: its initial length
    prefilled untimed, then `steps` timed decode steps (append one token on
    every layer, attention on each of the 4 layers)."""
    idx, steps = args
    _gate_wait()
    sys.path.insert(0, ROOT)
    import numpy as np
    from heterogeneous_compressed_kv_gb300 import gen
    from heterogeneous_compressed_kv_gb300.gen import workloads as W
    w = workload("mixed_serving")
    lens, _, _ = W.mixed_schedule(w, 1)
    L0, mp_, C = lens[idx], w["m_prime"], w["chunk"]
    nb = (L0 + steps + 2) // mp_ + 1
    o = _oracle_of(w, 1, nb, nb)
    r = o.alloc_request()[1]
    for p0 in range(0, L0, 4 * C):
        n = min(4 * C, L0 - p0)
        assert o.append([r], [n], *_host_tokens(w, [idx], [p0], [n])) == 0
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    dt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16_F32
    t0 = time.perf_counter()
    for s in range(steps):
        assert o.append([r], [1], *_host_tokens(w, [idx], [L0 + s], [1])) == 0
        for layer in range(w["n_layers"]):
            q = gen.fill_host(HD, dt, w["seed"], gen.token_runs(gen.Q, layer, [idx], [s], [1], HD))
            qi = gen.fill_host(XD, dt, w["seed"], gen.token_runs(gen.QIDX, layer, [idx], [s], [1], XD))
            rc, _, _ = o.decode_attend(layer, [r], q.reshape(1, HD), qi.reshape(1, XD), w["top_k"])
            assert rc == 0
    return time.perf_counter() - t0


def run_mixed_serving(args):
    """Mixed serving ("Ch 12 Inference framework: heterogeneous KV
    scheduling", Figure 12-1: layers of different kinds share one Block /
    State pool): 4 layers [SWA-only, CSA, HCA, CSA], window 4096, 256
    requests with lognormal lengths; every step 10% of the requests finish
    and as many arrive, prefilled in 2,048-token chunks, then one decode step
    appends a token to every request and attends on each layer.  value =
    decode tokens/s over the decode part of the steps (between CUDA events on
    the launching stream); the arrivals' prefill is reported as append
    throughput."""
    import numpy as np
    from heterogeneous_compressed_kv_gb300.gen import workloads as W
    world, rank, local = rank_env()
    w = workload("mixed_serving")
    B, mp_, C, nl = w["n_requests"], w["m_prime"], w["chunk"], w["n_layers"]
    K_, W_ = args.steps, args.warmup
    n_steps = w["decode_steps"]  # the protocol's 200 decode steps
    lens, plan, peak = W.mixed_schedule(w, n_steps)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_w = max(1, min(8, (os.cpu_count() or 2) - 1))
        cpool, gate = oracle_pool(n_w, gated=True)
        cpu = (n_w, cpool, cpool.map_async(_c5_oracle_worker, [(i, args.cpu_steps) for i in range(n_w)]), gate)

    import torch
    import torch.distributed as dist
    from heterogeneous_compressed_kv_gb300 import gen
    from heterogeneous_compressed_kv_gb300 import kvpool as K

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("gloo", rank=rank, world_size=world)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    g = gates(w)
    cfg = K.PoolConfig(m=w["m"], m_prime=mp_, n_win=w["n_win"], heads=w["heads"], head_dim=w["head_dim"],
                       idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"],
                       cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"], max_requests=B,
                       max_blocks=peak + B + 64, max_blocks_per_request=(w["len_cap"] + n_steps) // mp_ + 2,
                       max_batch=B, max_top_k=w["top_k"], gate_csa=g[0], gate_hca=g[1], gate_idx=g[2])
    arena = torch.empty(K.required_bytes(cfg), dtype=torch.uint8, device=dev)
    pool = K.Pool(cfg, arena, stream)
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    tdt = torch.float32 if w["in_dtype"] == 0 else torch.bfloat16
    gdt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16
    seed = w["seed"]
    wid_off = rank * 1_000_000  # every rank serves its own requests

    # prefill buffers: one round of at most B requests x C tokens, every layer
    # ([layer][T][width] views of flat buffers, T the round's tokens)
    fk = torch.empty(nl * B * C * HD, dtype=tdt, device=dev)
    fv, fx = torch.empty_like(fk), torch.empty(nl * B * C * XD, dtype=tdt, device=dev)

    def prefill(slots, wids, lengths):
        """Append `lengths` tokens to fresh requests in rounds of C tokens each."""
        done = [0] * len(slots)
        while True:
            sel = [j for j in range(len(slots)) if done[j] < lengths[j]]
            if not sel:
                break
            cnt = [min(C, lengths[j] - done[j]) for j in sel]
            ws, ps = [wids[j] + wid_off for j in sel], [done[j] for j in sel]
            T = sum(cnt)
            kk, vv = fk[:nl * T * HD].view(nl, T, HD), fv[:nl * T * HD].view(nl, T, HD)
            xx = fx[:nl * T * XD].view(nl, T, XD)
            for layer in range(nl):
                gen.fill_device(kk[layer].data_ptr(), gdt, seed, gen.token_runs(gen.K, layer, ws, ps, cnt, HD), sp)
                gen.fill_device(vv[layer].data_ptr(), gdt, seed, gen.token_runs(gen.V, layer, ws, ps, cnt, HD), sp)
                gen.fill_device(xx[layer].data_ptr(), gdt, seed, gen.token_runs(gen.IDXK, layer, ws, ps, cnt, XD), sp)
            pool.append([slots[j] for j in sel], cnt, kk, vv, xx, stream=sp)
            for j, c in zip(sel, cnt):
                done[j] += c
        return sum(lengths)

    t_setup = time.perf_counter()
    slots = [pool.alloc_request() for _ in range(B)]
    assert slots == list(range(B))
    wid_of = {s: s for s in range(B)}
    cur = {s: L for s, L in enumerate(lens)}
    prefill(slots, [wid_of[s] for s in slots], [cur[s] for s in slots])
    torch.cuda.synchronize()
    pool.check_device(sp)
    t_setup = time.perf_counter() - t_setup

    # decode inputs of one step, [layer][n][...] views of one flat buffer (the
    # end-to-end steps refill it from pinned host memory inside the bracket)
    n_in = nl * B * (3 * HD + 2 * XD)
    dflat = torch.empty(n_in, dtype=tdt, device=dev)
    out = torch.empty((nl, B, HD), dtype=torch.float32, device=dev)
    hin = torch.empty(n_in, dtype=tdt).pin_memory()
    hout = torch.empty((nl, B, HD), dtype=torch.float32).pin_memory()

    def dviews(n):
        o, res = 0, []
        for width in (HD, HD, XD, HD, XD):
            res.append(dflat[o:o + nl * n * width].view(nl, n, width))
            o += nl * n * width
        return res, o

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dec_ms, dec_bytes, dec_launches, pre_ms, pre_bytes, pre_tokens = [], [], [], 0.0, 0, 0
    e2e_ms, e2e_h2d, e2e_d2h = [], 0, 0
    clocks = Clocks(local)
    clk = None
    timed_target = 1e3 * MIN_TIMED_S
    phase = "warm"
    for step in range(n_steps):
        gone, arrivals = plan[step]
        for sl in gone:
            pool.free_request(sl)
            del cur[sl]
        if arrivals:
            for sl, wid, L in arrivals:
                assert pool.alloc_request() == sl
                wid_of[sl] = wid
                cur[sl] = L
            pool.profile_enable(True, kinds=[K.KERNEL_APPEND])
            pre_tok = prefill([a[0] for a in arrivals], [a[1] for a in arrivals], [a[2] for a in arrivals])
            a_ms, _, a_b = pool.profile_read(K.KERNEL_APPEND)
            if phase != "warm":
                pre_ms += a_ms
                pre_bytes += a_b
                pre_tokens += pre_tok
        act = sorted(cur)
        n = len(act)
        ws = [wid_of[sl] + wid_off for sl in act]
        pos = [cur[sl] for sl in act]
        (dk, dv, dx, dq, dqi), n_used = dviews(n)
        for layer in range(nl):
            for kind, buf, width in ((gen.K, dk, HD), (gen.V, dv, HD), (gen.IDXK, dx, XD)):
                gen.fill_device(buf[layer].data_ptr(), gdt, seed, gen.token_runs(kind, layer, ws, pos, [1] * n, width), sp)
            for kind, buf, width in ((gen.Q, dq, HD), (gen.QIDX, dqi, XD)):
                gen.fill_device(buf[layer].data_ptr(), gdt, seed,
                                gen.token_runs(kind, layer, ws, [step] * n, [1] * n, width), sp)
        if phase == "warm" and step >= W_:
            phase = "timed"
            clocks.start()
        if phase == "e2e":  # the step's inputs go to pinned host memory first (untimed)
            hin[:n_used].copy_(dflat[:n_used])
        pool.profile_enable(True, kinds=[], count=True)
        ids = np.asarray(act, np.int32)
        torch.cuda.synchronize()
        ev0.record(stream)
        if phase == "e2e":  # inputs from pinned host memory, outputs back, inside the bracket
            dflat[:n_used].copy_(hin[:n_used], non_blocking=True)
            e2e_h2d = n_used * dflat.element_size()
        pool.append(ids, np.ones(n, np.int32), dk, dv, dx, stream=sp)
        for layer in range(nl):
            pool.decode_attend(layer, ids, dq[layer], dqi[layer], w["top_k"], out[layer], None, stream=sp)
        if phase == "e2e":
            hout.copy_(out, non_blocking=True)
            e2e_d2h = out.numel() * 4
        ev1.record(stream)
        torch.cuda.synchronize()
        for sl in act:
            cur[sl] += 1
        t = ev0.elapsed_time(ev1)
        if phase == "timed":
            dec_ms.append(t)
            dec_bytes.append(sum(pool.profile_read(kk)[2] for kk in range(len(K.KERNEL_NAMES))))
            dec_launches.append(sum(pool.profile_read(kk)[1] for kk in range(len(K.KERNEL_NAMES))))
            if len(dec_ms) % K_ == 0 and sum(dec_ms) >= timed_target:
                phase = "e2e"
                clk = clocks.stop()
        elif phase == "e2e":
            e2e_ms.append(t)
            if len(e2e_ms) % K_ == 0 and sum(e2e_ms) >= timed_target / 2:
                break
    pool.profile_enable(False)
    pool.check_device(sp)
    if cpu is not None:  # the GPU measurements are done: release the oracle baseline
        cpu[-1].set()
    if phase == "timed":
        clk = clocks.stop()
    if rank != 0:
        return
    nwin = max(1, len(dec_ms) // K_)
    windows = [sum(dec_ms[i * K_:(i + 1) * K_]) for i in range(nwin)] if len(dec_ms) >= K_ else [sum(dec_ms)]
    steps_each = K_ if len(dec_ms) >= K_ else len(dec_ms)
    ms = statistics.median(windows)
    step_bytes = sum(dec_bytes) / len(dec_bytes)
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    gbs = step_bytes / (ms / steps_each / 1e3) / 1e9
    e2e_val = None
    if e2e_ms:
        e2e_val = B * len(e2e_ms) / (sum(e2e_ms) / 1e3)
    line = dict(metric=METRIC + " (mixed serving: decode tokens/s)", value=B * steps_each * world / (ms / 1e3),
                unit="tokens/s", n_gpus=world, steps=steps_each, warmup=W_, ms_per_step=ms / steps_each,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype=dtype_label(w),
                data="synthetic (seeded counter generator; no dataset)",
                config=dict(config_block(w, args), parallelism=f"replicas x{world} (requests per GPU fixed)",
                            l2=f"inputs larger than L2: {step_bytes / 1e9:.1f} GB algorithmic per decode step"),
                hbm_gbs=gbs, hbm_frac_of_8tbs=gbs / NOMINAL_HBM_GBS, hbm_frac_of_measured=gbs / hbm_peak,
                roofline=dict(kernel="decode step (append + 4 layers of attention)", bound="hbm", achieved=gbs,
                              peak=hbm_peak, unit="GB/s", frac=gbs / hbm_peak, traffic=None, peak_source=peak_kind,
                              bytes_per_launch=step_bytes, ms_per_launch=ms / steps_each),
                prefill=dict(tokens=pre_tokens, ms=pre_ms, tokens_per_s=(pre_tokens / (pre_ms / 1e3)) if pre_ms else None,
                             gbs=(pre_bytes / (pre_ms / 1e3) / 1e9) if pre_ms else None,
                             note="arrivals' prefill in 2048-token rounds, append launches between CUDA events"),
                e2e=dict(value=e2e_val, unit="tokens/s", h2d_bytes_per_step=e2e_h2d, d2h_bytes_per_step=e2e_d2h),
                timed_windows=dict(count=len(windows), steps_each=steps_each, reported="median window",
                                   ms_per_step_min=min(windows) / steps_each, ms_per_step_median=ms / steps_each,
                                   ms_per_step_max=max(windows) / steps_each),
                gpu_launches=round(sum(dec_launches) / len(dec_launches) * steps_each), setup_s=t_setup,
                clocks=clk)
    if cpu is not None:
        n_w, cpool, cres, _ = cpu
        try:
            t = max(cres.get(timeout=900))
            line["cpu_baseline"] = dict(value=n_w * args.cpu_steps / t, unit="tokens/s", cores=n_w, kind="oracle",
                                        sample=f"{n_w} of {B} requests at their initial lengths, {args.cpu_steps} "
                                               f"decode steps of all 4 layers each, one process per request; "
                                               f"prefill untimed")
        except Exception as e:  # noqa: BLE001
            line["cpu_baseline"] = dict(value=None, unit="tokens/s", cores=n_w, kind="oracle",
                                        sample=f"not completed: {type(e).__name__}")
        cpool.terminate()
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="steps per timed window (default: per config)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default: per config)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="long_context",
                    choices=["long_context", "decode_batch", "chunked_prefill", "mixed_serving"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-steps", type=int, default=3)
    ap.add_argument("--requests", type=int, default=0, help="override the request count (profiling cases)")
    ap.add_argument("--context", type=int, default=0, help="override the long-context length (profiling cases)")
    ap.add_argument("--timeline", type=int, default=0, help="print the launch timeline of this many extra steps")
    ap.add_argument("--idx-fp4", action="store_true", help="indexer entries in FP4 (e2m1 + one bf16 scale)")
    ap.add_argument("--idx-per-token", action="store_true", help="one indexer key per token instead of per CSA entry")
    ap.add_argument("--hisparse", type=float, default=0.0,
                    help="HiSparse: offload this fraction of the sealed blocks' CSA entries to host memory first")
    ap.add_argument("--prefix-image", action="store_true",
                    help="time prefix image export / restore of one long-context request instead of decode steps")
    args = ap.parse_args()
    steps0, warm0 = DEFAULT_STEPS[args.config]
    args.steps = steps0 if args.steps is None else args.steps
    args.warmup = warm0 if args.warmup is None else args.warmup
    if args.prefix_image:
        run_prefix_image(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.config == "chunked_prefill":
        run_chunked_prefill(args)
        return
    if args.config == "mixed_serving":
        run_mixed_serving(args)
        return

    world, rank, local = rank_env()
    w = workload(args.config, args.idx_fp4, args.idx_per_token)
    if args.requests or args.context:
        w["n_requests"] = args.requests or w["n_requests"]
        L = args.context or w.get("length", 0)
        w["lengths"] = [L] * w["n_requests"] if args.context else list(w["lengths"])[:w["n_requests"]]
        w["length"] = L
        args.no_cpu_baseline = True

    # the oracle baseline is spawned before the first CUDA call
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = (oracle_workers(w),) + start_oracle(args.config, oracle_workers(w), args.cpu_steps, 1, args.idx_fp4,
                                                         args.idx_per_token, gated=True)

    import numpy as np
    import torch
    import torch.distributed as dist
    from heterogeneous_compressed_kv_gb300 import gen
    from heterogeneous_compressed_kv_gb300 import kvpool as K

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("gloo", rank=rank, world_size=world)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    B, K_, W_ = w["n_requests"], args.steps, args.warmup
    lengths = [int(x) for x in w["lengths"]]
    mp_ = w["m_prime"]
    # the timed window of K steps repeats until MIN_TIMED_S have been timed
    # (at most MAX_TIMED_STEPS steps); every window appends K tokens
    max_windows = max(1, MAX_TIMED_STEPS // K_)
    extra = 3 * (K_ + W_) + 2 * K_ * max_windows + args.timeline + 2
    mbpr = (max(lengths) + extra) // mp_ + 2
    g = gates(w)
    cfg = K.PoolConfig(m=w["m"], m_prime=mp_, n_win=w["n_win"], heads=w["heads"], head_dim=w["head_dim"],
                       idx_heads=w["idx_heads"], idx_dim=w["idx_dim"], in_dtype=w["in_dtype"],
                       cache_dtype=w["cache_dtype"], layer_kinds=w["layer_kinds"], max_requests=B,
                       max_blocks=sum((L + extra) // mp_ + 1 for L in lengths), max_blocks_per_request=mbpr,
                       max_batch=B, max_top_k=w["top_k"], gate_csa=g[0], gate_hca=g[1], gate_idx=g[2],
                       idx_fp4=w["idx_fp4"], idx_per_token=w["idx_per_token"])
    n_sealed = sum(L // mp_ for L in lengths)
    if args.hisparse > 0:  # every block gets a GPU slot; a fraction moves to host slots after the prefill
        cfg.csa_hot_slots = cfg.max_blocks
        cfg.csa_host_slots = n_sealed
    arena = torch.empty(K.required_bytes(cfg), dtype=torch.uint8, device=dev)
    pool = K.Pool(cfg, arena, stream)
    host_slots = pool.set_host_pool() if args.hisparse > 0 else None
    slots = [pool.alloc_request() for _ in range(B)]
    wids = replica_wids(rank, B)
    HD, XD = w["heads"] * w["head_dim"], w["idx_heads"] * w["idx_dim"]
    tdt = torch.float32 if w["in_dtype"] == 0 else torch.bfloat16
    gdt = gen.OUT_F32 if w["in_dtype"] == 0 else gen.OUT_BF16
    seed = w["seed"]

    # ---- untimed prefill, in chunks, inputs generated on the device ----
    chunk = w["chunk"]
    kbuf = torch.empty((1, B * chunk, HD), dtype=tdt, device=dev)
    vbuf, xbuf = torch.empty_like(kbuf), torch.empty((1, B * chunk, XD), dtype=tdt, device=dev)

    def prefill(target):
        """Every request from empty to target[i] tokens (positions 0 ..
        target[i] - 1 of its input streams, which the decode steps continue)."""
        pos = [0] * B
        while True:
            cnt = [min(chunk, L - p) for L, p in zip(target, pos)]
            if sum(cnt) == 0:
                break
            gen.fill_device(kbuf.data_ptr(), gdt, seed, gen.token_runs(gen.K, 0, wids, pos, cnt, HD), sp)
            gen.fill_device(vbuf.data_ptr(), gdt, seed, gen.token_runs(gen.V, 0, wids, pos, cnt, HD), sp)
            gen.fill_device(xbuf.data_ptr(), gdt, seed, gen.token_runs(gen.IDXK, 0, wids, pos, cnt, XD), sp)
            pool.append(slots, cnt, kbuf, vbuf, xbuf, stream=sp)
            pos = [p + c for p, c in zip(pos, cnt)]
        torch.cuda.synchronize()
        pool.check_device(sp)

    t_setup = time.perf_counter()
    prefill(lengths)
    t_setup = time.perf_counter() - t_setup
    # Every step appends a token to every request.  Where a window's K tokens
    # are more than 1% of the mean context (the decode batch: U[1, 8192]), the
    # requests are rebuilt untimed at their post-warm-up lengths before each
    # timed window, so every window measures the workload's own lengths
    # (L .. L + K) instead of lengths that grew over the earlier windows.
    rebuild = args.hisparse == 0 and K_ > 0.01 * (sum(lengths) / B)
    if not rebuild:
        del kbuf, vbuf, xbuf
    n_rebuilds = 0

    def restore():
        nonlocal n_rebuilds
        if not rebuild:
            return
        for s_ in slots:
            pool.free_request(s_)
        assert [pool.alloc_request() for _ in range(B)] == slots
        prefill([L + W_ for L in lengths])
        n_rebuilds += 1

    # ---- HiSparse: offload an evenly spread fraction of every request's sealed blocks ----
    hisparse = None
    if args.hisparse > 0:
        off = []
        for s_ in slots:
            ids = pool.request_info(s_)[2]
            nb = len(ids)
            off += [int(ids[j]) for j in range(nb) if int((j + 1) * args.hisparse) != int(j * args.hisparse)]
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o0.record(stream)
        pool.offload(off, stream=sp)
        o1.record(stream)
        torch.cuda.synchronize()
        pool.check_device(sp)
        mv = len(off) * pool.host_slot_bytes()
        hisparse = dict(fraction=args.hisparse, offloaded_blocks=len(off), sealed_blocks=n_sealed,
                        offload_ms=o0.elapsed_time(o1), offload_gbs=mv / (o0.elapsed_time(o1) / 1e3) / 1e9,
                        hbm_freed_gb=mv / 1e9,
                        host_entry_bytes_per_step=round(args.hisparse * B * w["top_k"] * (2 * HD + 4)))

    # ---- step inputs, resident in HBM before timing ----
    S = 2 * (W_ + K_)  # device-timed steps then the end-to-end steps

    def step_inputs(s0, n):
        k = torch.empty((n, 1, B, HD), dtype=tdt, device=dev)
        v, x = torch.empty_like(k), torch.empty((n, 1, B, XD), dtype=tdt, device=dev)
        q, qi = torch.empty((n, B, HD), dtype=tdt, device=dev), torch.empty((n, B, XD), dtype=tdt, device=dev)
        for t in range(n):
            p = [L + s0 + t for L in lengths]
            one = [1] * B
            gen.fill_device(k[t].data_ptr(), gdt, seed, gen.token_runs(gen.K, 0, wids, p, one, HD), sp)
            gen.fill_device(v[t].data_ptr(), gdt, seed, gen.token_runs(gen.V, 0, wids, p, one, HD), sp)
            gen.fill_device(x[t].data_ptr(), gdt, seed, gen.token_runs(gen.IDXK, 0, wids, p, one, XD), sp)
            st = [s0 + t] * B
            gen.fill_device(q[t].data_ptr(), gdt, seed, gen.token_runs(gen.Q, 0, wids, st, one, HD), sp)
            gen.fill_device(qi[t].data_ptr(), gdt, seed, gen.token_runs(gen.QIDX, 0, wids, st, one, XD), sp)
        return k, v, x, q, qi

    sk, sv, sx, sq, sqi = step_inputs(0, W_ + K_)
    out = torch.empty((B, HD), dtype=torch.float32, device=dev)
    top_k = w["top_k"]
    slot_ids, one = np.asarray(slots, np.int32), np.ones(B, np.int32)  # converted once, not every call

    # every step's input views made once, outside the timed loops (a tensor
    # view costs about a microsecond of host time per input)
    views = {}

    def step(t, k, v, x, q, qi):
        key = (id(k), t)
        vw = views.get(key)
        if vw is None:
            vw = views[key] = (k[t], v[t], x[t], q[t], qi[t])
        pool.append(slot_ids, one, vw[0], vw[1], vw[2], stream=sp)
        pool.decode_attend(0, slot_ids, vw[3], vw[4], top_k, out, None, stream=sp)

    for t in range(W_ + K_):
        views[(id(sk), t)] = (sk[t], sv[t], sx[t], sq[t], sqi[t])

    # warm-up, every kernel kind recorded: the dominant kernel is the one with
    # the most algorithmic bytes
    pool.profile_enable(True)
    for t in range(W_):
        step(t, sk, sv, sx, sq, sqi)
    torch.cuda.synchronize()
    warm = {n: pool.profile_read(i) for i, n in enumerate(K.KERNEL_NAMES)}
    dom = max(("score", "attend", "append"), key=lambda n: warm[n][2])

    def barrier():
        if world > 1:
            dist.barrier()

    # timed region: windows of exactly K steps, each between CUDA events on the
    # launching stream with a barrier and a synchronize on both sides, repeated
    # until MIN_TIMED_S have been timed; the line reports the median window.
    # Events inside a window sit only around the dominant kernel's launches.
    clocks = Clocks(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.05)
    windows = []
    d_ms, d_n, d_b = 0.0, 0, 0
    while True:
        restore()
        pool.profile_enable(True, kinds=[K.KERNEL_NAMES.index(dom)])
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for t in range(W_, W_ + K_):
            step(t, sk, sv, sx, sq, sqi)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        windows.append(max_over_ranks(ev0.elapsed_time(ev1), world))
        a_ms, a_n, a_b = pool.profile_read(K.KERNEL_NAMES.index(dom))
        d_ms, d_n, d_b = d_ms + a_ms, d_n + a_n, d_b + a_b
        if sum(windows) >= 1e3 * MIN_TIMED_S or len(windows) >= max_windows:
            break
    clk = clocks.stop()
    ms = statistics.median(windows)
    pool.profile_enable(False)
    pool.check_device(sp)

    # host cost of a step: the enqueue time of a short burst (short enough not
    # to fill the launch queue, so the host never waits for the GPU)
    nb = min(K_, 16)
    h0 = time.perf_counter()
    for t in range(W_, W_ + nb):
        step(t, sk, sv, sx, sq, sqi)
    host_us = (time.perf_counter() - h0) / nb * 1e6
    torch.cuda.synchronize()

    # per-kernel breakdown: a second pass over the same step inputs, every
    # launch between events (the events themselves cost a little time)
    KB = min(K_, 200)
    restore()
    pool.profile_enable(True)
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for t in range(W_, W_ + KB):
        step(t, sk, sv, sx, sq, sqi)
    b1.record(stream)
    torch.cuda.synchronize()
    breakdown_ms = b0.elapsed_time(b1)
    prof = {n: pool.profile_read(i) for i, n in enumerate(K.KERNEL_NAMES)}
    pool.profile_enable(False)
    pool.check_device(sp)

    if args.timeline:
        pool.profile_enable(True)
        for t in range(args.timeline):
            step(W_ + t, sk, sv, sx, sq, sqi)
        torch.cuda.synchronize()
        tl = pool.profile_timeline()
        pool.profile_enable(False)
        for name, a, b in tl:
            print(f"timeline {name:8s} {a * 1e3:9.1f} {b * 1e3:9.1f} {1e3 * (b - a):8.1f} us", file=sys.stderr)

    # ---- end to end: pinned host inputs in, result out, every step ----
    # a step's inputs (K, V, indexer keys, query, indexer query) sit in one
    # pinned host row and move in one copy; the device views slice it
    ek, ev_, ex, eq, eqi = step_inputs(W_ + K_, W_ + K_)
    parts = [t.reshape(W_ + K_, -1) for t in (ek, ev_, ex, eq, eqi)]
    widths = [t.shape[1] for t in parts]
    hin = torch.cat(parts, dim=1).cpu().pin_memory()  # [steps][all inputs]
    del ek, ev_, ex, eq, eqi, parts
    din = torch.empty(hin.shape[1], dtype=tdt, device=dev)
    offs = [sum(widths[:j]) for j in range(5)]
    dk = din[offs[0]:offs[0] + widths[0]].view(1, 1, B, HD)
    dv = din[offs[1]:offs[1] + widths[1]].view(1, 1, B, HD)
    dx = din[offs[2]:offs[2] + widths[2]].view(1, 1, B, XD)
    dq = din[offs[3]:offs[3] + widths[3]].view(1, B, HD)
    dqi = din[offs[4]:offs[4] + widths[4]].view(1, B, XD)
    hout = torch.empty((W_ + K_, B, HD), dtype=torch.float32).pin_memory()

    def e2e_step(t):
        din.copy_(hin[t], non_blocking=True)
        step(0, dk, dv, dx, dq, dqi)
        hout[t].copy_(out, non_blocking=True)

    for t in range(W_):
        e2e_step(t)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_windows = []
    while True:  # windows of K steps as in the device-timed region (median reported)
        restore()
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for t in range(W_, W_ + K_):
            e2e_step(t)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_windows.append(max_over_ranks(e0.elapsed_time(e1), world))
        if sum(e2e_windows) >= 1e3 * MIN_TIMED_S / 2 or len(e2e_windows) >= max_windows:
            break
    e2e_ms = statistics.median(e2e_windows)
    if cpu is not None:  # the GPU measurements are done: release the oracle baseline
        cpu[-1].set()
    h2d = hin[0].numel() * hin.element_size()
    d2h = hout[0].numel() * 4

    tokens = B * K_ * world
    value = tokens / (ms / 1e3)
    e2e_value = tokens / (e2e_ms / 1e3)
    step_bytes = sum(b for (_, _, b) in prof.values()) / KB
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    src = {"score": "heterogeneous_compressed_kv_gb300/csrc/kvpool_score.cu",
           "attend": "heterogeneous_compressed_kv_gb300/csrc/kvpool_attend.cu",
           "append": "heterogeneous_compressed_kv_gb300/csrc/kvpool_append.cu"}[dom]
    launches_dom = d_n
    achieved = (d_b / launches_dom) / (d_ms / launches_dom / 1e3) / 1e9 if d_ms > 0 else None
    launches = round(sum(n for (_, n, _) in prof.values()) * K_ / KB)

    if rank != 0:
        return
    line = dict(metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=K_, warmup=W_,
                ms_per_step=ms / K_, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype=dtype_label(w), data="synthetic (seeded counter generator; no dataset)",
                config=dict(config_block(w, args), parallelism=f"replicas x{world} (requests per GPU fixed)",
                            l2=f"inputs larger than L2: {step_bytes / 1e6:.0f} MB algorithmic per step"),
                steps_per_s=K_ / (ms / 1e3),
                hbm_gbs=step_bytes / (ms / K_ / 1e3) / 1e9,
                hbm_frac_of_8tbs=step_bytes / (ms / K_ / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                hbm_frac_of_measured=step_bytes / (ms / K_ / 1e3) / 1e9 / hbm_peak,
                kernels={n: dict(ms_per_step=pm / KB, launches=pn, gb_per_step=pb / KB / 1e9,
                                 gbs=(pb / (pm / 1e3) / 1e9) if pm > 0 else None)
                         for n, (pm, pn, pb) in prof.items()},
                kernels_pass=dict(steps=KB, ms_per_step=breakdown_ms / KB,
                                  note="separate pass over the same inputs, every launch between CUDA events"),
                roofline=dict(kernel=dom, bound="hbm", achieved=achieved, peak=hbm_peak, unit="GB/s",
                              frac=(achieved / hbm_peak) if achieved else None,
                              # the records hold full-size launches: none for a resized workload
                              traffic=None if (args.requests or args.context) else
                              traffic_record(f"{w['name']}/{dom}" + ("_fp4" if dom == "score" and w["idx_fp4"] else "")
                                             + ("_per_token" if dom == "score" and w["idx_per_token"] else ""),
                                             src),
                              peak_source=peak_kind,
                              bytes_per_launch=d_b / launches_dom, ms_per_launch=d_ms / launches_dom),
                e2e=dict(value=e2e_value, unit="tokens/s", h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h),
                **({"hisparse": hisparse} if hisparse else {}),
                timed_windows=dict(count=len(windows), steps_each=K_, reported="median window",
                                   ms_per_step_min=min(windows) / K_, ms_per_step_median=ms / K_,
                                   ms_per_step_max=max(windows) / K_,
                                   lengths=(f"requests rebuilt at their post-warm-up lengths before each window "
                                            f"({n_rebuilds} rebuilds, untimed)") if rebuild else
                                   f"requests grow by one token per step ({K_} per window, < 1% of the mean context)"),
                gpu_launches=launches, setup_s=t_setup, clocks=clk, host_enqueue_us_per_step=host_us)
    if cpu is not None:
        n_w, cpool, cres, _ = cpu
        try:
            res = cres.get(timeout=900)
            t = max(r[0] for r in res)
            line["cpu_baseline"] = dict(value=n_w * args.cpu_steps / t, unit="tokens/s", cores=n_w, kind="oracle",
                                        sample=f"{n_w} of {B} requests at full context, {args.cpu_steps} decode "
                                               f"steps each, one process per request; oracle prefill "
                                               f"{max(r[1] for r in res):.0f} s untimed")
        except Exception as e:  # noqa: BLE001
            line["cpu_baseline"] = dict(value=None, unit="tokens/s", cores=n_w, kind="oracle",
                                        sample=f"not completed: {type(e).__name__}")
        cpool.terminate()
    print(json.dumps(line))


if __name__ == "__main__":
    main()
