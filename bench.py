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

  python bench.py [--steps K] [--warmup W] [--config long_context|decode_batch]
  python bench.py --impl reference   # the CPU oracle on the same workload
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
    else:
        raise SystemExit(f"unknown config {name}")
    w["idx_fp4"] = 1 if idx_fp4 else 0
    w["idx_per_token"] = 1 if idx_per_token else 0
    return w


def gates(w):
    from heterogeneous_compressed_kv_gb300 import gen
    nl = w["n_layers"]
    return (gen.gate_logits(w["seed"], gen.GATE_CSA, nl, w["heads"], w["m"]),
            gen.gate_logits(w["seed"], gen.GATE_HCA, nl, w["heads"], w["m_prime"]),
            gen.gate_logits(w["seed"], gen.GATE_IDX, nl, w["idx_heads"], w["m"]))


# ---------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference); no CUDA in here
# ---------------------------------------------------------------------------
def _oracle_worker(args):
    """Prefill one workload request into the oracle (untimed), then time
    `steps` decode steps (append 1 token + decode_attend) of it."""
    name, idx_fp4, wid, steps, warm, idx_per_token = args
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


def start_oracle(name, n_workers, steps, warm, idx_fp4=False, idx_per_token=False):
    """Spawned before any CUDA call: one oracle process per sampled request."""
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(n_workers)
    res = pool.map_async(_oracle_worker, [(name, idx_fp4, i, steps, warm, idx_per_token) for i in range(n_workers)])
    return pool, res


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
    n = oracle_workers(w)
    pool, res = start_oracle(args.config, n, args.steps, args.warmup, args.idx_fp4, args.idx_per_token)
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
    else:
        c["lengths"] = f"uniform[{w['len_lo']},{w['len_hi']}] seed {w['seed']}"
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
# the GPU arm
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="long_context", choices=["long_context", "decode_batch"])
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
    if args.prefix_image:
        run_prefix_image(args)
        return
    if args.impl == "reference":
        run_reference(args)
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
                                                         args.idx_per_token)

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
    extra = 3 * (K_ + W_) + args.timeline + 2
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
    t_setup = time.perf_counter()
    chunk = w["chunk"]
    kbuf = torch.empty((1, B * chunk, HD), dtype=tdt, device=dev)
    vbuf, xbuf = torch.empty_like(kbuf), torch.empty((1, B * chunk, XD), dtype=tdt, device=dev)
    pos = [0] * B
    while True:
        cnt = [min(chunk, L - p) for L, p in zip(lengths, pos)]
        if sum(cnt) == 0:
            break
        gen.fill_device(kbuf.data_ptr(), gdt, seed, gen.token_runs(gen.K, 0, wids, pos, cnt, HD), sp)
        gen.fill_device(vbuf.data_ptr(), gdt, seed, gen.token_runs(gen.V, 0, wids, pos, cnt, HD), sp)
        gen.fill_device(xbuf.data_ptr(), gdt, seed, gen.token_runs(gen.IDXK, 0, wids, pos, cnt, XD), sp)
        pool.append(slots, cnt, kbuf, vbuf, xbuf, stream=sp)
        pos = [p + c for p, c in zip(pos, cnt)]
    del kbuf, vbuf, xbuf
    torch.cuda.synchronize()
    pool.check_device(sp)
    t_setup = time.perf_counter() - t_setup

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

    def step(t, k, v, x, q, qi):
        pool.append(slot_ids, one, k[t], v[t], x[t], stream=sp)
        pool.decode_attend(0, slot_ids, q[t], qi[t], top_k, out, None, stream=sp)

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

    # timed region: events only around the dominant kernel's launches
    clocks = Clocks(local)
    pool.profile_enable(True, kinds=[K.KERNEL_NAMES.index(dom)])
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.05)
    ev0.record(stream)
    for t in range(W_, W_ + K_):
        step(t, sk, sv, sx, sq, sqi)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    ms = ev0.elapsed_time(ev1)
    d_ms, d_n, d_b = pool.profile_read(K.KERNEL_NAMES.index(dom))
    pool.check_device(sp)
    ms = max_over_ranks(ms, world)

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
    e0.record(stream)
    for t in range(W_, W_ + K_):
        e2e_step(t)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world)
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
                dtype="f32", data="synthetic (seeded counter generator; no dataset)",
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
                gpu_launches=launches, setup_s=t_setup, clocks=clk, host_enqueue_us_per_step=host_us)
    if cpu is not None:
        n_w, cpool, cres = cpu
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
