#!/usr/bin/env python
"""Benchmark of the MSA forward path on GB300.

Default (N=1): one JSON line for the 128K prefill step (select -> invert ->
KV-outer attention -> combine) on device-resident synthetic inputs, with a
"decode" object for the 1M-context decode step, the roofline of the dominant
kernel, sampled SM clocks, an end-to-end number through host buffers and the
fp64 oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (torchrun) every rank runs an independent replica of the step (the
path needs no exchange between GPUs); value = tokens of all ranks / max time.
--impl reference times the fp64 CPU oracle on the same workload instead.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA prefill tokens/s at 128K, decode tokens/s at 1M ctx; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="prefill_128k")
    ap.add_argument("--decode-config", default="decode_1m")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 (E4M3) index-input variants")
    ap.add_argument("--no-varlen", action="store_true", help="skip the varlen (packed sequences) prefill")
    ap.add_argument("--no-warmup", action="store_true", help="skip warmup mode (dense attention + index KL)")
    ap.add_argument("--no-other-prefill", action="store_true", help="skip the 32K and 1M prefill lines")
    ap.add_argument("--cpu-rows", type=int, default=2048, help="oracle rows timed for cpu_baseline (about 10 s)")
    ap.add_argument("--stage", default="all", choices=["all", "select", "attend", "decode", "select_fp8",
                                                       "decode_fp8", "warmup", "select_varlen"],
                    help="time one stage alone on --config (small-memory cases for profiler captures)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Dist:
    def __init__(self, use_cuda):
        import torch
        import torch.distributed as dist
        self.ws, self.rank, self.local = dist_setup()
        self.dist = dist
        self.on = self.ws > 1
        if self.on:
            dist.init_process_group(backend="nccl" if use_cuda else "gloo")

    def barrier(self):
        if self.on:
            self.dist.barrier()

    def max(self, x):
        if not self.on:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.on:
            self.dist.destroy_process_group()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while running; summarised for the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for i, n in enumerate(names):
                    if r[5 + i].lower().startswith("active"):
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- traffic from a committed ncu summary
def traffic_for(kernel_key, *src_files):
    """Per-launch DRAM bytes recorded in profiles/traffic.json for the given kernel sources' hash, else None
    (None as soon as any of those sources changed since the counters were taken)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f).get(kernel_key)
        h = hashlib.sha256()
        for src in src_files:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if d and d.get("source_sha") == h.hexdigest()[:16]:
            return d.get("bytes_per_launch")
    except (OSError, ValueError):
        return None
    return None


# --------------------------------------------------------------------------- the GPU arm
def prefill_slabs(cfg):
    """Query slabs of the attention call: one slab's partial results stay under ~36 GB."""
    per_pos = cfg.k * cfg.H_q * (2.0 * cfg.d + 8.0)
    cap = int(36.0e9 / per_pos)
    cap = max(1024, min(131072, cap))
    slab = min(cfg.N, cap)
    return (cfg.N + slab - 1) // slab


def prefill_launches(cfg):
    """Kernels libmsa launches for one msa_prefill step: select 1, invert 4, per query slab
    schedule 3, tiles 1, combine 1."""
    return 1 + 4 + 5 * prefill_slabs(cfg)


def bwd_launches(cfg):
    """Kernels libmsa launches for one msa_sparse_attn_bwd call: B* inversion 4, rowdot 1, then per query slab
    (at most 131072 positions, fewer when the G k Bk 2-byte teacher rows of a slab would pass 32 GB) the
    schedule 3, mark_repeats 1, index lse 1 and its combine 1, main 1, index gradient 1."""
    cap = int(32.0e9 / (cfg.G * cfg.k * cfg.Bk * 2.0))
    slab = min(cfg.N, max(1024, min(131072, cap)))
    return 5 + 8 * ((cfg.N + slab - 1) // slab)


def varlen_mix(N, Bk):
    """A fixed mix of sequence lengths (block multiples) filling N cells: 1/4, 3/16, 1/8, 1/8, 3/32, 3/32,
    1/16, 1/16 of N."""
    parts = [8, 6, 4, 4, 3, 3, 2, 2]  # in 32nds
    lengths = [N * p // 32 // Bk * Bk for p in parts]
    lengths[-1] += N - sum(lengths)
    return lengths


def bench_prefill(args, dist, torch, peaks):
    import datagen
    from block_sparse_long_index_gb300 import MsaPrefill
    cfg = datagen.CONFIGS[args.config]
    inp = datagen.prefill_device(cfg)
    run = MsaPrefill(cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    q, k, v, qi, ki = inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        run(q, k, v, qi, ki)
    torch.cuda.synchronize()
    if run.device_status() != 0:
        raise RuntimeError("device error during warm-up")
    K = args.steps
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # the step: msa_prefill (select, then the attention call)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = E(), E()
    t_start.record(stream)
    for _ in range(K):
        run(q, k, v, qi, ki)
    t_end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    assert run.device_status() == 0
    # the same work as two separate calls, for the per-stage durations behind the roofline objects
    for _ in range(min(args.warmup, 2)):
        run.select(qi, ki)
        run.attend(q, k, v)
    ev = [(E(), E(), E()) for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        ev[i][0].record(stream)
        run.select(qi, ki)
        ev[i][1].record(stream)
        run.attend(q, k, v)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    sel_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / K
    att_ms = sum(b.elapsed_time(c) for _, b, c in ev) / K
    assert run.device_status() == 0
    res = dict(cfg=cfg, total_ms=total_ms, sel_ms=sel_ms, att_ms=att_ms, clocks=clk)

    # ---- backward of the same step: main-branch gradients and the index branch's KL gradient
    if not args.no_backward:
        from block_sparse_long_index_gb300 import msa
        N, G = cfg.N, cfg.G
        dout = datagen.device_normal_(torch.empty((N, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda"),
                                      cfg.seed, datagen.TID["dout"])
        f32 = lambda *shp: torch.empty(shp, dtype=torch.float32, device="cuda")  # noqa: E731
        grads = (f32(N, cfg.H_q, cfg.d), f32(N, cfg.H_kv, cfg.d), f32(N, cfg.H_kv, cfg.d), f32(N, G, cfg.d_I),
                 f32(N, cfg.d_I), f32(G, N))
        wsb = torch.empty(msa.msa_sparse_attn_bwd_workspace(run.shape), dtype=torch.uint8, device="cuda")
        run(q, k, v, qi, ki)
        scale = 1.0 / math.sqrt(cfg.d)
        bwd = lambda: msa.msa_sparse_attn_bwd(q, k, v, qi, ki, run.block_idx, run.out, run.lse, dout, run.shape,  # noqa
                                              scale, 1.0, *grads, wsb)
        for _ in range(args.warmup):
            bwd()
        torch.cuda.synchronize()
        a, b = E(), E()
        a.record(stream)
        for _ in range(K):
            bwd()
        b.record(stream)
        torch.cuda.synchronize()
        assert msa.msa_check_device_error(wsb) == 0
        res["bwd_ms"] = a.elapsed_time(b) / K
        del dout, grads, wsb

    # ---- the same step on FP8 (E4M3) index inputs: msa_prefill_fp8 (q, k, v stay bf16)
    if not args.no_fp8:
        from block_sparse_long_index_gb300 import msa
        q8 = torch.empty(qi.shape, dtype=torch.uint8, device="cuda")
        k8 = torch.empty(ki.shape, dtype=torch.uint8, device="cuda")
        quant = lambda: (msa.msa_quantize_e4m3(qi, qi.numel(), 1.0, q8),  # noqa: E731
                         msa.msa_quantize_e4m3(ki, ki.numel(), 1.0, k8))
        scale = 1.0 / math.sqrt(cfg.d)
        step8 = lambda: msa.msa_prefill_fp8(q, k, v, q8, k8, run.shape, scale, run.block_idx, run.out,  # noqa
                                            run.lse, run.workspace)
        sel8 = lambda: msa.msa_select_blocks_fp8(q8, k8, cfg.N, cfg.G, cfg.d_I, cfg.Bk, cfg.k,  # noqa: E731
                                                 run.block_idx, run.workspace)
        quant()
        for _ in range(args.warmup):
            step8()
        torch.cuda.synchronize()
        tm = {}
        for name, fn in (("quant", quant), ("step", step8), ("select", sel8)):
            a, b = E(), E()
            a.record(stream)
            for _ in range(K):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            tm[name] = a.elapsed_time(b) / K
        assert run.device_status() == 0
        res["fp8"] = dict(step_ms=tm["step"], sel_ms=tm["select"], quant_ms=tm["quant"])
        del q8, k8

    # ---- the same cells as several sequences (msa_prefill_varlen): a fixed mix of lengths filling N
    if not args.no_varlen:
        from block_sparse_long_index_gb300 import msa
        lengths = varlen_mix(cfg.N, cfg.Bk)
        cu = [0]
        for n in lengths:
            cu.append(cu[-1] + n)
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        wsv = torch.empty(msa.msa_prefill_varlen_workspace(run.shape), dtype=torch.uint8, device="cuda")
        scale = 1.0 / math.sqrt(cfg.d)
        stepv = lambda: msa.msa_prefill_varlen(q, k, v, qi, ki, cu_d, len(lengths), run.shape, scale,  # noqa: E731
                                               run.block_idx, run.out, run.lse, wsv)
        selv = lambda: msa.msa_select_blocks_varlen(qi, ki, cu_d, len(lengths), cfg.N, cfg.G, cfg.d_I,  # noqa
                                                    cfg.Bk, cfg.k, run.block_idx, wsv)
        for _ in range(args.warmup):
            stepv()
        torch.cuda.synchronize()
        tv = {}
        for name, fn in (("step", stepv), ("select", selv)):
            a, b = E(), E()
            a.record(stream)
            for _ in range(K):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            tv[name] = a.elapsed_time(b) / K
        assert msa.msa_check_device_error(wsv) == 0
        res["varlen"] = dict(step_ms=tv["step"], sel_ms=tv["select"], lengths=lengths)
        del wsv

    # ---- end to end through host buffers (pinned), copies inside the timed region: every step copies
    # its five inputs in and out, lse back; PrefillHostPipeline overlaps those copies with compute
    if not args.no_e2e:
        from block_sparse_long_index_gb300.api import PrefillHostPipeline
        names = ("q", "k", "v", "q_idx", "k_idx")
        host = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in zip(names, (q, k, v, qi, ki))}
        for n, t in zip(names, (q, k, v, qi, ki)):
            host[n].copy_(t)
        del inp, q, k, v, qi, ki  # the pipeline keeps its own two device input sets
        torch.cuda.empty_cache()
        houts = [{"out": torch.empty(run.out.shape, dtype=run.out.dtype, pin_memory=True),
                  "lse": torch.empty(run.lse.shape, dtype=run.lse.dtype, pin_memory=True)} for _ in range(2)]
        pipe = PrefillHostPipeline(run)
        # at least 30 pipelined steps (about a second): on some hosts the copies of a run's first ~0.2 s go slower,
        # and a ten-step run would report that start rather than the pipeline's throughput
        Ke = max(30, K)
        pipe([host] * 2, houts)  # warm-up
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        a, b = E(), E()
        a.record(stream)
        pipe([host] * Ke, [houts[i % 2] for i in range(Ke)])
        b.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        assert run.device_status() == 0
        e2e_ms = a.elapsed_time(b) / Ke
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in houts[0].values())
        res["e2e"] = dict(ms=e2e_ms, h2d=h2d, d2h=d2h, steps=Ke)
        del pipe, host, houts
    else:
        del inp
    del run
    torch.cuda.empty_cache()
    return res


def bench_decode(args, dist, torch):
    import numpy as np

    import datagen
    from block_sparse_long_index_gb300 import MsaDecode
    cfg = datagen.CONFIGS[args.decode_config]
    inp = datagen.decode_device(cfg)
    run = MsaDecode(cfg.B, cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")  # 4x L2, rewritten between steps
    evict = torch.zeros(512 << 20, dtype=torch.uint8, device="cuda")  # then read, so the flush's dirty lines
    # are written back before the timed step starts (a cold, clean L2)

    def cold_l2(i):
        flush.fill_(i & 0xFF)
        evict.view(torch.int64).sum()

    args_ = (inp["q_t"], inp["q_idx_t"], inp["k_idx_cache"], inp["k_cache"], inp["v_cache"], inp["ctx_len"])
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        run(*args_)
    torch.cuda.synchronize()
    K = max(args.steps, 20)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(E(), E()) for _ in range(K)]
    dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        cold_l2(i)
        ev[i][0].record(stream)
        run(*args_)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    assert run.device_status() == 0
    times = sorted(a.elapsed_time(b) for a, b in ev)
    mean_ms = sum(times) / K
    res = dict(cfg=cfg, mean_ms=mean_ms, median_ms=times[K // 2], steps=K)
    # the same step right after the write-only flush: its dirty lines are written back inside the step
    evd = [(E(), E()) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        evd[i][0].record(stream)
        run(*args_)
        evd[i][1].record(stream)
    torch.cuda.synchronize()
    res["dirty_ms"] = sum(a.elapsed_time(b) for a, b in evd) / K
    # the same step over paged caches: the caches viewed as a pool of 128-token pages, each sequence's
    # pages scattered by a random page table (the bytes read are the same, in page order)
    from block_sparse_long_index_gb300 import msa
    page = 128
    mp = cfg.ctx // page
    n_pages = cfg.B * mp
    perm = torch.from_numpy(np.random.default_rng(11).permutation(n_pages).astype(np.int32)).view(cfg.B, mp).cuda()
    pools = (inp["k_idx_cache"].view(n_pages, page, cfg.d_I), inp["k_cache"].view(n_pages, page, cfg.H_kv, cfg.d),
             inp["v_cache"].view(n_pages, page, cfg.H_kv, cfg.d))
    scale = 1.0 / math.sqrt(cfg.d)
    paged = lambda: msa.msa_decode_paged(inp["q_t"], inp["q_idx_t"], pools[0], pools[1], pools[2], perm, mp,  # noqa
                                         n_pages, page, inp["ctx_len"], cfg.B, run.shape, scale, run.out, run.lse,
                                         run.block_idx, run.workspace)
    for _ in range(args.warmup):
        paged()
    torch.cuda.synchronize()
    evp = [(E(), E()) for _ in range(K)]
    for i in range(K):
        cold_l2(i)
        evp[i][0].record(stream)
        paged()
        evp[i][1].record(stream)
    torch.cuda.synchronize()
    assert run.device_status() == 0
    tp = sorted(a.elapsed_time(b) for a, b in evp)
    res["paged"] = dict(mean_ms=sum(tp) / K, median_ms=tp[K // 2], page=page)
    # the same step with an FP8 (E4M3) index-key cache and index query (msa_decode_fp8)
    if not args.no_fp8:
        ki8 = torch.empty(inp["k_idx_cache"].shape, dtype=torch.uint8, device="cuda")
        qi8 = torch.empty(inp["q_idx_t"].shape, dtype=torch.uint8, device="cuda")
        msa.msa_quantize_e4m3(inp["k_idx_cache"], ki8.numel(), 1.0, ki8)
        msa.msa_quantize_e4m3(inp["q_idx_t"], qi8.numel(), 1.0, qi8)
        dec8 = lambda: msa.msa_decode_fp8(inp["q_t"], qi8, ki8, inp["k_cache"], inp["v_cache"],  # noqa: E731
                                          inp["ctx_len"], cfg.B, run.shape, scale, run.out, run.lse, run.block_idx,
                                          run.workspace)
        for _ in range(args.warmup):
            dec8()
        torch.cuda.synchronize()
        ev8 = [(E(), E()) for _ in range(K)]
        for i in range(K):
            cold_l2(i)
            ev8[i][0].record(stream)
            dec8()
            ev8[i][1].record(stream)
        torch.cuda.synchronize()
        assert run.device_status() == 0
        t8 = sorted(a.elapsed_time(b) for a, b in ev8)
        res["fp8"] = dict(mean_ms=sum(t8) / K, median_ms=t8[K // 2])
        del ki8, qi8
    del inp, run, flush, evict
    torch.cuda.empty_cache()
    return res


def bench_prefill_other(name, args, dist, torch, steps):
    """The msa_prefill step (select, then the attention call) on another prefill workload, inputs resident;
    then the two stages as separate calls once more for their shares."""
    import datagen
    from block_sparse_long_index_gb300 import MsaPrefill
    cfg = datagen.CONFIGS[name]
    inp = datagen.prefill_device(cfg)
    run = MsaPrefill(cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    args_ = (inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"])
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        run(*args_)
    torch.cuda.synchronize()
    if run.device_status() != 0:
        raise RuntimeError("device error during warm-up (%s)" % name)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    dist.barrier()
    torch.cuda.synchronize()
    a, b = E(), E()
    a.record(stream)
    for _ in range(steps):
        run(*args_)
    b.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ms = a.elapsed_time(b) / steps
    e0, e1, e2 = E(), E(), E()
    e0.record(stream)
    run.select(inp["q_idx"], inp["k_idx"])
    e1.record(stream)
    run.attend(inp["q"], inp["k"], inp["v"])
    e2.record(stream)
    torch.cuda.synchronize()
    assert run.device_status() == 0
    res = dict(cfg=cfg, ms=ms, steps=steps, sel_ms=e0.elapsed_time(e1), att_ms=e1.elapsed_time(e2))
    del inp, run, args_
    torch.cuda.empty_cache()
    return res


WARMUP_CFG = dict(N=32768, H_q=64, H_kv=8, d=128, d_I=128, Bk=128, k=16, needles=0, index=7)


def bench_warmup(args, dist, torch):
    """Warmup mode on the 128K prefill's head shapes at N = 32K: msa_warmup_fwd, then msa_warmup_index_grad."""
    import datagen
    from block_sparse_long_index_gb300 import msa
    cfg = datagen.make_config("warmup_32k", **WARMUP_CFG)
    inp = datagen.prefill_device(cfg)
    N, G = cfg.N, cfg.G
    shp = msa.shape(N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    f32 = lambda *s_: torch.empty(s_, dtype=torch.float32, device="cuda")  # noqa: E731
    out = torch.empty((N, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
    lse, lse_idx = f32(cfg.H_q, N), f32(G, N)
    dq_idx, dk_idx, kl = f32(N, G, cfg.d_I), f32(N, cfg.d_I), f32(G, N)
    scale = 1.0 / math.sqrt(cfg.d)
    fwd = lambda: msa.msa_warmup_fwd(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], shp, scale, out,  # noqa
                                     lse, lse_idx)
    grad = lambda: msa.msa_warmup_index_grad(inp["q"], inp["k"], inp["q_idx"], inp["k_idx"], lse, lse_idx, shp,  # noqa
                                             scale, 1.0, dq_idx, dk_idx, kl)
    for _ in range(max(1, args.warmup)):
        fwd()
        grad()
    torch.cuda.synchronize()
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    stream = torch.cuda.current_stream()
    K = max(1, min(args.steps, 5))
    tm = {}
    for name, fn in (("fwd", fwd), ("grad", grad)):
        a, b = E(), E()
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        tm[name] = a.elapsed_time(b) / K
    del inp, out, lse, lse_idx, dq_idx, dk_idx, kl
    torch.cuda.empty_cache()
    return dict(cfg=cfg, fwd_ms=tm["fwd"], grad_ms=tm["grad"], steps=K)


# --------------------------------------------------------------------------- the oracle (CPU) leg
def oracle_prefill_sample(cfg, n_rows, seed=7):
    """Times the fp64 oracle (select + attention over every head) on n_rows sampled positions.
    Returns (seconds, rows, threads)."""
    import numpy as np

    import datagen
    import oracle
    rows = datagen.sample_rows(cfg.N, n_rows, seed)
    host = datagen.prefill_host(cfg, rows=rows)
    th = oracle.threads()
    t0 = time.perf_counter()
    blk, _ = oracle.select_blocks(host["q_idx"], host["k_idx"], rows, cfg.N, cfg.Bk, cfg.k, n_threads=th)
    oracle.sparse_attn(host["q"], host["k"], host["v"], blk, rows, cfg.Bk, 1.0 / math.sqrt(cfg.d), n_threads=th)
    dt = time.perf_counter() - t0
    return dt, len(rows), th


def run_reference(args):
    """--impl reference: the fp64 oracle on the host cores, same metric and workload."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import datagen
    cfg = datagen.CONFIGS[args.config]
    rows_per_step = 96
    for i in range(args.warmup):
        oracle_prefill_sample(cfg, rows_per_step // 4, seed=100 + i)
    total_s, total_rows, th = 0.0, 0, 1
    for i in range(args.steps):
        dt, n, th = oracle_prefill_sample(cfg, rows_per_step, seed=200 + i)
        total_s += dt
        total_rows += n
    value = total_rows / total_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(cfg), "sample": "%d seeded query rows per step" % rows_per_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": th, "kind": "oracle",
                             "sample": "%d rows x %d steps of the %s workload (select over all groups + "
                                       "attention over all heads per row)" % (rows_per_step, args.steps, cfg.name)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_name(cfg):
    if cfg.kind == "prefill":
        return ("%s: prefill N=%d H_q=%d H_kv=%d d=%d d_I=%d Bk=%d k=%d, %d needle blocks/group"
                % (cfg.name, cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k, cfg.needles))
    return ("%s: decode B=%d ctx=%d H_q=%d H_kv=%d d=%d d_I=%d Bk=%d k=%d, %d needle blocks/group"
            % (cfg.name, cfg.B, cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k, cfg.needles))


def run_stage(args):
    """One stage alone on --config, for profiler captures: prints {"stage", "ms", ...}."""
    import torch

    import datagen
    from block_sparse_long_index_gb300 import msa
    cfg = datagen.CONFIGS[args.config]
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    if args.stage == "warmup":  # msa_warmup_fwd + msa_warmup_index_grad on the prefill config's shapes
        inp = datagen.prefill_device(cfg)
        N, G = cfg.N, cfg.G
        shp = msa.shape(N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
        f32 = lambda *s_: torch.empty(s_, dtype=torch.float32, device="cuda")  # noqa: E731
        out = torch.empty((N, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
        lse, lse_idx = f32(cfg.H_q, N), f32(G, N)
        dq_idx, dk_idx, kl = f32(N, G, cfg.d_I), f32(N, cfg.d_I), f32(G, N)
        sc = 1.0 / math.sqrt(cfg.d)

        def call():
            msa.msa_warmup_fwd(inp["q"], inp["k"], inp["v"], inp["q_idx"], inp["k_idx"], shp, sc, out, lse, lse_idx)
            msa.msa_warmup_index_grad(inp["q"], inp["k"], inp["q_idx"], inp["k_idx"], lse, lse_idx, shp, sc, 1.0,
                                      dq_idx, dk_idx, kl)
    elif args.stage in ("decode", "decode_fp8"):
        from block_sparse_long_index_gb300 import MsaDecode
        inp = datagen.decode_device(cfg)
        run = MsaDecode(cfg.B, cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
        call = lambda: run(inp["q_t"], inp["q_idx_t"], inp["k_idx_cache"], inp["k_cache"], inp["v_cache"],  # noqa
                           inp["ctx_len"])
        if args.stage == "decode_fp8":
            ki8 = torch.empty(inp["k_idx_cache"].shape, dtype=torch.uint8, device="cuda")
            qi8 = torch.empty(inp["q_idx_t"].shape, dtype=torch.uint8, device="cuda")
            msa.msa_quantize_e4m3(inp["k_idx_cache"], ki8.numel(), 1.0, ki8)
            msa.msa_quantize_e4m3(inp["q_idx_t"], qi8.numel(), 1.0, qi8)
            del inp["k_idx_cache"]
            call = lambda: msa.msa_decode_fp8(inp["q_t"], qi8, ki8, inp["k_cache"], inp["v_cache"],  # noqa
                                              inp["ctx_len"], cfg.B, run.shape, 1.0 / math.sqrt(cfg.d), run.out,
                                              run.lse, run.block_idx, run.workspace)
    else:
        want = ("q_idx", "k_idx") if args.stage.startswith("select") else ("q", "k", "v", "q_idx", "k_idx")
        inp = datagen.prefill_device(cfg, want=want)
        blk = torch.empty((cfg.G, cfg.N, cfg.k), dtype=torch.int32, device="cuda")
        ws_sel = torch.empty(msa.msa_select_blocks_workspace(cfg.N, cfg.G, cfg.d_I, cfg.Bk, cfg.k),
                             dtype=torch.uint8, device="cuda")
        select = lambda: msa.msa_select_blocks(inp["q_idx"], inp["k_idx"], cfg.N, cfg.G, cfg.d_I, cfg.Bk,  # noqa
                                               cfg.k, blk, ws_sel)
        if args.stage == "select_fp8":
            q8 = torch.empty(inp["q_idx"].shape, dtype=torch.uint8, device="cuda")
            k8 = torch.empty(inp["k_idx"].shape, dtype=torch.uint8, device="cuda")
            msa.msa_quantize_e4m3(inp["q_idx"], q8.numel(), 1.0, q8)
            msa.msa_quantize_e4m3(inp["k_idx"], k8.numel(), 1.0, k8)
            call = lambda: msa.msa_select_blocks_fp8(q8, k8, cfg.N, cfg.G, cfg.d_I, cfg.Bk, cfg.k, blk,  # noqa
                                                     ws_sel)
        elif args.stage == "select":
            call = select
        elif args.stage == "select_varlen":  # the bench's packed sequence mix over the config's N cells
            cu = [0]
            for n in varlen_mix(cfg.N, cfg.Bk):
                cu.append(cu[-1] + n)
            cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
            wsv = torch.empty(msa.msa_select_blocks_varlen_workspace(cfg.N, cfg.G, cfg.d_I, cfg.Bk, cfg.k),
                              dtype=torch.uint8, device="cuda")
            call = lambda: msa.msa_select_blocks_varlen(inp["q_idx"], inp["k_idx"], cu_d, len(cu) - 1, cfg.N,  # noqa
                                                        cfg.G, cfg.d_I, cfg.Bk, cfg.k, blk, wsv)
        else:
            select()
            shp = msa.shape(cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
            ws = torch.empty(msa.msa_sparse_attn_fwd_workspace(shp), dtype=torch.uint8, device="cuda")
            out = torch.empty((cfg.N, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((cfg.H_q, cfg.N), dtype=torch.float32, device="cuda")
            call = lambda: msa.msa_sparse_attn_fwd(inp["q"], inp["k"], inp["v"], blk, shp,  # noqa
                                                   1.0 / math.sqrt(cfg.d), out, lse, ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    a, b = E(), E()
    a.record()
    for _ in range(args.steps):
        call()
    b.record()
    torch.cuda.synchronize()
    print(json.dumps({"stage": args.stage, "config": workload_name(cfg), "steps": args.steps,
                      "ms": a.elapsed_time(b) / args.steps}), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.stage != "all":
        return run_stage(args)
    import torch
    ws, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist = Dist(True)
    peaks, peak_src = load_peaks()

    pre = bench_prefill(args, dist, torch, peaks)
    cfg = pre["cfg"]
    total_ms = dist.max(pre["total_ms"])
    K = args.steps
    value = ws * cfg.N * K / (total_ms / 1000.0)
    flops_index = (cfg.N ** 2 / 2.0) * cfg.G * cfg.d_I * 2.0
    flops_main = cfg.N * cfg.H_q * cfg.k * cfg.Bk * cfg.d * 4.0
    step_s = total_ms / K / 1000.0
    sel_s, att_s = pre["sel_ms"] / 1000.0, pre["att_ms"] / 1000.0
    # Every tensor-bound region timed here lasts well under the seconds-long power-capped loop behind the
    # sustained figure and runs at the maximum SM clock, so fractions are taken against the burst peak.
    peak_t = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    burst_src = "%s bf16_tflops (burst; each timed region is under ~1.5 s at the maximum SM clock)" % peak_src
    sel_tf = flops_index / sel_s / 1e12
    roofline_select = {"kernel": "msa_select_blocks (index scoring + pooling + top-k, one launch)",
                       "bound": "tensor", "achieved": sel_tf, "peak": peak_t, "unit": "TFLOP/s",
                       "frac": sel_tf / peak_t,
                       "traffic": traffic_for("select_prefill_128k",
                                              "block_sparse_long_index_gb300/csrc/msa_select.cu"),
                       "algorithmic": "(N^2/2)*G*d_I*2 = %.4g FLOP per launch" % flops_index,
                       "peak_source": burst_src}
    # The attention call (inversion, schedule, KV-outer tiles, combine) is the larger share of the
    # step and is bound by HBM: each (t, group, slot) entry gathers its gs query rows once and
    # writes gs partial rows once; the combine reads the partials back; K/V of every (group, block)
    # once; block_idx, out and lse once.
    entries = cfg.N * cfg.G * cfg.k
    row = cfg.gs * cfg.d * 2
    attn_bytes = (entries * row * 3                      # Q gather, partial O write, partial O read
                  + entries * cfg.gs * 8 * 2             # (m, l) per partial row, written and read
                  + cfg.G * cfg.nb * cfg.Bk * cfg.d * 2 * 2  # K and V
                  + cfg.G * cfg.N * cfg.k * 4 * 3        # block_idx read twice, B* entries written
                  + cfg.N * cfg.H_q * (cfg.d * 2 + 4))   # out, lse
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    att_bw = attn_bytes / att_s / 1e9
    roofline = {"kernel": "msa_sparse_attn_fwd (B->B*, schedule, KV-outer tcgen05 tiles, LSE combine)",
                "bound": "hbm", "achieved": att_bw, "peak": hbm, "unit": "GB/s", "frac": att_bw / hbm,
                "traffic": traffic_for("attn_call_prefill_128k", "block_sparse_long_index_gb300/csrc/msa_attn.cu",
                                       "block_sparse_long_index_gb300/csrc/msa_attn_tile.cu",
                                       "block_sparse_long_index_gb300/csrc/msa_invert.cu"),
                "traffic_note": "DRAM bytes of every kernel of one call captured at prefill_16k (q larger than L2) "
                                "and scaled by 8 to 128K (all terms scale with N); null once a source changes",
                "algorithmic": "N*G*k*gs*d*2*3 + N*G*k*gs*16 + G*nb*Bk*d*4 + G*N*k*12 + N*H_q*(2d+4)"
                               " = %d bytes per call" % attn_bytes,
                "peak_source": "%s hbm_gbs" % peak_src}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(cfg), "parallelism": "replicas" if ws > 1 else "single",
                       "l2": "inputs larger than L2 (q alone is %.2f GB)" % (cfg.N * cfg.H_q * cfg.d * 2 / 1e9)},
            "clocks": pre["clocks"],
            "gpu_launches": prefill_launches(cfg) * K,
            "roofline": roofline,
            "roofline_select": roofline_select,
            "stages_ms": {"select": pre["sel_ms"], "attend": pre["att_ms"],
                          "note": "the two stages as separate calls (msa_select_blocks, msa_sparse_attn_fwd); "
                                  "the step runs them as one msa_prefill call"},
            "step_frac_of_tensor_peak": (flops_index + flops_main) / step_s / 1e12 / peak_t,
            "step_frac_of_tensor_peak_sustained": (flops_index + flops_main) / step_s / 1e12 / peak_sus,
            "step_tflops": (flops_index + flops_main) / step_s / 1e12,
            "step_peak_source": burst_src}
    if "bwd_ms" in pre:
        bms = dist.max(pre["bwd_ms"])
        bflops = cfg.N * cfg.H_q * cfg.k * cfg.Bk * cfg.d * 10.0 + cfg.N * cfg.G * cfg.k * cfg.Bk * cfg.d_I * 6.0
        btf = bflops / (bms / 1000.0) / 1e12
        line["backward"] = {"metric": "prefill backward tokens/s at 128K (main-branch gradients + index KL gradient, "
                                      "msa_sparse_attn_bwd)", "value": ws * cfg.N / (bms / 1000.0),
                            "unit": "tokens/s", "ms_per_step": bms,
                            "roofline": {"bound": "tensor", "achieved": btf, "peak": peak_t, "unit": "TFLOP/s",
                                         "frac": btf / peak_t, "traffic": None,
                                         "algorithmic": "N*H_q*k*Bk*d*10 (S, dP, dV, dK, dQ) + N*G*k*Bk*d_I*6 "
                                                        "(index logits, dk_idx, dq_idx) = %.4g FLOP per call" % bflops,
                                         "peak_source": burst_src},
                            "gpu_launches": bwd_launches(cfg) * K}
    if "e2e" in pre:
        e = pre["e2e"]
        e_ms = dist.max(e["ms"])
        line["e2e"] = {"value": ws * cfg.N / (e_ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": e["h2d"],
                       "d2h_bytes_per_step": e["d2h"], "steps": e["steps"], "ms_per_step": e_ms,
                       "how": "PrefillHostPipeline: per step pinned host -> device copies of q, k, v, q_idx, k_idx, "
                              "select + attention, device -> pinned host copies of out and lse; copies of one "
                              "step overlap the compute of its neighbours"}
    if "fp8" in pre:
        f8 = pre["fp8"]
        f8_ms = dist.max(f8["step_ms"])
        peak8 = 2.0 * peak_t
        sel8_tf = flops_index / (f8["sel_ms"] / 1000.0) / 1e12
        line["prefill_fp8"] = {
            "metric": "prefill tokens/s at 128K with FP8 (E4M3) index inputs (msa_prefill_fp8)",
            "value": ws * cfg.N / (f8_ms / 1000.0), "unit": "tokens/s", "ms_per_step": f8_ms,
            "stages_ms": {"select_fp8": f8["sel_ms"], "quantize_q_idx_k_idx": f8["quant_ms"]},
            "note": "the step takes q_idx and k_idx already in E4M3 (as an index projection emitting FP8 would); "
                    "msa_quantize_e4m3 of both from bf16 is timed apart",
            "roofline_select": {"bound": "tensor", "achieved": sel8_tf, "peak": peak8, "unit": "TFLOP/s",
                                "frac": sel8_tf / peak8,
                                "traffic": traffic_for("select_fp8_prefill_128k",
                                                       "block_sparse_long_index_gb300/csrc/msa_select.cu"),
                                "algorithmic": "(N^2/2)*G*d_I*2 = %.4g FLOP per launch" % flops_index,
                                "peak_source": burst_src + " x 2 (nominal fp8/bf16 dense ratio 4.5/2.25)"},
            "gpu_launches": (prefill_launches(cfg)) * K}
    if "varlen" in pre:
        vl = pre["varlen"]
        v_ms = dist.max(vl["step_ms"])
        flops_index_v = sum(n * n / 2.0 for n in vl["lengths"]) * cfg.G * cfg.d_I * 2.0
        selv_tf = flops_index_v / (vl["sel_ms"] / 1000.0) / 1e12
        line["prefill_varlen"] = {
            "metric": "prefill tokens/s at 128K cells holding %d sequences (msa_prefill_varlen)" % len(vl["lengths"]),
            "value": ws * cfg.N / (v_ms / 1000.0), "unit": "tokens/s", "ms_per_step": v_ms,
            "lengths": vl["lengths"], "stages_ms": {"select_varlen": vl["sel_ms"]},
            "roofline_select": {"bound": "tensor", "achieved": selv_tf, "peak": peak_t, "unit": "TFLOP/s",
                                "frac": selv_tf / peak_t, "traffic": None,
                                "algorithmic": "sum_s(len_s^2/2)*G*d_I*2 = %.4g FLOP per launch" % flops_index_v,
                                "peak_source": burst_src},
            "gpu_launches": (prefill_launches(cfg) + 1) * K}
    if not args.no_other_prefill and args.config == "prefill_128k":
        for nm, steps in (("prefill_32k", max(K, 10)), ("prefill_1m", 2)):
            o = bench_prefill_other(nm, args, dist, torch, steps)
            oc = o["cfg"]
            o_ms = dist.max(o["ms"])
            fi = (oc.N ** 2 / 2.0) * oc.G * oc.d_I * 2.0
            fm = oc.N * oc.H_q * oc.k * oc.Bk * oc.d * 4.0
            tf = (fi + fm) / (o_ms / 1000.0) / 1e12
            # a timed region of a second or more runs under the power cap: the sustained peak applies there
            long_region = o_ms * o["steps"] > 1000.0
            pk, pk_src = (peak_sus, "%s bf16_tflops_sustained (the timed region lasts over a second)" % peak_src) \
                if long_region else (peak_t, burst_src)
            line[nm] = {"metric": "prefill tokens/s (msa_prefill: select, invert, schedule, tiles, combine)",
                        "value": ws * oc.N / (o_ms / 1000.0), "unit": "tokens/s", "ms_per_step": o_ms,
                        "steps": o["steps"], "workload": workload_name(oc),
                        "stages_ms": {"select": o["sel_ms"], "attend": o["att_ms"]},
                        "roofline": {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s",
                                     "frac": tf / pk, "frac_of_burst": tf / peak_t, "traffic": None,
                                     "algorithmic": "(N^2/2)*G*d_I*2 + N*H_q*k*Bk*d*4 = %.4g + %.4g FLOP per step"
                                                    % (fi, fm),
                                     "peak_source": pk_src},
                        "gpu_launches": prefill_launches(oc) * o["steps"]}
    if not args.no_warmup:
        wu = bench_warmup(args, dist, torch)
        wc = wu["cfg"]
        f_ms, g_ms = dist.max(wu["fwd_ms"]), dist.max(wu["grad_ms"])
        tri = wc.N * wc.N / 2.0
        f_fl = tri * (4.0 * wc.H_q * wc.d + 2.0 * wc.G * wc.d_I)
        g_fl = tri * (2.0 * wc.H_q * wc.d + 6.0 * wc.G * wc.d_I)
        line["warmup_mode"] = {
            "metric": "warmup-mode tokens/s (dense main attention + index KL and its gradients, msa_warmup_fwd + "
                      "msa_warmup_index_grad)",
            "value": ws * wc.N / ((f_ms + g_ms) / 1000.0), "unit": "tokens/s", "ms_per_step": f_ms + g_ms,
            "stages_ms": {"fwd": f_ms, "index_grad": g_ms}, "steps": wu["steps"],
            "workload": workload_name(wc),
            "roofline": {"bound": "tensor", "achieved": (f_fl + g_fl) / ((f_ms + g_ms) / 1000.0) / 1e12,
                         "peak": peak_t, "unit": "TFLOP/s",
                         "frac": (f_fl + g_fl) / ((f_ms + g_ms) / 1000.0) / 1e12 / peak_t, "traffic": None,
                         "algorithmic": "N^2/2 * (4 H_q d + 2 G d_I) forward + N^2/2 * (2 H_q d + 6 G d_I) index "
                                        "gradient (teacher scores, index logits, dq^I, dk^I) = %.4g FLOP per step"
                                        % (f_fl + g_fl),
                         "peak_source": burst_src},
            "gpu_launches": 3 * wu["steps"]}
    if not args.no_decode:
        dec = bench_decode(args, dist, torch)
        dcfg = dec["cfg"]
        d_ms = dist.max(dec["mean_ms"])
        bytes_step = dcfg.B * (dcfg.ctx * dcfg.d_I * 2 + dcfg.k * dcfg.Bk * 2 * dcfg.H_kv * dcfg.d * 2)
        bw = bytes_step / (d_ms / 1000.0) / 1e9
        hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        line["decode"] = {"metric": "decode tokens/s at 1M ctx", "value": ws * dcfg.B / (d_ms / 1000.0),
                          "unit": "tokens/s", "ms_per_step": d_ms, "median_ms": dec["median_ms"],
                          "steps": dec["steps"], "workload": workload_name(dcfg),
                          "l2": "between steps (outside the timed events) a 512 MB buffer is written, then another "
                                "512 MB buffer is read, so each step starts on a cold L2 with no dirty lines",
                          "ms_per_step_after_write_flush": dist.max(dec["dirty_ms"]),
                          "roofline": {"bound": "hbm", "achieved": bw, "peak": hbm, "unit": "GB/s",
                                       "frac": bw / hbm, "traffic": None,
                                       "algorithmic": "B*(ctx*d_I*2 + k*Bk*2*H_kv*d*2) = %d bytes per step"
                                                      % bytes_step,
                                       "peak_source": "%s hbm_gbs" % peak_src},
                          "gpu_launches": 2 * dec["steps"]}
        pg = dec["paged"]
        pg_ms = dist.max(pg["mean_ms"])
        pbw = bytes_step / (pg_ms / 1000.0) / 1e9
        line["decode_paged"] = {"metric": "decode tokens/s at 1M ctx, paged caches (msa_decode_paged)",
                                "value": ws * dcfg.B / (pg_ms / 1000.0), "unit": "tokens/s", "ms_per_step": pg_ms,
                                "median_ms": pg["median_ms"], "page_tokens": pg["page"],
                                "workload": workload_name(dcfg) + ", pages scattered by a random page table",
                                "roofline": {"bound": "hbm", "achieved": pbw, "peak": hbm, "unit": "GB/s",
                                             "frac": pbw / hbm, "traffic": None,
                                             "peak_source": "%s hbm_gbs" % peak_src},
                                "gpu_launches": 2 * dec["steps"]}
        if "fp8" in dec:
            f8 = dec["fp8"]
            f8_ms = dist.max(f8["mean_ms"])
            bytes8 = dcfg.B * (dcfg.ctx * dcfg.d_I * 1 + dcfg.k * dcfg.Bk * 2 * dcfg.H_kv * dcfg.d * 2)
            bw8 = bytes8 / (f8_ms / 1000.0) / 1e9
            line["decode_fp8"] = {"metric": "decode tokens/s at 1M ctx with an FP8 (E4M3) index-key cache "
                                            "(msa_decode_fp8)",
                                  "value": ws * dcfg.B / (f8_ms / 1000.0), "unit": "tokens/s", "ms_per_step": f8_ms,
                                  "median_ms": f8["median_ms"],
                                  "roofline": {"bound": "hbm", "achieved": bw8, "peak": hbm, "unit": "GB/s",
                                               "frac": bw8 / hbm, "traffic": None,
                                               "algorithmic": "B*(ctx*d_I*1 + k*Bk*2*H_kv*d*2) = %d bytes per step"
                                                              % bytes8,
                                               "peak_source": "%s hbm_gbs" % peak_src},
                                  "gpu_launches": 2 * dec["steps"]}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        dt, n, th = oracle_prefill_sample(cfg, args.cpu_rows)
        line["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": th, "kind": "oracle",
                                "sample": "%d seeded query rows of the %s workload (select over all %d groups + "
                                          "attention over all %d heads), %.1f s" % (n, cfg.name, cfg.G, cfg.H_q, dt)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
