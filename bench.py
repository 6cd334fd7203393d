"""Benchmark: decode attention over the packed low-bit KV cache, plus block append.

One timed step = one block period of streaming decode on the configured workload: 128 decode
calls (kvq_decode_attn) over the full packed cache with the fp tail growing 0..127 tokens,
then one kvq_append_block that quantizes the 128-token block the tail formed. value = packed
cache bytes the 128 decodes read (codes + fp16 metadata + CSR: the algorithmic count) / step
time, in GB/s. Decodes rotate over enough copies of the cache that every decode reads data
that is not in L2 (the copies together exceed 3x L2).

Default workload: LLaMA-7B-shaped MHA layer (32 heads x 128), batch 1, context 32768, nuq3
keys (pre-RoPE, per channel) / values (per token), 8-entry per-head N(0,1)-quantile codebook,
1% fp16 outliers in CSR. --config selects another workload (1..5).

--impl reference times the CPU oracle (test infrastructure) on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as WL  # noqa: E402

L2_BYTES = 126.5 * 2 ** 20
DECODES_PER_STEP = 128
# The cache's code layout: the tensor-core tile format (3-bit codes as 48-byte bit planes per 128
# codes, 2/4-bit value tiles one row per channel), which the tensor-core decode kernels read. The
# row layout of the KVQuant page's bit listing is the library's default and is covered by the
# parity tests; its decode runs on the CUDA-core kernel.
BENCH_LAYOUT = "mma"

# DRAM traffic of the decode kernel per block record (dram__bytes_read.sum + dram__bytes_write.sum
# of an ncu capture of one launch, divided by the records that launch reads), by workload. A
# launch reads every record once, so the traffic of a full launch is this figure times its
# records. Each entry holds the sources it was measured on (sha256 of the kernel file and the
# shared header); once they change the traffic reads null until a new capture replaces it.
# Captures and commands: profiles/dram_traffic_decode_kernels.md.
PROFILED_TRAFFIC = {
    2: {"bytes_per_record": 14879.5, "sources": ("kvq_decode_nuq.cu", "kvq_internal.cuh"),
        "sha256_16": "1ed2f05845bc2c91", "capture": "same workload at L = 16384 (4096 records)"},
    3: {"bytes_per_record": 9955.2, "sources": ("kvq_decode_mma.cu", "kvq_internal.cuh"),
        "sha256_16": "26b1444736ac01df", "capture": "full workload (8192 records)"},
    4: {"bytes_per_record": 17039.0, "sources": ("kvq_decode_mma.cu", "kvq_internal.cuh"),
        "sha256_16": "26b1444736ac01df", "capture": "same workload at L = 16384 (32768 records)"},
    5: {"bytes_per_record": 9318.0, "sources": ("kvq_decode_mma.cu", "kvq_internal.cuh"),
        "sha256_16": "26b1444736ac01df", "capture": "same workload at L = 131072 (32768 records)"},
}


def _profiled_traffic(cfg_id, records):
    """DRAM bytes of one full decode launch from the captured per-record traffic, or (None, why)."""
    import hashlib
    e = PROFILED_TRAFFIC.get(cfg_id)
    if e is None:
        return None, "no capture for this workload"
    m = hashlib.sha256()
    for f in e["sources"]:
        with open(os.path.join(ROOT, "bit_kv_cache_block_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    if m.hexdigest()[:16] != e["sha256_16"]:
        return None, "kernel sources changed since the capture"
    return round(e["bytes_per_record"] * records), f"ncu capture of the {e['capture']}, scaled by records"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the job's step time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_gbs(bytes_per_step_per_rank: int, step_ms: float, world: int) -> float:
    """Whole-job throughput: every rank streams its own replica (weak scaling), so the job moves
    world times one rank's bytes in the slowest rank's step time."""
    return world * bytes_per_step_per_rank / (step_ms * 1e-3) / 1e9


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.p = None
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
            self.f.close()

    def summary(self):
        if self.p is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                             parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 200] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def _gen_device(w, torch, dev, shape, kind, seed):
    """Large synthetic inputs drawn on the device (performance runs only; parity tests use the
    seeded numpy generators)."""
    g = torch.Generator(device=dev)
    g.manual_seed(1000003 * seed + 17 * kind + w.cfg_id)
    if kind == 0 and w.k_dist == "student_t3":
        z = torch.randn(shape, generator=g, device=dev)
        chi = torch.randn((3,) + tuple(shape), generator=g, device=dev).pow(2).sum(0) / 3
        x = z / chi.sqrt()
    else:
        x = torch.randn(shape, generator=g, device=dev)
    if kind == 0 and w.k_outlier_channels:
        x[..., list(w.k_outlier_channels)] *= w.k_outlier_gain
    return x.to(torch.float16 if w.dtype == "f16" else torch.bfloat16)


def _inputs(w, torch, dev, rank):
    """Prefill K/V for the whole context, the tail block and the decode query, resident on the device."""
    nb = w.n_blocks
    shape = (w.batch, w.n_kv_heads, nb * 128, 128)
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    n_elem = 2 * math.prod(shape)
    if n_elem * 4 <= 2 * 2 ** 30:   # seeded numpy generators (same as the tests)
        K, V = WL.blocks(w, 0, nb, seed=rank)
        to = lambda x: torch.from_numpy(WL.to_storage(x, w.dtype).view(np.int16)).to(dev).view(dt)
        Kd, Vd = to(K), to(V)
        tk, tv = WL.tail(w, 127, seed=rank)
        q = WL.query(w, seed=rank)
        return Kd, Vd, to(tk), to(tv), to(q), "numpy"
    Kd = _gen_device(w, torch, dev, shape, 0, rank)
    Vd = _gen_device(w, torch, dev, shape, 1, rank)
    tshape = (w.batch, w.n_kv_heads, 127, 128)
    tk = _gen_device(w, torch, dev, tshape, 0, rank + 7)
    tv = _gen_device(w, torch, dev, tshape, 1, rank + 7)
    q = _gen_device(w, torch, dev, (w.batch, w.n_q_heads, 128), 1, rank + 11)
    return Kd, Vd, tk, tv, q, "torch-device"


def _workload(args):
    """The chosen workload, with the context and the absmax format overrides applied."""
    w = WL.WORKLOADS[args.config]
    if args.ctx:
        w = w.scaled(ctx=args.ctx)
    if args.bits or args.scale_group:
        if w.method != "int4":
            raise SystemExit("--bits and --scale-group apply to the absmax (int4) workload")
        w = w.scaled(bits=args.bits or w.bits, scale_group=args.scale_group or w.scale_group)
        w = w.scaled(name=w.name.replace("int4", f"int{w.bits}") +
                     (", 64-channel scales" if w.scale_group == 64 else ""))
    return w


def run_kvq(args):
    import torch
    import bit_kv_cache_block_gb300 as K
    import __graft_entry__
    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    K._lib.lib()
    w = _workload(args)
    nb = w.n_blocks
    n_pages = w.batch * (nb + 1) if args.paged else 0
    if (args.key_calib or args.sink or args.v_csc) and w.method != "nuq":
        raise SystemExit("--key-calib, --sink and --v-csc apply to nuq workloads")
    cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, nb + 1, w.dtype, w.pre_rope,
                        w.rope_theta, w.outlier_frac, w.varn_iters, True, BENCH_LAYOUT, n_pages, args.key_calib,
                        args.sink, w.scale_group, args.v_csc)
    table = None
    if args.paged:  # every block on a page of a shuffled pool
        perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(5 + rank)).to(torch.int32)
        table = perm.view(w.batch, nb + 1)
    lay = K.kvq_layout(cfg)
    cb = None
    if w.method == "nuq":
        from statistics import NormalDist
        inv = NormalDist().inv_cdf
        n = 2 ** w.bits
        vals = [inv((j + 0.5) / n) / inv((n - 0.5) / n) for j in range(n)]
        cb = torch.tensor([vals] * w.n_kv_heads, dtype=torch.float32)
    cache_bytes = K.kvq_decode_bytes(cfg, nb)
    n_copies = max(1, math.ceil(3 * L2_BYTES / max(1, int(lay.records_bytes))))
    caches = [K.KVCache(cfg, cb, device=dev, block_table=table)]
    Kd, Vd, tk, tv, q, gen = _inputs(w, torch, dev, rank)
    if args.key_calib:  # offline statistics from 3 blocks of the workload's keys drawn with another seed
        kc = np.stack([np.concatenate([WL.tile(w, 0, h, blk, WL.KIND_K, seed=99) for blk in range(3)])
                       for h in range(w.n_kv_heads)])
        caches[0].calibrate_keys(torch.from_numpy(WL.to_storage(kc, w.dtype).view(np.int16)).to(dev).view(Kd.dtype))
    caches[0].append(Kd, Vd)
    # bulk append: the whole context in one call, timed on a second cache (warm kernels)
    bulk_ms = None
    if n_copies > 1:
        c = K.KVCache(cfg, cb, device=dev, block_table=table)
        if args.key_calib:
            c.base.copy_(caches[0].base)  # the calibration table
            K.kvq_truncate(c.cache, 0)
            c.cache.calibrated = 1
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        c.append(Kd, Vd)
        e1.record()
        e1.synchronize()
        bulk_ms = e0.elapsed_time(e1)
        caches.append(c)
    del Kd, Vd
    for _ in range(n_copies - len(caches)):
        c = K.KVCache(cfg, cb, device=dev, block_table=table)
        c.base.copy_(caches[0].base)
        K.kvq_truncate(c.cache, 0)
        c.cache.n_blocks = nb
        caches.append(c)
    out = torch.empty(w.batch, w.n_q_heads, 128, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    tail_k = tk.contiguous()
    tail_v = tv.contiguous()
    # tail prefixes for n_tail = 1..127 as contiguous views ([B][H][n][128] each)
    tails = [None] + [(tail_k[:, :, :j].contiguous(), tail_v[:, :, :j].contiguous()) for j in range(1, 128)]
    blk_k = torch.cat([tail_k, tail_k[:, :, :1]], dim=2).contiguous()   # the block the tail completes
    blk_v = torch.cat([tail_v, tail_v[:, :, :1]], dim=2).contiguous()
    ws = caches[0].workspace

    R_DEC, R_APP = 32, 8

    def step_ops(st):
        for d in range(DECODES_PER_STEP):
            c = caches[d % n_copies]
            tkk, tvv = (tails[d] if d else (None, None))
            K.kvq_decode_attn(c.cache, q, tkk, tvv, d, out, ws, st)
        caches[0].append(blk_k, blk_v, stream=st)
        K.kvq_truncate(caches[0].cache, nb)

    def dec_ops(st):
        for d in range(R_DEC):
            K.kvq_decode_attn(caches[d % n_copies].cache, q, None, None, 0, out, ws, st)

    def app_ops(st):
        for _ in range(R_APP):
            caches[0].append(blk_k, blk_v, stream=st)
            K.kvq_truncate(caches[0].cache, nb)

    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for _ in range(args.warmup):       # eager warm-up (also settles every launch attribute)
            step_ops(cap)
            dec_ops(cap)
            app_ops(cap)
        cap.synchronize()
        graphs = {}
        for name, fn in (("step", step_ops), ("dec", dec_ops), ("app", app_ops)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn(cap)
            graphs[name] = g
        for g in graphs.values():           # warm replays
            g.replay()
        cap.synchronize()

        def timed(g, reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(cap)
            for _ in range(reps):
                g.replay()
            e1.record(cap)
            e1.synchronize()
            return e0.elapsed_time(e1) / reps

        if world > 1:
            torch.distributed.barrier()
        try:
            gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
        except Exception:
            gpu_id = str(local)
        with Clocks(gpu_id) as clk:
            torch.cuda.synchronize()
            step_ms = timed(graphs["step"], args.steps)
            torch.cuda.synchronize()
        dec0_us = 1e3 * timed(graphs["dec"], 3) / R_DEC
        app_us = 1e3 * timed(graphs["app"], 3) / R_APP
    total_ms = step_ms * args.steps
    status = max(int(c.status.item()) for c in caches)
    if status != 0:
        raise RuntimeError(f"device status {status} ({K.kvq_status_str(status)})")
    step_ms = _max_over_ranks(step_ms, world, dev)
    dec_bytes_step = cache_bytes * DECODES_PER_STEP
    value = _job_gbs(dec_bytes_step, step_ms, world)
    dec_avg_us = (1e3 * step_ms - app_us) / DECODES_PER_STEP
    peak, peak_kind = _peaks()
    achieved = cache_bytes / (dec0_us * 1e-6) / 1e9   # decode call with an empty tail
    base_w = WL.WORKLOADS[w.cfg_id]
    same_format = (w.bits, w.scale_group) == (base_w.bits, base_w.scale_group)
    traffic, traffic_note = (_profiled_traffic(w.cfg_id, w.batch * w.n_kv_heads * nb) if same_format
                             else (None, "no capture for this format"))
    res = {
        "metric": "quantized decode-attn packed-KV GB/s (% of 8 TB/s HBM), us/step; append tokens/s",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"rtn": "u%d codes, fp32 accumulate" % w.bits, "nuq": "u3 codes + fp16 csr, fp32 accumulate",
                  "varn": "u2 codes, fp32 accumulate", "int4": "s%d codes, fp32 accumulate" % w.bits}[w.method],
        "data": f"synthetic ({gen}, seeded)",
        "config": {"workload": w.name, "method": w.method, "bits": w.bits, "batch": w.batch,
                   "n_kv_heads": w.n_kv_heads, "n_q_heads": w.n_q_heads, "context": w.ctx,
                   "decodes_per_step": DECODES_PER_STEP, "tail_tokens": "0..127",
                   "layout": BENCH_LAYOUT, "scale_group": w.scale_group,
                   "paged": bool(args.paged), "key_calib": bool(args.key_calib),
                   "sink": bool(args.sink), "v_csc": bool(args.v_csc),
                   "packed_bytes_per_decode": cache_bytes, "cache_copies": n_copies,
                   "l2": f"{n_copies} cache copies rotated ({n_copies * int(lay.records_bytes) / 2**20:.0f} MiB > 3x L2)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_8TBs": round(100 * value / 8000, 2),
        "decode_us": round(dec_avg_us, 3),
        "decode_us_empty_tail": round(dec0_us, 3),
        "append_us_per_block": round(app_us, 3),
        "append_tokens_per_s": round(w.batch * 128 / (app_us * 1e-6), 1),
        "append_bulk": None if bulk_ms is None else {
            "ms": round(bulk_ms, 3), "tokens_per_s": round(w.batch * nb * 128 / (bulk_ms * 1e-3), 1),
            "gbs": round((2 * w.batch * w.n_kv_heads * nb * 128 * 128 * 2 + int(lay.record_bytes) * w.batch
                          * w.n_kv_heads * nb) / (bulk_ms * 1e-3) / 1e9, 1),
            "note": "the whole context in one kvq_append_block call: fp16 read + packed write"},
        "timed_region_ms": round(total_ms, 3),
        "timing": "CUDA graph replays, CUDA events on the launching stream",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_note,
                     "kernel": _decode_kernel_name(w) + " + combine_kernel (kvq_decode_attn, empty tail)",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "gpu_launches": args.steps * (2 * DECODES_PER_STEP + 1),
        "roofline_decodes": R_DEC,
        "clocks": clk.summary(),
    }
    if args.e2e:
        res["e2e"] = run_e2e(args, K, torch, dev, caches, cfg, w, nb, q, tail_k, tail_v, cache_bytes)
    if args.per_config and not args.ctx and (args.bits, args.scale_group) == (0, 0):
        # the other workloads of the benchmark, one empty-tail decode each at full size
        others = [c for c in (1, 2, 3, 4, 5) if c != w.cfg_id]
        del caches, ws
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        with Clocks(gpu_id) as pclk:
            pc = per_config_decodes(K, torch, dev, rank, others, peak)
        pc["clocks"] = pclk.summary()
        pc["timing"] = ("CUDA graph replays of empty-tail decodes (kvq_decode_attn + combine), CUDA events on "
                        "the launching stream; cache copies rotated so that each decode reads data not in L2")
        res["per_config"] = pc
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_sample_heads)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return res if rank == 0 else None


def per_config_decodes(K, torch, dev, rank, cfg_ids, peak):
    """One decode with an empty tail per workload, timed like the headline roofline entry: CUDA
    graph replays of R decodes that rotate over enough cache copies to exceed 3x L2, events on the
    launching stream, clocks sampled meanwhile. Inputs are drawn on the device (performance only);
    each workload's cache is freed before the next one is built."""
    out = {}
    cap = torch.cuda.Stream(device=dev)
    for cid in cfg_ids:
        w = WL.WORKLOADS[cid]
        nb = w.n_blocks
        cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, nb, w.dtype, w.pre_rope,
                            w.rope_theta, w.outlier_frac, w.varn_iters, True, BENCH_LAYOUT, 0, False, False,
                            w.scale_group, False)
        lay = K.kvq_layout(cfg)
        cb = None
        if w.method == "nuq":
            from statistics import NormalDist
            inv = NormalDist().inv_cdf
            n = 2 ** w.bits
            cb = torch.tensor([[inv((j + 0.5) / n) / inv((n - 0.5) / n) for j in range(n)]] * w.n_kv_heads,
                              dtype=torch.float32)
        shape = (w.batch, w.n_kv_heads, nb * 128, 128)
        caches = [K.KVCache(cfg, cb, device=dev)]
        Kd = _gen_device(w, torch, dev, shape, 0, rank)
        Vd = _gen_device(w, torch, dev, shape, 1, rank)
        caches[0].append(Kd, Vd)
        del Kd, Vd
        n_copies = max(1, math.ceil(3 * L2_BYTES / max(1, int(lay.records_bytes))))
        for _ in range(n_copies - 1):
            c = K.KVCache(cfg, cb, device=dev)
            c.base.copy_(caches[0].base)
            c.cache.n_blocks = nb
            caches.append(c)
        q = _gen_device(w, torch, dev, (w.batch, w.n_q_heads, 128), 1, rank + 11)
        o = torch.empty(w.batch, w.n_q_heads, 128, dtype=torch.float32, device=dev)
        ws = caches[0].workspace
        reps = 8 if w.n_blocks * w.batch * w.n_kv_heads > 100000 else 32
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            for i in range(3):
                K.kvq_decode_attn(caches[i % n_copies].cache, q, None, None, 0, o, ws, cap)
            cap.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                for i in range(reps):
                    K.kvq_decode_attn(caches[i % n_copies].cache, q, None, None, 0, o, ws, cap)
            gr.replay()
            cap.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cap)
            for _ in range(3):
                gr.replay()
            e1.record(cap)
            e1.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / (3 * reps)
        status = max(int(c.status.item()) for c in caches)
        if status != 0:
            raise RuntimeError(f"config {cid}: device status {status} ({K.kvq_status_str(status)})")
        dec_bytes = K.kvq_decode_bytes(cfg, nb)
        gbs = dec_bytes / (us * 1e-6) / 1e9
        out[str(cid)] = {"workload": w.name, "decode_us_empty_tail": round(us, 3), "gbs": round(gbs, 1),
                         "frac": round(gbs / peak, 4), "packed_bytes_per_decode": dec_bytes,
                         "kernel": _decode_kernel_name(w) + " + combine_kernel", "cache_copies": n_copies}
        del caches, gr, q, o, ws
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_e2e(args, K, torch, dev, caches, cfg, w, nb, q, tail_k, tail_v, cache_bytes):
    """Same step through the C ABI from pinned host buffers. Row d of one staging buffer holds
    decode d's query and the tail token it adds (K and V), so each decode uploads one contiguous
    row; kvq_decode_attn_ex reads the tail in place through a token stride of one row (token t
    sits in row t + 1). The 128 outputs of the step come back in one copy, and the block append
    reads the step's tail."""
    stream = torch.cuda.current_stream()
    BH = w.batch * w.n_kv_heads
    nq, nkv = q.numel(), BH * 128
    row = nq + 2 * nkv                                   # elements per staging row
    hbuf = torch.empty((DECODES_PER_STEP + 1, row), dtype=q.dtype).pin_memory()
    tk_tok = tail_k.permute(2, 0, 1, 3).reshape(127, nkv).cpu()   # token-major
    tv_tok = tail_v.permute(2, 0, 1, 3).reshape(127, nkv).cpu()
    for d in range(DECODES_PER_STEP + 1):
        hbuf[d, :nq] = q.reshape(-1).cpu()
        if d > 0:
            t = (d - 1) % 127
            hbuf[d, nq:nq + nkv] = tk_tok[t]
            hbuf[d, nq + nkv:] = tv_tok[t]
    dbuf = torch.empty((DECODES_PER_STEP + 1, row), dtype=q.dtype, device=dev)
    outs = torch.empty((DECODES_PER_STEP, w.batch, w.n_q_heads, 128), dtype=torch.float32, device=dev)
    hout = torch.empty_like(outs, device="cpu").pin_memory()
    ws = caches[0].workspace
    n_copies = len(caches)
    h2d = d2h = 0

    def step(i):
        nonlocal h2d, d2h
        h2d = d2h = 0
        for d in range(DECODES_PER_STEP):
            dbuf[d].copy_(hbuf[d], non_blocking=True)
            h2d += hbuf[d].numel() * hbuf.element_size()
            c = caches[(i * DECODES_PER_STEP + d) % n_copies]
            qd = dbuf[d, :nq].view(q.shape)
            tk_ = dbuf[1, nq:] if d else None                  # K token t in row t + 1
            tv_ = dbuf[1, nq + nkv:] if d else None
            K.kvq_decode_attn_ex(c.cache, qd, tk_, tv_, d, 128, row, outs[d], ws, stream)
        dbuf[DECODES_PER_STEP].copy_(hbuf[DECODES_PER_STEP], non_blocking=True)  # the token completing the block
        h2d += hbuf[DECODES_PER_STEP].numel() * hbuf.element_size()
        hout.copy_(outs, non_blocking=True)
        d2h += outs.numel() * 4
        kt = dbuf[1:, nq:nq + nkv].view(128, w.batch, w.n_kv_heads, 128).permute(1, 2, 0, 3).contiguous()
        vt = dbuf[1:, nq + nkv:].view(128, w.batch, w.n_kv_heads, 128).permute(1, 2, 0, 3).contiguous()
        c = caches[i % n_copies]
        c.append(kt, vt, stream=stream)
        K.kvq_truncate(c.cache, nb)
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    return {"value": round(cache_bytes * DECODES_PER_STEP / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "wall clock per step, host buffers pinned, copies inside the timed region"}


def _oracle_sample(w, heads, seed=0):
    """Oracle append (timed) and decode (timed) for a few (b, h) of the workload."""
    import oracle as O
    oc = O.OracleCache.for_workload(w, layout=O.LAYOUT_MMA if BENCH_LAYOUT == "mma" else O.LAYOUT_ROWS)
    t_app = 0.0
    for blk in range(w.n_blocks):
        K = np.empty((w.batch, w.n_kv_heads, 128, 128), np.float32)
        V = np.empty_like(K)
        for (b, h) in heads:
            K[b, h] = WL.tile(w, b, h, blk, 0, seed)
            V[b, h] = WL.tile(w, b, h, blk, 1, seed)
        t = time.perf_counter()
        oc.append(K, V, only_heads=set(heads))
        t_app += time.perf_counter() - t
    q = WL.query(w, seed=seed)
    t = time.perf_counter()
    oc.decode(q, only_heads=set(heads))
    t_dec = time.perf_counter() - t
    return t_app, t_dec


def _oracle_pool_worker(cid, pair, n_blocks, barrier, cmd_q, out_q):
    """One worker of the multi-core oracle runs: builds its (b, h) pair's cache over n_blocks
    (append timed), then per command decodes it once, all workers starting together at the
    barrier; reports the monotonic times of each phase."""
    import oracle as O
    ws = WL.WORKLOADS[cid].scaled(ctx=128 * n_blocks)
    oc = O.OracleCache.for_workload(ws, layout=O.LAYOUT_MMA if BENCH_LAYOUT == "mma" else O.LAYOUT_ROWS)
    a0 = time.perf_counter()
    for blk in range(n_blocks):
        K = np.zeros((ws.batch, ws.n_kv_heads, 128, 128), np.float32)
        V = np.zeros_like(K)
        K[pair] = WL.tile(ws, pair[0], pair[1], blk, 0)
        V[pair] = WL.tile(ws, pair[0], pair[1], blk, 1)
        oc.append(K, V, only_heads={pair})
    out_q.put((a0, time.perf_counter()))
    while True:
        step = cmd_q.get()
        if step is None:
            break
        q = WL.query(ws, step)
        barrier.wait()
        d0 = time.perf_counter()
        oc.decode(q, only_heads={pair})
        out_q.put((d0, time.perf_counter()))


class OraclePool:
    """The oracle on n_procs spawned processes, one (b, h) pair of workload cid each, over the first
    n_blocks blocks of its context. Run with BLAS pinned to one thread per process, so n_procs is
    the number of host cores in use. append_s = wall time of all workers' appends; step(i) = wall
    time of one decode of every pair, all started together."""

    def __init__(self, cid, n_blocks, n_procs):
        import multiprocessing as mp
        w = WL.WORKLOADS[cid]
        self.pairs = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)][:max(1, n_procs)]
        ctx = mp.get_context("spawn")
        barrier = ctx.Barrier(len(self.pairs))
        self.cmd_q, self.out_q = ctx.Queue(), ctx.Queue()
        self.procs = [ctx.Process(target=_oracle_pool_worker,
                                  args=(cid, pr, n_blocks, barrier, self.cmd_q, self.out_q))
                      for pr in self.pairs]
        for p in self.procs:
            p.start()
        res = [self.out_q.get() for _ in self.procs]
        self.append_s = max(r[1] for r in res) - min(r[0] for r in res)

    def step(self, i):
        for _ in self.procs:
            self.cmd_q.put(i)
        res = [self.out_q.get() for _ in self.procs]
        return max(r[1] for r in res) - min(r[0] for r in res)

    def close(self):
        for _ in self.procs:
            self.cmd_q.put(None)
        for p in self.procs:
            p.join()


def _host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def _pair_bytes(w, nb):
    """Packed-cache bytes one decode reads for one (b, h) pair over nb blocks."""
    import bit_kv_cache_block_gb300 as K
    cfg = K.make_config(w.method, w.bits, 1, 1, w.group, nb, w.dtype, w.pre_rope, w.rope_theta,
                        w.outlier_frac, w.varn_iters, True, BENCH_LAYOUT)
    return K.kvq_decode_bytes(cfg, nb)


def oracle_baseline_run():
    """All the oracle timings of the CPU baseline (run in a subprocess with BLAS on one thread):
    the headline workload on every host core and on one, and a single-core sample of each other
    workload (append per block and decode per step extrapolated from a sample of blocks)."""
    n_cores = _host_cores()
    res = {"cores": n_cores, "cpu": _cpu_model(), "per_config": {}}
    w = WL.WORKLOADS[2]
    nb = w.n_blocks
    for key, n in (("all_cores", min(n_cores, w.batch * w.n_kv_heads)), ("one_core", 1)):
        pool = OraclePool(2, nb, n)
        dec = min(pool.step(i) for i in range(2))
        pool.close()
        npairs = len(pool.pairs)
        res[key] = {"pairs": npairs, "blocks": nb, "decode_s": round(dec, 3), "append_s": round(pool.append_s, 3),
                    "decode_gbs": round(npairs * _pair_bytes(w, nb) / dec / 1e9, 5),
                    "append_tokens_per_s": round(npairs * nb * 128 / pool.append_s, 1)}
    for cid in (1, 2, 3, 4, 5):
        wc = WL.WORKLOADS[cid]
        ns = min(wc.n_blocks, {1: 16, 2: 256, 3: 32, 4: 32, 5: 256}[cid])
        ws = wc.scaled(ctx=128 * ns)
        pool = OraclePool(cid, ns, 1)
        t_dec = min(pool.step(i) for i in range(2))
        pool.close()
        t_app = pool.append_s
        units = wc.batch * wc.n_kv_heads
        res["per_config"][str(cid)] = {
            "workload": wc.name, "sample": f"1 (batch, KV head) pair, {ns} of {wc.n_blocks} blocks, one core",
            "append_ms_per_block_all_heads": round(1e3 * t_app / ns * units, 3),
            "decode_ms_per_step": round(1e3 * t_dec / ns * units * wc.n_blocks, 3),
            "decode_gbs_one_core": round(_pair_bytes(ws, ns) / t_dec / 1e9, 5)}
    return res


def cpu_baseline(w, n_heads):
    """The oracle as it stands, timed on the host cores in a subprocess with BLAS pinned to one
    thread per process: the headline workload on every core (one worker process per core, one
    (b, h) pair each, whole context) and on one core, plus a single-core sample of every workload.
    value = the headline decode throughput on all cores (GB/s of packed cache decoded)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, json; sys.path.insert(0, %r); import bench; print(json.dumps(bench.oracle_baseline_run()))"
            % ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle", "error": r.stderr[-400:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    ac = d["all_cores"]
    return {"value": ac["decode_gbs"], "unit": "GB/s", "cores": ac["pairs"], "kind": "oracle",
            "sample": f"{ac['pairs']} (batch, KV head) pairs of {WL.WORKLOADS[2].name}, all {ac['blocks']} blocks, "
                      f"one worker process per core (decode {ac['decode_s']} s wall, append {ac['append_s']} s)",
            "append_tokens_per_s": ac["append_tokens_per_s"], "one_core": d["one_core"],
            "per_config_one_core": d["per_config"], "host_cores": d["cores"], "cpu": d["cpu"]}


def _cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def run_reference(args):
    """The oracle as it stands, as the reference arm: one spawned process per host core (BLAS on one
    thread each), one (batch, KV head) pair of the workload each; a step is one decode of every
    pair, all started together, over a bounded sample of the context."""
    rank, world, local = _dist()
    if rank != 0:
        return None
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    w = WL.WORKLOADS[args.config]
    # bound the run to a few minutes of CPU work at ~4 ms of oracle decode per block and core
    n_sample = min(w.n_blocks, max(16, int(120.0 / (0.004 * (args.steps + args.warmup)))))
    pool = OraclePool(args.config, n_sample, min(_host_cores(), w.batch * w.n_kv_heads))
    try:
        for i in range(args.warmup):
            pool.step(i)
        per = [pool.step(args.warmup + i) for i in range(args.steps)]
    finally:
        pool.close()
    npairs = len(pool.pairs)
    nbytes = npairs * _pair_bytes(w, n_sample)
    ms = 1e3 * statistics.mean(per)
    v = nbytes / (ms * 1e-3) / 1e9
    sample = (f"decode of {npairs} (batch, KV head) pairs over {n_sample} of {w.n_blocks} blocks per step, "
              f"one process per pair and core")
    return {"impl": "reference", "metric": "quantized decode-attn packed-KV GB/s (% of 8 TB/s HBM), us/step; append tokens/s",
            "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (oracle)", "data": "synthetic (numpy, seeded)",
            "config": {"workload": w.name, "sample": sample},
            "append_tokens_per_s": round(npairs * n_sample * 128 / pool.append_s, 1),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": npairs, "kind": "oracle",
                             "sample": sample, "host_cores": _host_cores(), "cpu": _cpu_model()},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_diag(args):
    """Error diagnostics ([KVN] Figures 1a/1b) over the whole cache of a workload: kvq_error_stats
    (per-token |x|, norm deviation, E_T, E_D for K and V) timed as one launch, then
    kvq_error_topk; the JSON line carries the E_M / E_T shares of the largest errors, and for
    RTN / KVarN workloads the same shares with the other of the two methods on the same inputs."""
    import torch
    import bit_kv_cache_block_gb300 as K
    import __graft_entry__
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    __graft_entry__.build()
    K._lib.lib()
    w = _workload(args)
    nb = w.n_blocks
    Kd, Vd, _, _, _, gen = _inputs(w, torch, dev, 0)
    fracs = [0.001, 0.01, 0.05, 0.1, 1.0]

    def build(method):
        cfg = K.make_config(method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, nb, w.dtype, w.pre_rope,
                            w.rope_theta, w.outlier_frac, w.varn_iters, True, BENCH_LAYOUT,
                            scale_group=w.scale_group if method == "int4" else 128)
        cb = None
        if method == "nuq":
            from statistics import NormalDist
            inv = NormalDist().inv_cdf
            n = 2 ** w.bits
            cb = torch.tensor([[inv((j + 0.5) / n) / inv((n - 0.5) / n) for j in range(n)]] * w.n_kv_heads,
                              dtype=torch.float32)
        c = K.KVCache(cfg, cb, device=dev)
        c.append(Kd, Vd)
        return cfg, c

    def shares(c):
        sk, sv = c.error_stats(Kd, Vd)
        res = {}
        for name, S in (("K", sk), ("V", sv)):
            t = K.error_topk(S, fracs).cpu().numpy()
            res[name] = {"top_frac": fracs, "k": [int(x) for x in t[:, 0]],
                         "E_M_over_E_T": [round(float(x), 4) for x in t[:, 2] / t[:, 1]],
                         "mean_E_T": [float("%.5g" % x) for x in t[:, 1] / t[:, 0]]}
            nd = S[..., 1] / S[..., 0]
            res[name]["token_norm_dev_p99_abs"] = float("%.4g" % torch.quantile(nd.abs().flatten()[:2 ** 24].float(), 0.99).item())
        return res

    cfg, cache = build(w.method)
    shape = (w.batch, w.n_kv_heads, nb * 128, 4)
    sk = torch.empty(shape, dtype=torch.float32, device=dev)
    sv = torch.empty_like(sk)
    n_rows = sk.numel() // 4
    out = torch.empty(len(fracs), 4, dtype=torch.float64, device=dev)
    tws = torch.empty(K.kvq_error_topk_workspace_bytes(), dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()

    def one():
        K.kvq_error_stats(cache.cache, 0, nb, Kd, Vd, sk, sv, st)

    def topk():
        K.kvq_error_topk(sk, fracs, out, tws, st)

    for _ in range(args.warmup):
        one()
        topk()
    torch.cuda.synchronize()

    def timed(fn, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(0).uuid)
    except Exception:
        gpu_id = "0"
    with Clocks(gpu_id) as clk:
        torch.cuda.synchronize()
        ms = timed(one, args.steps)
        topk_ms = timed(topk, max(3, args.steps // 4))
        torch.cuda.synchronize()
    if cache.device_status() != 0:
        raise RuntimeError("device status %d" % cache.device_status())
    in_bytes = 2 * Kd.numel() * Kd.element_size()
    rec_bytes = K.kvq_decode_bytes(cfg, nb)
    out_bytes = 2 * sk.numel() * 4
    alg = in_bytes + rec_bytes + out_bytes
    gbs = alg / (ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    diag = {w.method: shares(cache)}
    if w.method in ("rtn", "varn"):
        other = "varn" if w.method == "rtn" else "rtn"
        _, c2 = build(other)
        diag[other] = shares(c2)
    return {
        "metric": "error-stats GB/s (kvq_error_stats over the whole cache, K and V)", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 dequantise and sums", "data": f"synthetic ({gen}, seeded)",
        "config": {"workload": w.name, "method": w.method, "bits": w.bits, "batch": w.batch,
                   "n_kv_heads": w.n_kv_heads, "context": w.ctx, "layout": BENCH_LAYOUT, "rows": n_rows,
                   "l2": f"inputs {in_bytes / 2**20:.0f} MiB per launch (> L2)"},
        "us_error_stats": round(1e3 * ms, 2), "us_error_topk": round(1e3 * topk_ms, 2),
        "topk_rows_per_s": round(n_rows / (topk_ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None, "traffic_source": "not captured",
                     "kernel": "error_stats_kernel", "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes": alg},
        "gpu_launches": args.steps + 19 * max(3, args.steps // 4),
        "diagnostics": diag,
        "clocks": clk.summary(),
    }


FIT_HEADS, FIT_SAMPLES = 32, 16 * 2048 * 128   # one layer of LLaMA-7B: 16 sequences of 2K tokens


def _fit_inputs_np(n, seed):
    """Calibration samples of one head: normalised pre-RoPE key entries (tanh of a Gaussian, in
    [-1, 1]) and Fisher weights (squared Gaussian gradients over their maximum, in [0, 1])."""
    rng = np.random.default_rng(seed)
    a = np.tanh(0.8 * rng.standard_normal(n)).astype(np.float32)
    g = rng.standard_normal(n) ** 2
    return a, (g / g.max()).astype(np.float32)


def _fit_cpu(n, passes):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, time, json; sys.path.insert(0, %r); import bench, oracle as O; "
            "a, w = bench._fit_inputs_np(%d, 1); t = time.perf_counter(); c, it = O.fit_codebook(a, w, 3, %d); "
            "print(json.dumps([time.perf_counter() - t, it]))" % (ROOT, n, passes))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "error": r.stderr[-400:]}
    t, it = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": round(8 * n * it / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"one head, {n} samples, 3 bits, {it} passes in {t:.2f} s", "cpu": _cpu_model()}


FIT_TRAFFIC = (1077113088, "kvq_fit.cu")   # dram read + write bytes of one assign_kernel launch (ncu)
FIT_TRAFFIC_SHA = "73c2a64531debfc9"   # sha256 prefix of kvq_fit.cu as captured


def _fit_traffic():
    """The ncu traffic of the fit pass, or None once kvq_fit.cu has changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "bit_kv_cache_block_gb300", "csrc", FIT_TRAFFIC[1])
    h = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    return FIT_TRAFFIC[0] if h == FIT_TRAFFIC_SHA else None


def run_fit(args):
    """Sensitivity-weighted codebook fitting ([KVQ] Algorithm 2) for one layer: 32 KV heads of
    16 x 2048 x 128 samples each, 3 bits. The roofline is one Lloyd pass (kvq_fit_codebook with
    max_iter = 1: every sample read once, 8 bytes); the JSON line also carries the time of a whole
    fit (max_iter = 50)."""
    import torch
    import bit_kv_cache_block_gb300 as K
    import __graft_entry__
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    __graft_entry__.build()
    lib = K._lib.lib()
    H, n = FIT_HEADS, FIT_SAMPLES
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    a = torch.tanh(0.8 * torch.randn(H, n, device=dev, generator=gen))
    g = torch.randn(H, n, device=dev, generator=gen) ** 2
    w = g / g.amax(dim=1, keepdim=True)
    del g
    cb = torch.empty(H, 8, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, int(lib.kvq_fit_codebook_workspace_bytes(H, n))), dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()

    def fit(max_iter):
        K._lib.check(lib.kvq_fit_codebook(K._ptr(a), K._ptr(w), H, n, 3, max_iter, K._ptr(cb), K._ptr(ws),
                                          ws.numel(), K._stream(st)), "kvq_fit_codebook")

    def timed(fn, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    for _ in range(args.warmup):
        fit(1)
    fit(50)
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(0).uuid)
    except Exception:
        gpu_id = "0"
    reps_full = max(3, args.steps // 20)
    with Clocks(gpu_id) as clk:
        torch.cuda.synchronize()
        ms = timed(lambda: fit(1), args.steps)
        full_ms = timed(lambda: fit(50), reps_full)
        torch.cuda.synchronize()
    alg = 8 * H * n
    gbs = alg / (ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    res = {
        "metric": "codebook-fit GB/s (one weighted Lloyd pass, 8 B per sample)", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 samples, exact int64 fixed-point sums", "data": "synthetic (torch device generator, seeded)",
        "config": {"workload": "nuq3 codebook fit, one LLaMA-7B layer: 32 KV heads x 16 x 2048 x 128 samples",
                   "n_heads": H, "samples_per_head": n, "bits": 3,
                   "l2": f"inputs {alg / 2**20:.0f} MiB per pass (> L2)"},
        "us_per_pass": round(1e3 * ms, 2), "ms_whole_fit_max_iter_50": round(full_ms, 3),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": _fit_traffic(),
                     "traffic_source": "ncu capture of assign_kernel at this workload",
                     "kernel": "assign_kernel + update_kernel (kvq_fit_codebook, max_iter 1)",
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": alg},
        "gpu_launches": 3 * args.steps + 101 * reps_full,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = _fit_cpu(1 << 23, 20)
    return res


def _decode_kernel_name(w):
    """The decode kernel the library picks for this workload (mirrors its dispatch rules)."""
    if w.method == "nuq" and w.bits == 3 and w.group == 1 and w.pre_rope:
        return "decode_nuq_kernel"
    if (w.method in ("rtn", "varn", "int4") and (w.bits in (2, 4) or (w.method, w.bits) == ("int4", 8))
            and w.group <= 4 and w.scale_group == 128):
        return "decode_mma_kernel"
    return "decode_kernel"


def _decode_bytes_per_head(w):
    """Algorithmic packed bytes of one (b, h) over the context (same count as kvq_decode_bytes)."""
    # 3-bit tiles: 48 B per 128 codes as bit planes, 52 B as 10-code rows
    W = 12 if (w.bits == 3 and BENCH_LAYOUT == "mma") else -(-128 // (32 // w.bits))
    meta = {"rtn": 2, "nuq": 2, "varn": 3, "int4": 2 if w.scale_group == 64 else 1}[w.method] * 256
    csr = 0
    if w.method == "nuq":
        n = math.ceil(float(np.float32(w.outlier_frac)) * 16384)
        csr = 3 * n + 258 if n else 0
    return 2 * (128 * W * 4 + meta + csr) * w.n_blocks


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the empty-tail decode of every other workload at full size")
    ap.add_argument("--key-calib", dest="key_calib", action="store_true",
                    help="nuq: offline-calibrated key statistics (calibration keys drawn with another seed)")
    ap.add_argument("--sink", action="store_true", help="nuq: keep the first token in the input precision")
    ap.add_argument("--v-csc", dest="v_csc", action="store_true", help="nuq: value outliers stored by column (CSC)")
    ap.add_argument("--paged", action="store_true",
                    help="records on the pages of a shuffled pool, found through a block table")
    ap.add_argument("--cpu-sample-heads", type=int, default=10)
    ap.add_argument("--ctx", type=int, default=0, help="override the context length (tokens, multiple of 128)")
    ap.add_argument("--bits", type=int, default=0, choices=[0, 4, 8],
                    help="absmax workload: code width (8: the sensitive-layer precision)")
    ap.add_argument("--scale-group", dest="scale_group", type=int, default=0, choices=[0, 64, 128],
                    help="absmax workload: channels per scale")
    ap.add_argument("--diag", action="store_true",
                    help="time the error diagnostics (kvq_error_stats, kvq_error_topk) instead of decode")
    ap.add_argument("--fit", action="store_true",
                    help="time the sensitivity-weighted codebook fitting (kvq_fit_codebook) instead of decode")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.fit:
        res = run_fit(args) if args.impl == "kvq" else {"impl": "reference", "unavailable": "--fit has no CPU arm"}
    elif args.diag:
        res = run_diag(args) if args.impl == "kvq" else {"impl": "reference", "unavailable": "--diag has no CPU arm"}
    else:
        res = run_reference(args) if args.impl == "reference" else run_kvq(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
