"""Benchmark of the paged decode attention hot path on GB300.

One step = one call through the C ABI over one batch of seeded synthetic
input of the chosen workload: for GQA (bf16 or FP8 pools, decode or verify)
the split-KV attention kernel and the combine; for MLA the absorb, the
attention core and the merge fused with the W_UV projection; for the KV writes the
write kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``value`` is the achieved HBM bandwidth of the
whole call: algorithmic bytes (visible K/V rows of every KV head, or latent
rows for MLA, plus q and the outputs; weights too for MLA; rows read and
written for the KV writes) divided by the
device time per call, with the inputs resident in HBM and a 512 MB buffer
written between timed calls (outside the timed events) so no call reads a
warm L2.  ``roofline`` reports the dominant kernel (the split-KV attention
kernel) alone, timed with events recorded on the call's stream by the
library's profiling hook.  ``e2e`` repeats the measurement through the same
C ABI call with host buffers: per step the decode inputs that change every
step (q, block table, context lengths) are copied from pinned host memory and
the outputs (out, lse) are copied back; the KV cache is device-resident state.

With --gpus N under torchrun every rank runs its own replica of the workload
on its GPU (decode attention exchanges nothing between GPUs: replicas / weak
scaling); the time is the max over ranks and value the sum of all ranks'
bytes over it.

--impl reference times the fp64 CPU oracle (the reference arm) on the host
cores, on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (frac of ~8 TB/s) for paged decode attention"
FLUSH_BYTES = 512 << 20
CLEAN_BYTES = 512 << 20
DEFAULT_WORKLOAD = "qwen3-32b"
WORKLOADS = ["tiny", "llama3-8b", "qwen3-32b", "hd256-window", "mla", "kv-write", "qwen3-32b-verify4",
             "qwen3-32b-fp8", "kv-write-fp8", "qwen3-32b-nvfp4", "kv-write-nvfp4"]
# sources of the kernel each roofline line profiles (a change voids its committed ncu traffic)
KERNEL_SOURCES = {"gqa": ("pa_gqa.cuh", "pa_partition.cuh", "pa_common.cuh", "pa_api.cu"),
                  "gqa_f8": ("pa_gqa_f8.cuh", "pa_gqa.cuh", "pa_partition.cuh", "pa_common.cuh", "pa_api.cu"),
                  "gqa_fp4": ("pa_gqa_fp4.cuh", "pa_gqa.cuh", "pa_partition.cuh", "pa_common.cuh", "pa_api.cu"),
                  "mla": ("pa_mla_tc.cuh", "pa_tcgen05.cuh", "pa_mla.cu", "pa_gqa.cuh", "pa_partition.cuh",
                          "pa_common.cuh"),
                  "write": ("pa_kv_write.cu", "pa_common.cuh")}


def compute_dtype(w):
    """(dtype, description) of the arithmetic the timed path computes in."""
    import synth
    if isinstance(w, synth.KVWriteWorkload):
        if w.nvfp4:
            return "f32", "fp32 divides by the pool and block scales, e4m3 block-scale and e2m1 encode"
        return ("f32", "fp32 divide by the scale, e4m3 encode") if w.fp8 else ("bf16", "bf16 copy")
    if getattr(w, "nvfp4", False):
        return "bf16", "e2m1 x e4m3 block values dequantized exactly to bf16, bf16 tensor-core mma, f32 softmax"
    if getattr(w, "fp8", False):
        return "e4m3", "e4m3 tensor-core mma (two-term q and p), f32 softmax and accumulation"
    return "bf16", "bf16 tensor-core mma, f32 softmax and accumulation"


def kernel_kind(workload: str) -> str:
    if workload.startswith("kv-write"):
        return "write"
    if workload.endswith("-nvfp4"):
        return "gqa_fp4"
    return "mla" if workload == "mla" else "gqa_f8" if workload.endswith("-fp8") else "gqa"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=WORKLOADS)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(values, world: int):
    """Max over ranks of a list of floats (timings): the slowest replica sets the job's time.
    A host-side gloo all-reduce; the decode itself exchanges nothing between GPUs."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def kernel_hash(kind: str = "gqa") -> str:
    h = hashlib.sha256()
    for n in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "paged_kv_attention_19_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the split kernel from the committed ncu summary
    (profiles/traffic.json); None if there is none or the kernel sources changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            e = json.load(f)[workload]
        return float(e["dram_bytes"]) if e["kernel_hash"] == kernel_hash(kernel_kind(workload)) else None
    except Exception:
        return None


def describe(w, name):
    import synth
    if isinstance(w, synth.KVWriteWorkload):
        return {"workload": name, "tokens": w.num_tokens, "kv_heads": int(w.k.shape[1]),
                "head_dim": int(w.k.shape[2]), "page_size": w.page_size, "pool_pages": w.num_pages,
                "slots": "prefill order: token t at position t % P of page perm[t // P]",
                "algorithmic_bytes": w.algorithmic_bytes(), "seed": w.seed,
                **({"pools": "fp8 e4m3 codes", "k_scale": w.k_scale, "v_scale": w.v_scale} if w.fp8 else {}),
                **({"pools": "nvfp4 rows (e2m1 code pairs, e4m3 scale per 16 values, 16-byte padding)",
                    "k_scale": w.k_scale, "v_scale": w.v_scale} if w.nvfp4 else {})}
    if isinstance(w, synth.MLAWorkload):
        return {"workload": name, "batch": w.batch, "heads": w.num_heads, "q_dim": 192, "cache_dim": 576,
                "v_dim": 128, "page_size": w.layout.page_size, "context": "uniform[1024,8192]",
                "visible_tokens": w.visible_tokens(), "algorithmic_bytes": w.algorithmic_bytes(),
                "algorithmic_bytes_without_weights": w.algorithmic_bytes(with_weights=False), "seed": w.seed}
    ctx = {"tiny": "fixed{1,31,32,33,64,100}", "llama3-8b": "uniform[512,4096]",
           "qwen3-32b": "loguniform[128,16384]", "hd256-window": "uniform[2048,32768], window 4096",
           "qwen3-32b-verify4": "loguniform[128,16384] (the qwen3-32b lengths), 4 query positions per row, "
                                "causal among them",
           "qwen3-32b-fp8": "loguniform[128,16384] (the qwen3-32b lengths)",
           "qwen3-32b-nvfp4": "loguniform[128,16384] (the qwen3-32b lengths)"}[name]
    return {"workload": name, "batch": w.batch, "query_positions": w.num_query, "q_heads": w.num_q_heads,
            "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "page_size": w.layout.page_size, "context": ctx, "window": w.window,
            "visible_tokens": w.visible_tokens(), "algorithmic_bytes": w.algorithmic_bytes(), "seed": w.seed,
            **({"kv_cache": "fp8 e4m3 codes, per-pool scales", "k_scale": w.k_scale, "v_scale": w.v_scale}
               if w.fp8 else
               {"kv_cache": "nvfp4 rows: e2m1 codes, e4m3 scale per 16 values, per-pool scales; algorithmic "
                            "bytes count 9/16 byte per value, not the row padding",
                "k_scale": w.k_scale, "v_scale": w.v_scale} if w.nvfp4 else {"kv_cache": "bf16"})}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [(t, s.split(", ")) for t, s in self.samples]
        if self.t0 is not None:
            inside = [(t, r) for t, r in rows if self.t0 - 0.05 <= t <= self.t1 + 0.05]
            rows = inside or rows
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                for n, v in zip(names, r[4:8]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except Exception:
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class OracleSample:
    """A bounded sample of the workload for the fp64 oracle: every stride-th (row, head) output,
    the stride chosen so that one pass takes about `target_s` seconds on the host cores."""

    def __init__(self, w, name, target_s: float = 1.0):
        import oracle
        import synth
        self.cores = oracle.num_threads()
        if isinstance(w, synth.KVWriteWorkload):
            # the oracle writes token by token into copies of the pools: time it on all tokens
            kp, vp = w.empty_pool(), w.empty_pool()
            if w.nvfp4:
                self.fn = lambda rows: oracle.kv_write_nvfp4(w.k, w.v, w.slots, kp, vp, w.k_scale, w.v_scale)
            elif w.fp8:
                self.fn = lambda rows: oracle.kv_write_fp8(w.k, w.v, w.slots, kp, vp, w.k_scale, w.v_scale)
            else:
                self.fn = lambda rows: oracle.kv_write(w.k, w.v, w.slots, kp, vp)
            self.rows, self.bytes = None, w.algorithmic_bytes()
            self.desc = f"all {w.num_tokens} tokens of the {name} workload"
            self.cores = 1
            return
        is_mla = isinstance(w, synth.MLAWorkload)
        H = w.num_heads if is_mla else w.num_q_heads
        Q = 1 if is_mla else w.num_query
        rows_all = [(b, h) for b in range(w.batch) for h in range(H)]
        win = 0 if is_mla else w.window
        vis = [synth.visible_range(int(L), win, Q) for L in w.layout.context_lens]
        total_work = sum(hi - lo for lo, hi in vis) * H
        if not is_mla and w.nvfp4:
            self.fn = lambda rows: oracle.gqa_nvfp4(w.q, w.k_pool, w.v_pool, w.layout.block_table,
                                                    w.layout.context_lens, w.scale, w.k_scale, w.v_scale,
                                                    w.window, rows=[(b, i, h) for b, h in rows for i in range(Q)],
                                                    num_query=Q)
        elif not is_mla and w.fp8:
            self.fn = lambda rows: oracle.gqa_fp8(w.q, w.k_pool, w.v_pool, w.layout.block_table,
                                                  w.layout.context_lens, w.scale, w.k_scale, w.v_scale, w.window,
                                                  rows=[(b, i, h) for b, h in rows for i in range(Q)],
                                                  num_query=Q)
        elif Q > 1:
            # every query position of a sampled (row, head)
            self.fn = lambda rows: oracle.verify_gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table,
                                                     w.layout.context_lens, w.scale, w.window,
                                                     rows=[(b, i, h) for b, h in rows for i in range(Q)])
        elif is_mla:
            self.fn = lambda rows: oracle.mla(w.q, w.cache, w.w_uk, w.w_uv, w.layout.block_table,
                                              w.layout.context_lens, w.scale, rows=rows)
        else:
            self.fn = lambda rows: oracle.gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table,
                                              w.layout.context_lens, w.scale, w.window, rows=rows)
        stride = max(1, len(rows_all) // 64)
        while True:
            rows = rows_all[::stride]
            t = time.perf_counter()
            self.fn(rows)
            dt = time.perf_counter() - t
            if dt > target_s / 2 or stride == 1:
                break
            stride = max(1, int(stride * max(0.05, dt / target_s)))
        self.rows = rows
        # the sample's share of the algorithmic bytes, in proportion to the keys its outputs read
        self.bytes = w.algorithmic_bytes() * sum(vis[b][1] - vis[b][0] for b, _ in rows) / max(total_work, 1)
        self.desc = f"{len(rows)} of {len(rows_all)} (row, head) outputs of the {name} workload (stride {stride})"

    def run(self):
        t = time.perf_counter()
        self.fn(self.rows)
        return time.perf_counter() - t


def cpu_oracle_time(w, name, budget_s: float = 10.0):
    """Time the oracle, as it stands, on a bounded sample of the workload; returns (GB/s, desc, cores)."""
    s = OracleSample(w, name)
    reps, tot = 0, 0.0
    while tot < budget_s or reps == 0:
        tot += s.run()
        reps += 1
    return s.bytes / (tot / reps) / 1e9, f"{s.desc}, {reps} timed passes", s.cores


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import synth
    w = synth.workload(args.workload)
    cfg = describe(w, args.workload)
    s = OracleSample(w, args.workload)
    for _ in range(args.warmup):
        s.run()
    times = [s.run() for _ in range(args.steps)]
    value = s.bytes / (sum(times) / len(times)) / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1000 * sum(times) / len(times), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": cfg,
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": s.cores, "kind": "oracle",
                             "sample": s.desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, local_rank, world):
    import torch

    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    import paged_kv_attention_19_gb300 as pa
    import synth
    import synth.device as gu

    w = synth.workload(args.workload)
    cfg = describe(w, args.workload)
    is_mla = isinstance(w, synth.MLAWorkload)
    is_write = isinstance(w, synth.KVWriteWorkload)
    # per workload: the device inputs a step copies in end to end, the outputs it reads back,
    # and call(*inputs) running the step on device tensors
    if is_write:
        ins = [gu.dev(w.k), gu.dev(w.v), torch.from_numpy(w.slots).cuda()]
        kp = gu.dev(w.empty_pool())
        vp = None if w.mla else gu.dev(w.empty_pool())
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs = [status]
        if w.mla:
            def call(c, r, s):
                pa.pa_mla_cache_write(c, r, s, kp, status=status)
        elif w.nvfp4:
            def call(k, v, s):
                pa.pa_kv_write_nvfp4(k, v, s, kp, vp, k_scale=w.k_scale, v_scale=w.v_scale, status=status)
        elif w.fp8:
            def call(k, v, s):
                pa.pa_kv_write_fp8(k, v, s, kp, vp, k_scale=w.k_scale, v_scale=w.v_scale, status=status)
        else:
            def call(k, v, s):
                pa.pa_kv_write(k, v, s, kp, vp, status=status)
    elif is_mla:
        d = gu.MlaDev(w)
        B = w.batch
        out = torch.empty(B, w.num_heads, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, w.num_heads, dtype=torch.float32, device="cuda")
        ws = pa.workspace_for_mla(d.q, d.cache, d.bt, args.num_splits)
        ins, outs = [d.q, d.bt, d.lens], [out, lse]

        def call(q, bt, lens):
            pa.pa_decode_mla_absorbed(q, d.cache, d.wuk, d.wuv, bt, lens, out, lse, scale=w.scale, workspace=ws,
                                      num_splits=args.num_splits)
    else:
        d = gu.GqaDev(w)
        out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(w.q.shape[:-1], dtype=torch.float32, device="cuda")
        ws = pa.workspace_for_gqa(d.q, d.k, d.bt, args.num_splits)
        ins, outs = [d.q, d.bt, d.lens], [out, lse]
        if w.nvfp4:
            def call(q, bt, lens):
                pa.pa_decode_gqa_nvfp4(q, d.k, d.v, bt, lens, out, lse, scale=w.scale, k_scale=w.k_scale,
                                       v_scale=w.v_scale, window=w.window, workspace=ws,
                                       num_splits=args.num_splits)
        elif w.fp8:
            def call(q, bt, lens):
                pa.pa_decode_gqa_fp8(q, d.k, d.v, bt, lens, out, lse, scale=w.scale, k_scale=w.k_scale,
                                     v_scale=w.v_scale, window=w.window, workspace=ws, num_splits=args.num_splits)
        else:
            entry = pa.pa_verify_gqa if w.num_query > 1 else pa.pa_decode_gqa

            def call(q, bt, lens):
                entry(q, d.k, d.v, bt, lens, out, lse, scale=w.scale, window=w.window, workspace=ws,
                      num_splits=args.num_splits)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clean = torch.zeros(CLEAN_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush_l2():
        # write a buffer larger than L2, then read another one, so the timed call finds no
        # input in L2 and no dirty line whose write-back would compete with its reads
        flush.zero_()
        clean.sum()

    stream = torch.cuda.current_stream()
    abytes = cfg["algorithmic_bytes"]

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    clocks = ClockSampler(local_rank)
    clocks.start()
    for _ in range(args.warmup):
        flush_l2()
        call(*ins)
    launches_per_call = pa.pa_last_launch_count()
    torch.cuda.synchronize()

    # ---- device-resident timing: the whole call (no events inside it, so the launches of
    # one call overlap as they do in use), then the split-KV kernel alone (events around it)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks.t0 = time.time()
    for i in range(args.steps):
        flush_l2()
        evs[i][0].record(stream)
        call(*ins)
        evs[i][1].record(stream)
    for i in range(args.steps):
        flush_l2()
        pa.pa_set_profile_events(*kev[i])
        call(*ins)
    torch.cuda.synchronize()
    clocks.t1 = time.time()
    barrier()
    pa.pa_set_profile_events(None, None)
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    kms = sum(a.elapsed_time(b) for a, b in kev) / args.steps
    gpu_launches = args.steps * launches_per_call
    ms, kms = reduce_max([ms, kms], world)
    value = world * abytes / (ms * 1e-3) / 1e9
    kernel_gbs = abytes / (kms * 1e-3) / 1e9

    # ---- end to end through the C ABI with host buffers
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    ins_h = [pin(t) for t in ins]
    for h, t in zip(ins_h, ins):
        h.copy_(t)
    outs_h = [pin(t) for t in outs]
    ins_d = [torch.empty_like(t) for t in ins]
    h2d = sum(t.numel() * t.element_size() for t in ins_h)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    e2e_steps = max(1, min(args.steps, 200))
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(e2e_steps):
        flush_l2()
        eev[i][0].record(stream)
        for dd, h in zip(ins_d, ins_h):
            dd.copy_(h, non_blocking=True)
        call(*ins_d)
        for h, dd in zip(outs_h, outs):
            h.copy_(dd, non_blocking=True)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    ems = reduce_max([sum(a.elapsed_time(b) for a, b in eev) / e2e_steps], world)[0]
    e2e_value = world * abytes / (ems * 1e-3) / 1e9
    clocks.stop()
    if rank != 0:
        return 0

    peak, peak_kind = measured_peaks()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1000, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": compute_dtype(w)[0], "arithmetic": compute_dtype(w)[1],
        "data": "synthetic", "impl": "ours",
        "config": dict(cfg, num_splits=args.num_splits or "auto", parallelism=f"replicas x{world}",
                       l2="between timed calls, outside the timed events: a 512 MB buffer written, then another 512 MB read"),
        "roofline": {"bound": "alu" if is_mla else "hbm",
                     "kernel": (("kv_write_nvfp4_kernel" if w.nvfp4 else "kv_write_fp8_kernel" if w.fp8
                                 else "kv_write_kernel") if is_write
                                else "mla_tc_split_kernel" if is_mla
                                else "gqa_fp4_split_kernel" if getattr(w, "nvfp4", False)
                                else "gqa_f8_split_kernel" if getattr(w, "fp8", False) else "gqa_split_kernel"),
                     "achieved": round(kernel_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(kernel_gbs / peak, 4), "peak_source": f"hbm_gbs of {peak_kind}",
                     "kernel_us": round(kms * 1000, 2), "traffic": ncu_traffic(args.workload)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "us_per_call": round(ems * 1000, 2),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": gpu_launches,
        "launches_per_call": launches_per_call,
        "clocks": clocks.summary(),
    }
    if is_mla:
        # the MLA attention core is a tensor-core contraction: its roofline is the bf16 tensor peak
        # (the algorithmic flops: 2 x (576 + 512) per (head, visible token); the two column-half
        # CTAs of a head tile each compute the full scores, 2 x 576 more per (head, token) that is
        # executed but not counted).  Its HBM rate counts the bytes the core itself reads: the
        # visible cache rows and q_abs, not the projection weights.
        flops = 2.0 * w.visible_tokens() * w.num_heads * (576 + 512)
        tf_peak, tf_kind = measured_bf16_tflops()
        achieved = flops / (kms * 1e-3) / 1e12
        core_gbs = w.algorithmic_bytes(with_weights=False) / (kms * 1e-3) / 1e9
        line["roofline"].update({"bound": "tensor", "achieved": round(achieved, 2), "peak": tf_peak,
                                 "unit": "TFLOP/s", "frac": round(achieved / tf_peak, 4),
                                 "peak_source": f"bf16_tflops of {tf_kind} (cuBLAS bf16 burst)",
                                 "hbm_gbs": round(core_gbs, 2), "hbm_frac": round(core_gbs / peak, 4)})
    if not args.no_cpu_baseline:
        v, desc, cores = cpu_oracle_time(w, args.workload)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    sys.exit(main())
