"""Benchmark: one step = K/V append + paged attention over a synthetic batch,
issued as one pa_step call (the attention kernel launched as a programmatic
dependent of the append).

Default workload (N = 1): the 0.6B-class batched decode shape -- 512
sequences, contexts U{64..2662}, 16 query / 8 KV heads, head_dim 128, bf16,
32-token pages from a shuffled pool, one decode row per sequence plus its K/V
append.  The K/V the step reads (2.87 GB) is 22x the 129 MB L2, so steps run
back to back without an L2 flush; a workload whose K/V fits a few times in L2
(--workload shared_prefix) is timed step by step after an L2 flush.

Prints ONE JSON line (rank 0).  `value` is rows/s over the timed steps with
inputs resident in HBM; `e2e` is the same metric with the step's inputs copied
host->device and the output copied back inside the timed region; `roofline`
is the attention kernel's algorithmic bytes (valid K/V slots, shared pages
once, plus Q and O) per launch over its CUDA-event time, against the measured
HBM copy bandwidth.  `cpu_baseline` times the CPU oracle on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload batched_decode|mixed_step|shared_prefix|long_context|tiny_decode|
                              batched_decode_fp8|long_context_fp8]
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attention rows/s and KV-read GB/s vs GB300 HBM roofline (1 GPU)"
L2_BYTES = 129 * 1000 * 1000  # GB300 L2
W_CONFIG_NAMES = ("batched_decode", "mixed_step", "shared_prefix", "long_context", "tiny_decode",
                  "batched_decode_fp8", "long_context_fp8")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0  # burst


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "paged_kv_continuous_pa_gb300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 peak for a kernel timed alone (burst), measured; else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_tiles_alone(pa, torch, st, wl, steps: int, stream):
    """The chunk rows of the step attended alone (one launch of prefill tiles
    only, after the step's append): tensor-pipe fraction of the tiles.
    Algorithmic FLOPs: 4 * D per (chunk row, visible key, query head) --
    Q.K and P.V, one multiply-add each."""
    import numpy as np
    rows = np.concatenate([np.arange(b, b + n) for b, n in wl.chunks])
    flops = 4.0 * wl.D * wl.Hq * float(np.sum(wl.positions[rows].astype(np.int64) + 1))
    idx = torch.as_tensor(rows, dtype=torch.long, device=st.q.device)
    q = st.q[idx].contiguous()
    out = torch.empty_like(q)
    seq, pos = st.seq_ids[idx].contiguous(), st.positions[idx].contiguous()
    starts, b = [], 0
    for _, n in wl.chunks:
        starts.append((b, n))
        b += n
    wsb = pa.workspace_bytes(st.pool, len(rows), wl.Hq, wl.max_blocks, starts)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=q.device) if wsb else None
    call = lambda: pa.attention(st.pool, q, seq, pos, st.block_tables, out, chunks=starts,
                                softmax_scale=wl.softmax_scale, workspace=ws, status=st.status, stream=stream)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, e in ev:
        a.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(e) for a, e in ev)
    peak, kind = measured_bf16_tflops()
    tflops = flops / (ms / 1e3) / 1e12
    return {"gflop": flops / 1e9, "ms": ms, "tflops": tflops, "peak_tflops": peak, "frac": tflops / peak,
            "peak_source": f"{kind} (MEASURED_PEAKS.json bf16_tflops, burst)", "kernel": "mixed_kernel tiles only"}


def profiled_traffic(workload: str, src_hash: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_decode_attention_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_hash") != src_hash:
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # start timing only once the sampler is producing lines
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            lines = [l.strip() for l in f if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_workload(name: str, seqs: int = 0):
    import workloads as W
    if seqs > 0:
        if name in ("batched_decode", "batched_decode_fp8", "long_context", "long_context_fp8"):
            return W.CONFIGS[name](n_seqs=seqs)
        if name == "shared_prefix":
            return W.shared_prefix(n_seqs=seqs)
        raise ValueError("--seqs applies to batched_decode, long_context and shared_prefix")
    return W.CONFIGS[name]()


class OracleLeg:
    """The CPU oracle, as it stands, on a bounded sample of the step: the
    step's append for the sample rows plus exact FP64 attention for them, over
    all host cores.  The sample is the step's first rows, as many as take about
    `target_s` seconds of wall time on these cores."""

    def __init__(self, wl, target_s: float = 3.0):
        import numpy as np
        import oracle
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from ref import oracle_pools  # test-side oracle setup

        self.wl, self.oracle, self.np = wl, oracle, np
        self.cores = oracle.host_cores()
        # calibrate on one row, single-threaded, then size the sample
        probe = np.arange(1)
        seqs = sorted(set(int(s) for s in wl.seq_ids[probe]))
        kp, vp = oracle_pools(wl, rows_of_seqs=seqs, include_step=False)
        t0 = time.perf_counter()
        self._attend(probe, kp, vp, 1)
        t_row = max(time.perf_counter() - t0, 1e-6) * float(np.mean(wl.positions + 1)) / float(wl.positions[0] + 1)
        n = int(min(wl.n_rows, max(8, target_s * self.cores / t_row)))
        self.rows = np.arange(n)
        seqs = sorted(set(int(s) for s in wl.seq_ids[self.rows]))
        self.kp, self.vp = oracle_pools(wl, rows_of_seqs=seqs, include_step=False)
        self.sample = (f"first {n} of {wl.n_rows} rows of one step (their K/V append + attention), "
                       f"FP64 C oracle over {self.cores} threads")

    def _attend(self, rows, kp, vp, threads):
        wl = self.wl
        self.oracle.attention(wl.q[rows], wl.q_dtype, wl.Hq, wl.seq_ids[rows], wl.positions[rows],
                              wl.block_tables, wl.num_pages, wl.P, wl.Hkv, wl.D, wl.kv_dtype, wl.k_scale,
                              wl.v_scale, kp, vp, softmax_scale=wl.softmax_scale, n_threads=threads)

    def step(self):
        """One timed pass; returns (rows/s, seconds)."""
        wl, r = self.wl, self.rows
        t0 = time.perf_counter()
        self.oracle.append(wl.k_new[r], wl.v_new[r], wl.in_dtype, wl.seq_ids[r], wl.positions[r], wl.block_tables,
                           wl.num_pages, wl.P, wl.Hkv, wl.D, wl.kv_dtype, wl.k_scale, wl.v_scale, self.kp, self.vp)
        self._attend(r, self.kp, self.vp, self.cores)
        dt = time.perf_counter() - t0
        return len(r) / dt, dt


def run_reference(args):
    """The reference arm: the CPU oracle timed as it stands on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = make_workload(args.workload, args.seqs)
    leg = OracleLeg(wl, target_s=2.0)
    for _ in range(args.warmup):
        leg.step()
    rates, times = [], []
    for _ in range(args.steps):
        r, dt = leg.step()
        rates.append(r)
        times.append(dt)
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.description},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": leg.cores, "kind": "oracle",
                             "sample": leg.sample},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of every rank's x: the slowest replica sets the job's time.
    `dist` is torch.distributed with an initialised process group, or None
    for one process."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the rows every replica processed in one step over
    the step time (already the maximum over ranks)."""
    return rows_per_rank * world / (ms_per_step / 1e3)


def attention_kernel_name(wl) -> str:
    """The kernel pa_attention launches for this workload's decode rows."""
    import workloads as W
    G = wl.Hq // wl.Hkv
    if wl.chunks and wl.kv_dtype == W.BF16 and wl.q_dtype == W.BF16:
        return "mixed_kernel"
    if wl.kv_dtype == W.E4M3 and wl.D == 128 and 1 <= G <= 8 and wl.q_dtype == W.BF16:
        return "decode_mma_kernel"
    if wl.kv_dtype == W.BF16 and wl.D == 128 and 3 <= G <= 8 and wl.q_dtype == W.BF16:
        return "decode_mma_bf16_kernel"
    return "decode_kernel"


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import pa_setup
    import paged_kv_continuous_pa_gb300 as pa
    import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    def barrier():
        if world > 1:
            dist.barrier()

    wl = make_workload(args.workload, args.seqs)
    st = pa_setup.upload(wl, device=dev)
    stream = torch.cuda.current_stream()

    def step():  # pa_step: the append, then the attention as its programmatic dependent
        st.step()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st.status.zero_()

    # A step whose inputs fit a few times in L2 is timed alone after an L2
    # flush: write a buffer twice the L2 (evicts everything), then read
    # another one (so the evicted dirty lines are written back before the
    # step, not during it).  Larger steps run back to back.
    kv_unique = wl.kv_bytes_unique()
    flush = kv_unique <= 4 * L2_BYTES
    if flush:
        fl_w = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        fl_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        fl_w.fill_(1)
        fl_r.max()

    # ---- timed region: K steps (one pa_step call each), each bracketed by events
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches0 = pa.kernel_launches()
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        ev_start.record(stream)
        for i in range(args.steps):
            if flush:
                flush_l2()
            step_ev[i][0].record(stream)
            step()
            step_ev[i][1].record(stream)
        ev_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    launches = pa.kernel_launches() - launches0
    status = int(st.status.item())
    if status != 0:
        raise RuntimeError(f"device status {status} ({pa.status_string(status)}) during the timed steps")
    # the steps' own device time (the flushes between them excluded)
    ms_total = sum(a.elapsed_time(b) for a, b in step_ev) if flush else ev_start.elapsed_time(ev_end)

    # ---- the attention launch alone, K times, for its roofline (same flush rule)
    att_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        if flush:
            flush_l2()
        att_ev[i][0].record(stream)
        st.attend()
        att_ev[i][1].record(stream)
    torch.cuda.synchronize()
    att_ms = [a.elapsed_time(b) for a, b in att_ev]
    ms_total = max_over_ranks(ms_total, dist if world > 1 else None, dev)
    ms_per_step = ms_total / args.steps
    value = job_rows_per_s(wl.n_rows, world, ms_per_step)

    # ---- e2e: the same step through the public API with host buffers
    pin = lambda t: t.detach().cpu().pin_memory()
    h_q, h_k, h_v = pin(st.q), pin(st.k_new), pin(st.v_new)
    h_seq, h_pos, h_bt = pin(st.seq_ids), pin(st.positions), pin(st.block_tables)
    h_out = torch.empty_like(h_q).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_seq, h_pos, h_bt))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        st.q.copy_(h_q, non_blocking=True)
        st.k_new.copy_(h_k, non_blocking=True)
        st.v_new.copy_(h_v, non_blocking=True)
        st.seq_ids.copy_(h_seq, non_blocking=True)
        st.positions.copy_(h_pos, non_blocking=True)
        st.block_tables.copy_(h_bt, non_blocking=True)
        step()
        h_out.copy_(st.out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = max_over_ranks(e2e_ms, dist if world > 1 else None, dev)
    e2e_value = job_rows_per_s(wl.n_rows, world, e2e_ms)

    # ---- roofline of the attention kernel
    alg_bytes = kv_unique + wl.qo_bytes()
    att_avg_ms = statistics.mean(att_ms)
    achieved = alg_bytes / (att_avg_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    src_hash = kernel_source_hash()
    traffic = profiled_traffic(args.workload, src_hash)
    kv_gbs = kv_unique / (att_avg_ms / 1e3) / 1e9
    tiles = None
    if attention_kernel_name(wl) == "mixed_kernel":
        tiles = prefill_tiles_alone(pa, torch, st, wl, max(10, min(args.steps, 50)), stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        leg = OracleLeg(wl, target_s=3.0)
        r, _ = leg.step()
        cpu = {"value": r, "unit": "rows/s", "cores": leg.cores, "kind": "oracle", "sample": leg.sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.description, "rows": wl.n_rows, "kv_dtype": W.DTYPE_NAMES[wl.kv_dtype],
                       "q_dtype": W.DTYPE_NAMES[wl.q_dtype], "kv_bytes_unique": kv_unique,
                       "alg_bytes_per_attention": alg_bytes, "l2": "inputs larger than L2, no flush "
                       f"(KV {kv_unique / 1e9:.2f} GB per step vs 129 MB L2)" if not flush else
                       f"L2 flushed before every step (write {2 * L2_BYTES >> 20} MiB, then read "
                       f"{2 * L2_BYTES >> 20} MiB: the step starts with a clean L2); flush time excluded",
                       "split_tokens": pa.get_split_tokens(), "parallelism": f"replicas x{world}"},
            "kv_read_gbs": kv_gbs,
            "attention_ms": att_avg_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s", "kernel": f"{attention_kernel_name(wl)} (pa_attention)",
                         "kernel_source_hash": src_hash},
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            "gpu_launches": launches,
            **({"prefill_tiles": tiles} if tiles else {}),
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="batched_decode",
                    choices=sorted(W_CONFIG_NAMES))
    ap.add_argument("--seqs", type=int, default=0, help="shrink the workload to this many sequences (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
