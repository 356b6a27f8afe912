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
At N = 1 the default line also carries `workloads`: every config (tiny
decode, batched decode, mixed step with its prefill tiles run alone, shared
prefix, long context, both fp8 variants) timed the same way in the same
process, each with its step and attention times, its HBM fractions (the
attention launch alone, and the whole step with the append's bytes) and its
own clock record.  --no-workloads skips them.

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
# the per-config entries of the default line, in the order they are timed
ALL_WORKLOADS = ("tiny_decode", "batched_decode", "mixed_step", "shared_prefix", "long_context",
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
    only, after the step's append: the warp-specialised tile CTAs, whose
    chunk rows have the mixed launch's bits): tensor-pipe fraction of the tiles.
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
            "peak_source": f"{kind} (MEASURED_PEAKS.json bf16_tflops, burst)", "kernel": "prefill_kernel (chunk tiles only)"}


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
    if name == "long_prefill":  # a prefill step (not a headline config): the tile path at full-GPU size
        return W.long_prefill()
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
        oracle_pools = oracle.workload_pools

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
        # every row in a chunk: the launch of chunk tiles only
        if sum(n for _, n in wl.chunks) == wl.n_rows and min(n for _, n in wl.chunks) >= 16:
            return "prefill_kernel"
        return "mixed_kernel"
    if wl.kv_dtype == W.E4M3 and wl.D == 128 and 1 <= G <= 8 and wl.q_dtype == W.BF16:
        return "decode_mma_kernel"
    if wl.kv_dtype == W.BF16 and wl.D == 128 and 3 <= G <= 8 and wl.q_dtype == W.BF16:
        return "decode_mma_bf16_kernel"
    return "decode_kernel"


class Env:
    """The device, stream and library handles one benchmark process uses."""

    def __init__(self, torch, pa, W, pa_setup, dist, dev, world, rank):
        self.torch, self.pa, self.W, self.pa_setup, self.dist = torch, pa, W, pa_setup, dist
        self.dev, self.world, self.rank = dev, world, rank
        self.stream = torch.cuda.current_stream()

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max_over_ranks(self, x):
        return max_over_ranks(x, self.dist if self.world > 1 else None, self.dev)


def gpu_head_start(torch, launches: int = 0):
    """Queue GPU spinning (about 1 ms, or 60 us for each of `launches` calls
    the host is about to enqueue back to back, whichever is longer) so that the
    host enqueues the timed launches while the GPU is still busy: the events
    then measure device time only, not the host's launch latency in front of
    an idle GPU."""
    try:
        torch.cuda._sleep(max(2_000_000, 120_000 * launches))
    except (AttributeError, RuntimeError):  # pragma: no cover - older or newer torch
        pass


def time_steps(env, st, wl, steps: int, warmup: int):
    """Warm up, then time `steps` pa_step calls (append + attention) and as many
    attention launches alone, each bracketed by CUDA events on the launching
    stream.  A step whose distinct K/V fits a few times in L2 is timed alone
    after an L2 flush (write a buffer twice the L2, which evicts everything,
    then read another one, so the evicted dirty lines are written back before
    the step and not inside it); larger steps run back to back.  Returns a
    dict of times plus the clock record and the library's launch count over
    the timed steps."""
    torch, pa = env.torch, env.pa
    stream = env.stream
    kv_unique = wl.kv_bytes_unique()
    flush = kv_unique <= 4 * L2_BYTES
    if flush:
        fl_w = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=env.dev)
        fl_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device=env.dev)

    def flush_l2():
        fl_w.fill_(1)
        fl_r.max()

    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(env.dev.index) as clk:
        # warm-up steps right before the timed ones (the sampler's start-up can
        # leave the GPU idle for a while), then the timed steps back to back
        for _ in range(warmup):
            if flush:
                flush_l2()
            st.step()
        torch.cuda.synchronize()
        st.status.zero_()
        env.barrier()
        torch.cuda.synchronize()
        launches0 = pa.kernel_launches()
        gpu_head_start(torch)
        ev_start.record(stream)
        for i in range(steps):
            if flush:
                flush_l2()
            step_ev[i][0].record(stream)
            st.step()
            step_ev[i][1].record(stream)
        ev_end.record(stream)
        torch.cuda.synchronize()
        env.barrier()
    launches = pa.kernel_launches() - launches0
    status = int(st.status.item())
    if status != 0:
        raise RuntimeError(f"device status {status} ({pa.status_string(status)}) during the timed steps of {wl.name}")
    # the steps' own device time (the flushes between them excluded)
    ms_total = sum(a.elapsed_time(b) for a, b in step_ev) if flush else ev_start.elapsed_time(ev_end)

    att_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for _ in range(warmup):
        st.attend()
    gpu_head_start(torch)
    for i in range(steps):
        if flush:
            flush_l2()
        att_ev[i][0].record(stream)
        st.attend()
        att_ev[i][1].record(stream)
    torch.cuda.synchronize()
    att_ms = [a.elapsed_time(b) for a, b in att_ev]
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    warm = None
    if flush:
        # the same calls back to back without the flush, labelled: the step's
        # K/V then largely stays in L2, which overstates the HBM rate
        warm_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        gpu_head_start(torch, steps)  # short calls back to back: the host must stay ahead of all of them
        for i in range(steps):
            warm_ev[i][0].record(stream)
            st.attend()
            warm_ev[i][1].record(stream)
        torch.cuda.synchronize()
        warm_att = [a.elapsed_time(b) for a, b in warm_ev]
        warm = {"attention_ms": statistics.mean(warm_att), "attention_ms_median": statistics.median(warm_att),
                "label": "warm L2: no flush between calls, the K/V largely L2-resident; overstates the HBM rate"}
    ms_total = env.max_over_ranks(ms_total)
    l2 = (f"inputs larger than L2, no flush (KV {kv_unique / 1e9:.2f} GB per step vs 129 MB L2)" if not flush else
          f"L2 flushed before every step (write {2 * L2_BYTES >> 20} MiB, then read {2 * L2_BYTES >> 20} MiB: "
          "the step starts with a clean L2); flush time excluded")
    return {"ms_per_step": ms_total / steps, "attention_ms": statistics.mean(att_ms), "launches": launches,
            "ms_per_step_median": statistics.median(step_ms), "attention_ms_median": statistics.median(att_ms),
            "clocks": clk.summary(), "flush": flush, "l2": l2, "warm_l2": warm}


def workload_entry(env, name: str, steps: int, warmup: int, seqs: int = 0):
    """One config under the same clock as the headline: its step and attention
    times, throughput and roofline fractions.  Frees its device memory after."""
    torch, pa, W = env.torch, env.pa, env.W
    wl = make_workload(name, seqs)
    st = env.pa_setup.upload(wl, device=env.dev)
    t = time_steps(env, st, wl, steps, warmup)
    kv_unique = wl.kv_bytes_unique()
    alg = kv_unique + wl.qo_bytes()
    alg_step = alg + wl.append_bytes()
    peak, peak_kind = measured_peaks()
    att_gbs = alg / (t["attention_ms"] / 1e3) / 1e9
    step_gbs = alg_step / (t["ms_per_step"] / 1e3) / 1e9
    src_hash = kernel_source_hash()
    entry = {
        "workload": wl.description, "rows": wl.n_rows, "kv_dtype": W.DTYPE_NAMES[wl.kv_dtype],
        "q_dtype": W.DTYPE_NAMES[wl.q_dtype], "steps": steps, "warmup": warmup,
        "ms_per_step": t["ms_per_step"], "rows_per_s": wl.n_rows / (t["ms_per_step"] / 1e3),
        "attention_ms": t["attention_ms"], "kernel": f"{attention_kernel_name(wl)} (pa_attention)",
        "kv_bytes_unique": kv_unique, "alg_bytes_per_attention": alg, "alg_bytes_per_step": alg_step,
        "kv_read_gbs": kv_unique / (t["attention_ms"] / 1e3) / 1e9,
        "achieved_gbs": att_gbs, "frac": att_gbs / peak, "step_gbs": step_gbs, "step_frac": step_gbs / peak,
        "peak_gbs": peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
        "traffic": profiled_traffic(name, src_hash), "l2": t["l2"], "gpu_launches": t["launches"],
        "clocks": t["clocks"], "ms_per_step_median": t["ms_per_step_median"],
        "attention_ms_median": t["attention_ms_median"],
        "frac_median": alg / (t["attention_ms_median"] / 1e3) / 1e9 / peak,
    }
    if t["warm_l2"] is not None:
        w = t["warm_l2"]
        entry["warm_l2"] = {**w, "frac": alg / (w["attention_ms"] / 1e3) / 1e9 / peak}
    if attention_kernel_name(wl) == "mixed_kernel":
        entry["prefill_tiles"] = prefill_tiles_alone(pa, torch, st, wl, max(10, min(steps, 50)), env.stream)
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def row_groups_entry(env, steps: int, warmup: int):
    """The shared-prefix step with its rows listed prefix by prefix, timed with
    one row per tensor-core CTA and with row groups (pa_set_row_groups: the
    pages all rows of a group share are staged once per CTA).  Output bits are
    the same in every form; only the times differ."""
    torch, pa, W = env.torch, env.pa, env.W
    wl = W.group_by_prefix(W.shared_prefix())
    st = env.pa_setup.upload(wl, device=env.dev)
    alg = wl.kv_bytes_unique() + wl.qo_bytes()
    peak, _ = measured_peaks()
    out = {"workload": wl.description, "rows": wl.n_rows, "times": {}}
    old = pa.get_row_groups()
    try:
        for rg in (1, 2, 4, 8):
            pa.set_row_groups(rg)
            t = time_steps(env, st, wl, steps, warmup)
            out["times"][str(rg)] = {"ms_per_step": t["ms_per_step"], "attention_ms": t["attention_ms"],
                                     "frac": alg / (t["attention_ms"] / 1e3) / 1e9 / peak,
                                     "clocks": t["clocks"]}
    finally:
        pa.set_row_groups(old)
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def long_prefill_entry(env, steps: int, warmup: int):
    """A prefill step of one 4096-token causal chunk: 512 tiles on the
    tensor-core path (the launch of chunk tiles only), enough to occupy every
    SM.  Algorithmic FLOPs: 4 * D per (row, visible key, query head)."""
    import numpy as np
    torch, pa, W = env.torch, env.pa, env.W
    wl = W.long_prefill()
    st = env.pa_setup.upload(wl, device=env.dev)
    t = time_steps(env, st, wl, steps, warmup)
    flops = 4.0 * wl.D * wl.Hq * float(np.sum(wl.positions.astype(np.int64) + 1))
    peak, kind = measured_bf16_tflops()
    tflops = flops / (t["attention_ms"] / 1e3) / 1e12
    out = {"workload": wl.description, "rows": wl.n_rows, "gflop": flops / 1e9, "attention_ms": t["attention_ms"],
           "ms_per_step": t["ms_per_step"], "tflops": tflops, "peak_tflops": peak, "frac": tflops / peak,
           "peak_source": f"{kind} (MEASURED_PEAKS.json bf16_tflops, burst)",
           "kernel": "prefill_kernel (chunk tiles only)", "gpu_launches": t["launches"], "clocks": t["clocks"]}
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_ours(args):
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
    env = Env(torch, pa, W, pa_setup, dist, dev, world, rank)
    stream = env.stream

    wl = make_workload(args.workload, args.seqs)
    st = pa_setup.upload(wl, device=dev)
    t = time_steps(env, st, wl, args.steps, args.warmup)
    ms_per_step = t["ms_per_step"]
    value = job_rows_per_s(wl.n_rows, world, ms_per_step)
    kv_unique = wl.kv_bytes_unique()

    # ---- e2e: the same step through the public API with host buffers.  Every
    # step copies its own inputs from pinned host memory and its output back,
    # as a serving loop does, with the copies on a second stream so that they
    # overlap the neighbouring steps' compute: two device input/output sets,
    # ordered by events (inputs of step k+1 land while step k computes; the
    # output of step k is read back while step k+1 computes).
    pin = lambda x: x.detach().cpu().pin_memory()
    h_in = [pin(x) for x in (st.q, st.k_new, st.v_new, st.seq_ids, st.positions, st.block_tables)]
    h_out = torch.empty_like(h_in[0]).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = h_out.numel() * h_out.element_size()
    d_in = [[torch.empty_like(x) for x in (st.q, st.k_new, st.v_new, st.seq_ids, st.positions, st.block_tables)]
            for _ in range(2)]
    d_out = [torch.empty_like(st.out) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of a set landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step of a set finished
    ev_free = [torch.cuda.Event() for _ in range(2)]  # a set's output read back: the set may take new inputs

    def h2d_copy(k):
        b = k % 2
        with torch.cuda.stream(copy_stream):
            if k >= 2:
                copy_stream.wait_event(ev_free[b])
            for dst, src in zip(d_in[b], h_in):
                dst.copy_(src, non_blocking=True)
            ev_in[b].record(copy_stream)

    def run_step(k):
        b = k % 2
        stream.wait_event(ev_in[b])
        q, kn, vn, seq, pos, bt = d_in[b]
        pa.step(st.pool, q, kn, vn, seq, pos, bt, d_out[b], chunks=wl.chunks, softmax_scale=wl.softmax_scale,
                workspace=st.workspace, status=st.status, stream=stream)
        ev_done[b].record(stream)

    def d2h_copy(k):
        b = k % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_done[b])
            h_out.copy_(d_out[b], non_blocking=True)
            ev_free[b].record(copy_stream)

    def e2e_steps(n):
        h2d_copy(0)
        for k in range(n):
            if k + 1 < n:
                h2d_copy(k + 1)
            run_step(k)
            d2h_copy(k)

    e2e_steps(max(2, args.warmup))
    torch.cuda.synchronize()
    env.barrier()
    # the host's wall clock around the K calls, ending when their results are
    # in host memory: it includes the binding's and the library's host-side
    # work and every launch's latency, not only the device's time
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    e0.record(copy_stream)
    e2e_steps(args.steps)
    e1.record(copy_stream)
    torch.cuda.synchronize()
    e2e_ms = env.max_over_ranks((time.perf_counter() - t_wall) * 1e3 / args.steps)
    e2e_device_ms = e0.elapsed_time(e1) / args.steps
    e2e_value = job_rows_per_s(wl.n_rows, world, e2e_ms)
    del d_in, d_out

    # ---- roofline of the attention kernel
    alg_bytes = kv_unique + wl.qo_bytes()
    att_avg_ms = t["attention_ms"]
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
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ---- every other config under the same clock (one process, one GPU)
    entries = None
    if world == 1 and not args.no_workloads:
        entries = {}
        for name in ALL_WORKLOADS:
            entries[name] = workload_entry(env, name, max(args.steps, 50), max(args.warmup, 3))
        entries["shared_prefix_row_groups"] = row_groups_entry(env, max(args.steps, 20), max(args.warmup, 3))
        entries["long_prefill"] = long_prefill_entry(env, max(args.steps, 50), max(args.warmup, 3))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.description, "rows": wl.n_rows, "kv_dtype": W.DTYPE_NAMES[wl.kv_dtype],
                       "q_dtype": W.DTYPE_NAMES[wl.q_dtype], "kv_bytes_unique": kv_unique,
                       "alg_bytes_per_attention": alg_bytes, "l2": t["l2"],
                       "split_tokens": pa.get_split_tokens(), "parallelism": f"replicas x{world}"},
            "kv_read_gbs": kv_gbs,
            "attention_ms": att_avg_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s", "kernel": f"{attention_kernel_name(wl)} (pa_attention)",
                         "kernel_source_hash": src_hash},
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "timer": "host wall clock, K calls through the public API, ending "
                    "with the results in pinned host memory", "device_ms_per_step": e2e_device_ms,
                    "pipelining": "each step's inputs copied from pinned host memory on a copy stream while the "
                    "previous step computes, its output copied back while the next one computes"},
            "gpu_launches": t["launches"],
            **({"prefill_tiles": tiles} if tiles else {}),
            "clocks": t["clocks"],
            "cpu_baseline": cpu,
            **({"workloads": entries} if entries is not None else {}),
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
                    choices=sorted(W_CONFIG_NAMES) + ["long_prefill"])
    ap.add_argument("--seqs", type=int, default=0, help="shrink the workload to this many sequences (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the selected workload only (no per-config entries)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
