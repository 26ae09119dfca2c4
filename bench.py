"""Benchmark: MLA decode (weight-absorbed, paged latent cache) on GB300.

One step = one pass of the whole hot path over one decode batch: plan
(split-KV partition) + q-absorb bmm + split-KV latent attention + LSE combine
+ W_UV bmm, all through the C ABI of libmla_decode.so, inputs resident in HBM.

Prints ONE JSON line (rank 0).  value = latent-cache GB/s (1152 B per cached
token per sequence, read once per step) summed over all ranks.  Also reports
TFLOP/s (2176 FLOP per query row and key + the two bmms) and decode tokens/s,
the roofline of the dominant kernel (the attention step) against the measured
HBM copy bandwidth, an end-to-end figure through the same C ABI with host
buffers (every step copies all of its inputs up from pinned host memory and
reads its result back; the next step's copy overlaps this step's compute),
and the fp64 CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
                  [--weights bf16|fp8] [--no-per-config]

The attention kernel's time (the roofline's "achieved") is always taken over
ATTEND_LAUNCHES back-to-back launches, whatever --steps is.  "per_config"
repeats the step and attention timing (CONFIG_STEPS steps, ATTEND_LAUNCHES
launches) on every full-size workload, so one line carries all of them.

--weights fp8 gives the two bmms W_UK and W_UV as FP8 E4M3 codes with one
fp32 scale per 128 x 128 block (decompressed to bf16 inside the bmm kernels).

N > 1 runs under torch.distributed.run, one independent replica per GPU
(the path needs no exchange between GPUs: weak scaling).
"""
import argparse
import copy
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mla_decode_attention_uk_gb300.inputs import WORKLOADS, workload_inputs  # noqa: E402

METRIC = "MLA decode latent-KV GB/s, TFLOPS & tokens/s vs GB300 roofline (1 GPU)"
# The headline runs on the largest single-GPU workload (811 MB of latent
# cache, ~200 GFLOP per step); every other full-size workload is measured in
# the same run and reported under "per_config".
DEFAULT_WORKLOAD = "full_head"
PER_CONFIG = ("tp_shard", "long", "full_head", "mixed_spec", "draft_q8")
PER_GRAPH = 10  # decode steps captured in one CUDA graph replay
ATTEND_LAUNCHES = 300  # back-to-back launches that time the attention kernel
CONFIG_STEPS = 300  # graph-replayed steps that time each per-config workload
BYTES_PER_TOKEN = 1152          # 576 bf16 per cached token
FLOP_PER_ROW_KEY = 2 * (576 + 512)
FLOP_PER_ROW_BMM = 2 * 2 * 128 * 512


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def decode_source_hash():
    h = hashlib.sha256()
    for f in ("decode.cu", "ptx.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "mla_decode_attention_uk_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per attention launch from the committed ncu summary, if the
    kernel source is unchanged since the capture; else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != decode_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def workload_stats(inp, fp8_weights=False):
    B, T, H = inp.q.shape[:3]
    sum_len = int(inp.seq_lens.sum())
    rows_keys = 0
    for L in inp.seq_lens.tolist():
        for t in range(T):
            rows_keys += H * (L - T + t + 1)
    cache_bytes = BYTES_PER_TOKEN * sum_len
    weight_bytes = H * 2 * (128 * 512 * 2)
    if fp8_weights:  # one byte per weight plus one fp32 scale per 128 x 128 block
        weight_bytes = H * 2 * (128 * 512 + 4 * 4)
    flops = FLOP_PER_ROW_KEY * rows_keys + FLOP_PER_ROW_BMM * B * T * H
    return dict(B=B, T=T, H=H, sum_len=sum_len, cache_bytes=cache_bytes,
                weight_bytes=weight_bytes, flops=flops, attn_flops=FLOP_PER_ROW_KEY * rows_keys,
                tokens=B * T)


def attention_roofline(stats, attend_s, hbm, bf16, peak_src, traffic):
    """Roofline object of the attention kernel (the dominant one): bound by
    the slower of streaming the latent cache at the measured copy bandwidth
    (GB/s) and its FLOPs at the measured bf16 peak (TF/s); achieved figures
    are algorithmic bytes / FLOPs over the kernel's average launch time."""
    attend_gbs = stats["cache_bytes"] / attend_s / 1e9
    attend_tf = stats["attn_flops"] / attend_s / 1e12
    if stats["attn_flops"] / (bf16 * 1e12) > stats["cache_bytes"] / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": attend_tf, "peak": bf16, "unit": "TFLOP/s",
                "frac": attend_tf / bf16,
                "peak_source": peak_src + " (bf16_tflops, MEASURED_PEAKS.json)"}
    else:
        roof = {"bound": "hbm", "achieved": attend_gbs, "peak": hbm, "unit": "GB/s",
                "frac": attend_gbs / hbm,
                "peak_source": peak_src + " (hbm_gbs, MEASURED_PEAKS.json)"}
    roof.update({"traffic": traffic, "kernel": "decode_kernel (attend step)",
                 "kernel_us": attend_s * 1e6, "hbm_frac": attend_gbs / hbm,
                 "tensor_frac": attend_tf / bf16})
    return roof


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def _one(self):
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                "--format=csv,noheader,nounits"], capture_output=True, text=True,
                               timeout=10)
            for line in r.stdout.strip().splitlines():
                self.rows.append([x.strip() for x in line.split(",")])
        except Exception:
            pass

    def start(self):
        self._one()
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                          "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=10)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            for line in out.strip().splitlines():
                self.rows.append([x.strip() for x in line.split(",")])
        self._one()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample(inp_cpu, budget_s):
    """Pick a bounded sample of query rows for the fp64 oracle: whole leading
    sequences while they fit the budget, else the first rows of sequence 0.
    Each sequence's cache bytes (and its tokens) are attributed evenly to its
    T*H query rows, so the sample's throughput is in the workload's units.
    Returns (rows or None, sample bytes, sample flops, sample tokens, text)."""
    import oracle
    B, T, H = inp_cpu.q.shape[:3]
    TH = T * H
    lens = inp_cpu.seq_lens.tolist()
    # calibrate on a few rows of sequence 0
    probe = list(range(min(TH, 4)))
    t0 = time.perf_counter()
    oracle.decode(inp_cpu.q, inp_cpu.cache, inp_cpu.block_table, inp_cpu.seq_lens, inp_cpu.w_uk,
                  inp_cpu.w_uv, inp_cpu.scale, rows=probe)
    per_row = (time.perf_counter() - t0) / len(probe) / max(1, lens[0])  # s per row-key
    par = max(1, oracle.threads())
    rows, keys = [], 0
    for b in range(B):
        for r in range(TH):
            rows.append(b * TH + r)
            keys += lens[b]
            if keys * per_row / par >= budget_s:
                break
        else:
            continue
        break
    # The calibration ignores how well the oracle's threads scale on a small
    # sample: time the sample itself and shrink it until it fits the budget.
    for _ in range(4):
        t0 = time.perf_counter()
        oracle.decode(inp_cpu.q, inp_cpu.cache, inp_cpu.block_table, inp_cpu.seq_lens,
                      inp_cpu.w_uk, inp_cpu.w_uv, inp_cpu.scale, rows=rows)
        dt = time.perf_counter() - t0
        if dt <= 1.3 * budget_s or len(rows) == 1:
            break
        rows = rows[:max(1, int(len(rows) * budget_s / dt))]
    nbytes = sum(BYTES_PER_TOKEN * lens[row // TH] / TH for row in rows)
    flops = sum(FLOP_PER_ROW_KEY * (lens[row // TH] - T + (row % TH) // H + 1) + FLOP_PER_ROW_BMM
                for row in rows)
    tokens = len(rows) / H
    text = "%d query rows (first %d sequence(s)) of %d; cache bytes attributed per row" % (
        len(rows), rows[-1] // TH + 1, B * TH)
    return rows, nbytes, flops, tokens, text


def time_oracle(inp_cpu, budget_s):
    import oracle
    rows, nbytes, flops, tokens, text = oracle_sample(inp_cpu, budget_s)
    t0 = time.perf_counter()
    oracle.decode(inp_cpu.q, inp_cpu.cache, inp_cpu.block_table, inp_cpu.seq_lens, inp_cpu.w_uk,
                  inp_cpu.w_uv, inp_cpu.scale, rows=rows)
    dt = time.perf_counter() - t0
    return dt, nbytes, flops, tokens, text


def dist_setup(n_gpus):
    if n_gpus > 1 or "RANK" in os.environ:
        import torch.distributed as dist
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        local = int(os.environ.get("LOCAL_RANK", "0"))
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def max_over_ranks(x, dist, dev):
    """The largest value of x over all ranks (the job takes as long as its
    slowest rank); x itself on a single process."""
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores,
    each step a bounded row sample of the same workload."""
    rank, world, local, dist = dist_setup(args.gpus)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    import oracle
    inp = workload_inputs(args.workload)
    if args.weights == "fp8":  # the oracle decompresses the FP8 weights, then decodes
        from mla_decode_attention_uk_gb300.inputs import quantize_fp8_blockwise
        inp.w_uk = oracle.dequant_fp8_weight(*quantize_fp8_blockwise(inp.w_uk))
        inp.w_uv = oracle.dequant_fp8_weight(*quantize_fp8_blockwise(inp.w_uv))
    budget = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    rows, nbytes, flops, tokens, text = oracle_sample(inp, budget)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk, inp.w_uv,
                      inp.scale, rows=rows)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    value = nbytes / per_step / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "note": WORKLOADS[args.workload].note,
                   "weights": "fp8 e4m3, 128x128 block scales" if args.weights == "fp8"
                   else "bf16"},
        "tflops": flops / per_step / 1e12, "tokens_per_s": tokens / per_step,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": text},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


class WorkloadRunner:
    """One workload's inputs on the device, a workspace through the binding,
    and CUDA graphs of PER_GRAPH consecutive decode steps and of PER_GRAPH
    attention launches (same kernels and arguments as host launches; the
    graphs keep host launch overhead from starving the GPU on small batches)."""

    def __init__(self, name, dev, fp8, use_graph=True):
        from mla_decode_attention_uk_gb300 import binding
        self.binding = binding
        self.name = name
        self.dev = dev
        self.fp8 = fp8
        self.inp_cpu = workload_inputs(name)
        self.stats = workload_stats(self.inp_cpu, fp8)
        g = self.g = self.inp_cpu.to(dev)
        if fp8:
            from mla_decode_attention_uk_gb300.inputs import quantize_fp8_blockwise
            uk8, uk_s = quantize_fp8_blockwise(self.inp_cpu.w_uk)
            uv8, uv_s = quantize_fp8_blockwise(self.inp_cpu.w_uv)
            self.wts = {k: (t, t.to(dev)) for k, t in (("uk8", uk8), ("uk_s", uk_s),
                                                       ("uv8", uv8), ("uv_s", uv_s))}
        else:
            self.wts = {"w_uk": (self.inp_cpu.w_uk, g.w_uk), "w_uv": (self.inp_cpu.w_uv, g.w_uv)}
        self.W = {k: v[1] for k, v in self.wts.items()}
        self.m = binding.MlaDecode(binding.dims_for(g.q, g.cache, g.block_table), dev)
        B, T, H = self.stats["B"], self.stats["T"], self.stats["H"]
        self.out = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B, T, H, dtype=torch.float32, device=dev)
        self.use_graph = use_graph
        self.graph_step = self.graph_attend = None

    # -- the path, one call per step of it
    def absorb(self):
        if self.fp8:
            self.m.absorb_fp8w(self.g.q, self.W["uk8"], self.W["uk_s"])
        else:
            self.m.absorb(self.g.q, self.W["w_uk"])

    def attend(self):
        g = self.g
        self.m.attend(g.cache, g.block_table, g.seq_lens, g.scale, self.lse)

    def combine(self):
        self.m.combine(self.g.scale, self.lse)

    def up_project(self):
        if self.fp8:
            self.m.up_project_fp8w(self.W["uv8"], self.W["uv_s"], self.out)
        else:
            self.m.up_project(self.W["w_uv"], self.out)

    def plan(self, g=None):
        self.m.plan((self.g if g is None else g).seq_lens)

    def step(self):
        # One decode step as a caller makes it: the plan, then the whole run
        # (absorb, attend, combine, up-project) in one call.  The per-step
        # calls above serve the --breakdown timings.
        self.plan()
        self.run_all()

    def run_all(self, g=None, W=None):
        # g, W: another device copy of the inputs and weights (the end-to-end
        # run alternates two); by default the runner's own.
        g = self.g if g is None else g
        W = self.W if W is None else W
        if self.fp8:
            self.m.run_fp8w(g.q, g.cache, g.block_table, g.seq_lens, W["uk8"], W["uk_s"], W["uv8"],
                            W["uv_s"], g.scale, self.out, self.lse)
        else:
            self.m.run(g.q, g.cache, g.block_table, g.seq_lens, W["w_uk"], W["w_uv"], g.scale,
                       self.out, self.lse)

    def check(self, where):
        st = self.m.check()
        if st != 0:
            raise SystemExit("%s: device status %d %s" % (self.name, st, where))

    def prepare(self, warmup):
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        self.check("after warm-up")
        if not self.use_graph:
            return
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            self.step()
            self.attend()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        self.graph_step, self.graph_attend = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_step):
            for _ in range(PER_GRAPH):
                self.step()
        with torch.cuda.graph(self.graph_attend):
            for _ in range(PER_GRAPH):
                self.attend()
        torch.cuda.synchronize()
        for _ in range(max(1, warmup // PER_GRAPH)):
            self.graph_step.replay()
        torch.cuda.synchronize()

    def per_call(self):
        return PER_GRAPH if self.graph_step is not None else 1

    def steps_call(self):
        return self.graph_step.replay if self.graph_step is not None else self.step

    def attends_call(self):
        return self.graph_attend.replay if self.graph_attend is not None else self.attend

    def time_calls(self, fn, calls):
        """Seconds per call of fn over `calls` back-to-back calls (CUDA events
        on the launching stream, synchronised on both sides)."""
        stream = torch.cuda.current_stream()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(calls):
            fn()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / 1e3 / calls

    def time_attend(self, launches=ATTEND_LAUNCHES):
        """Average attention-kernel launch time over `launches` back-to-back
        launches (inputs larger than L2: every launch streams the cache)."""
        n = max(1, launches // self.per_call())
        return self.time_calls(self.attends_call(), n) / self.per_call(), n * self.per_call()

    def free(self):
        self.graph_step = self.graph_attend = None
        self.g = self.W = self.wts = self.m = self.out = self.lse = None


def per_config_entry(r, step_s, attend_s, attend_launches, hbm, bf16, peak_src):
    st = r.stats
    roof = attention_roofline(st, attend_s, hbm, bf16, peak_src, ncu_traffic(r.name))
    return {
        "note": WORKLOADS[r.name].note, "step_us": step_s * 1e6,
        "value_gbs": st["cache_bytes"] / step_s / 1e9, "tflops": st["flops"] / step_s / 1e12,
        "tokens_per_s": st["tokens"] / step_s,
        "attend_us": attend_s * 1e6, "attend_launches": attend_launches,
        "bound": roof["bound"], "frac": roof["frac"], "hbm_frac": roof["hbm_frac"],
        "tensor_frac": roof["tensor_frac"], "traffic": roof["traffic"],
        "cache_bytes": st["cache_bytes"], "attn_flops": st["attn_flops"],
        "t_roof_us": 1e6 * max((st["cache_bytes"] + st["weight_bytes"]) / (hbm * 1e9),
                               st["flops"] / (bf16 * 1e12)),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch every step from the host")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only --workload (e.g. for short profiler runs)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8"],
                    help="W_UK / W_UV as bf16, or FP8 E4M3 with 128x128 block scales")
    ap.add_argument("--breakdown", action="store_true",
                    help="also time each step of the path alone (graph replays)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    from mla_decode_attention_uk_gb300 import binding
    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    fp8 = args.weights == "fp8"
    hbm, bf16, bf16_sus, peak_src = measured_peaks()

    r = WorkloadRunner(args.workload, dev, fp8, use_graph=not args.no_graph)
    launches_per_step = 1 + binding.kernels_per_run(r.m.dims, fp8)  # plan + the run's kernels
    stats, inp_cpu, g = r.stats, r.inp_cpu, r.g
    B, T, H = stats["B"], stats["T"], stats["H"]
    r.prepare(args.warmup)
    per_graph = r.per_call()
    rem = args.steps % per_graph
    graph_rem = None
    if rem and r.graph_step is not None:
        graph_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_rem):
            for _ in range(rem):
                r.step()
        torch.cuda.synchronize()
    run_steps = r.steps_call()
    run_rem = graph_rem.replay if graph_rem is not None else (lambda: None)

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    t_start.record(stream)
    for i in range(args.steps // per_graph):  # exactly args.steps steps
        run_steps()
    run_rem()
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks.stop()
    r.check("in timed region")
    want_out, want_lse = r.out.cpu(), r.lse.cpu()  # for the end-to-end check below
    elapsed = t_start.elapsed_time(t_end) / 1e3

    # Average duration of the dominant kernel (attention step): CUDA events on
    # the launching stream around ATTEND_LAUNCHES back-to-back launches.
    attend_s, attend_launches = r.time_attend()
    r.check("while timing the attention step")
    elapsed = max_over_ranks(elapsed, dist, dev)
    per_step = elapsed / args.steps

    # ---- end to end through the same C ABI with host buffers
    # Every step copies all of its inputs from pinned host memory and reads
    # its result back, in the form of a serving loop: two device copies of
    # the inputs are used in turn, and step i + 1's inputs go up on a copy
    # stream while step i computes (the copy into a set waits until the step
    # that last read it has finished).
    in_keys = ("q", "cache", "block_table", "seq_lens")
    w_keys = list(r.wts)
    host = [(getattr(inp_cpu, k).pin_memory(), k) for k in in_keys]
    host_w = [(r.wts[k][0].pin_memory(), k) for k in w_keys]
    g_alt = copy.copy(g)
    for k in in_keys:
        setattr(g_alt, k, torch.empty_like(getattr(g, k)))
    dsets = [(g, r.W), (g_alt, {k: torch.empty_like(r.W[k]) for k in w_keys})]
    out_h = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    lse_h = torch.empty(r.lse.shape, dtype=r.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t, _ in host + host_w)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in dsets]
    consumed = [torch.cuda.Event() for _ in dsets]
    for ev in consumed:
        ev.record(stream)

    def e2e_step(i):
        gj, wj = dsets[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[i % 2])
            for t, k in host:
                getattr(gj, k).copy_(t, non_blocking=True)
            for t, k in host_w:
                wj[k].copy_(t, non_blocking=True)
            copied[i % 2].record(copy_stream)
        stream.wait_event(copied[i % 2])
        r.plan(gj)
        r.run_all(gj, wj)
        consumed[i % 2].record(stream)
        out_h.copy_(r.out, non_blocking=True)
        lse_h.copy_(r.lse, non_blocking=True)

    n_e2e = max(3, min(args.e2e_steps, args.steps))
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e0.record(stream)
    copy_stream.wait_stream(stream)  # no copy of the timed steps starts before e0
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    r.check("in the end-to-end run")
    # The same inputs through either device set give the same bits.
    if not (torch.equal(out_h, want_out) and torch.equal(lse_h, want_lse)):
        raise SystemExit("end-to-end run: results read back differ from the timed steps'")
    e2e_s = e0.elapsed_time(e1) / 1e3 / n_e2e
    e2e_s = max_over_ranks(e2e_s, dist, dev)

    breakdown = None
    if args.breakdown:
        stages = {"plan": r.plan, "absorb": r.absorb, "attend": r.attend, "combine": r.combine,
                  "up_project": r.up_project}
        breakdown = {}
        for name, fn in stages.items():
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                fn()
            for _ in range(5):
                gr.replay()
            breakdown[name] = r.time_calls(gr.replay, 200) * 1e6
        r.check("in the per-stage timing")

    wts_host = {k: v[0] for k, v in r.wts.items()}  # the oracle leg below needs them

    # ---- every full-size workload, same kernels, measured in this run
    per_config = None
    if not args.no_per_config:
        per_config = {args.workload: per_config_entry(r, per_step, attend_s, attend_launches,
                                                      hbm, bf16, peak_src)}
        r.free()
        cfg_clocks = ClockSampler(local)
        cfg_clocks.start()
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            rc = WorkloadRunner(name, dev, fp8, use_graph=not args.no_graph)
            rc.prepare(args.warmup)
            step_s = rc.time_calls(rc.steps_call(), max(1, CONFIG_STEPS // rc.per_call())) / \
                rc.per_call()
            a_s, a_n = rc.time_attend()
            rc.check("in the per-config timing")
            per_config[name] = per_config_entry(rc, step_s, a_s, a_n, hbm, bf16, peak_src)
            rc.free()
            torch.cuda.empty_cache()
        cfg_clocks.stop()
        per_config["clocks"] = cfg_clocks.summary()

    if rank != 0:
        dist.destroy_process_group()
        return

    gbs = world * stats["cache_bytes"] / per_step / 1e9
    tflops = world * stats["flops"] / per_step / 1e12
    roof = attention_roofline(stats, attend_s, hbm, bf16, peak_src, ncu_traffic(args.workload))
    roof["launches_timed"] = attend_launches
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "batch": B, "q_len": T, "heads": H,
                   "sum_seq_len": stats["sum_len"],
                   "seq_len": int(inp_cpu.seq_lens[0]) if len(set(inp_cpu.seq_lens.tolist())) == 1
                   else "varied", "page": 64, "parallelism": "replica x%d" % world,
                   "weights": "fp8 e4m3, 128x128 block scales" if fp8 else "bf16",
                   "l2": "inputs larger than L2 (latent cache %.0f MB > 129 MB L2)" %
                         (stats["cache_bytes"] / 1e6)},
        "tflops": tflops, "tokens_per_s": world * stats["tokens"] / per_step,
        "roofline_step": {"t_roof_us": 1e6 * max(
            (stats["cache_bytes"] + stats["weight_bytes"]) / (hbm * 1e9),
            stats["flops"] / (bf16 * 1e12)), "hbm_frac": gbs / world / hbm,
            "tensor_frac": tflops / world / bf16},
        "roofline": roof,
        "e2e": {"value": world * stats["cache_bytes"] / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3},
        "gpu_launches": args.steps * launches_per_step,
        "launch_mode": ("cuda_graph, %d steps per replay" % per_graph) if per_graph > 1 else "host",
        "clocks": clocks.summary(),
    }
    if breakdown is not None:
        line["stage_us"] = breakdown
    if per_config is not None:
        line["per_config"] = per_config
    if not args.no_cpu_baseline:
        import oracle
        inp_or = inp_cpu
        if fp8:  # the oracle decompresses the FP8 weights, then decodes
            inp_or = copy.copy(inp_cpu)
            inp_or.w_uk = oracle.dequant_fp8_weight(wts_host["uk8"], wts_host["uk_s"])
            inp_or.w_uv = oracle.dequant_fp8_weight(wts_host["uv8"], wts_host["uv_s"])
        dt, nbytes, flops, tokens, text = time_oracle(inp_or, budget_s=15.0)
        line["cpu_baseline"] = {"value": nbytes / dt / 1e9, "unit": "GB/s",
                                "cores": oracle.threads(), "kind": "oracle", "sample": text,
                                "seconds": dt, "tflops": flops / dt / 1e12}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
