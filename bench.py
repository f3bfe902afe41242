#!/usr/bin/env python
"""Benchmark of the GB300 attention step through its C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]

One step = one pass of the whole step over one batch of synthetic input: da_rope_tables_build,
da_kv_cache_update, then da_attn_prefill for the prefill chunks and da_attn_decode for the decode tokens,
for every layer of the workload. Default workload: the Qwen3-8B-shaped prefill (4 x 2048 tokens, Hq 32,
Hkv 8, d 128, q/k RMSNorm). Inputs are resident in HBM when timing starts; L2 (129 MB) is flushed by a
256 MB write before every timed step, outside the timed events. Each timed step has events only around
it (its kernels may overlap one another's launch through programmatic dependent launch); the per-stage
breakdown and the kernel roofline come from a second pass with an event after every stage. Prints one JSON
line (rank 0).

Multi-GPU: the step does not exchange data between GPUs; N ranks run N independent replicas of the
workload (weak scaling), and the time is the maximum over ranks.

--impl reference times the fp64 CPU oracle (single-threaded) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn decode HBM GB/s (frac of peak); prefill attn TFLOP/s; tokens/s"
DEFAULT_WORKLOAD = "qwen3_8b_prefill"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Bounded samples of each workload for the CPU oracle: (prefill chunk indices, decode token indices, KV heads
# or None for all) per layer. "baseline" is the one-shot figure in the native line (about 5-30 s of one
# core); "step" is what the reference arm repeats once per step, so that warm-up + steps end in minutes.
ORACLE_SAMPLES = {
    "baseline": {
        "tiny_prefill_fp32": ([0], [], None),
        "qwen3_8b_prefill": ([0], [], None),
        "mistral_swa_decode": ([], list(range(16)), None),
        "llama31_8b_long_decode": ([], [0, 1], None),
        "phi4_gemma2_mixed": ([0], list(range(16)), None),
    },
    "step": {
        "tiny_prefill_fp32": ([0], [], None),
        "qwen3_8b_prefill": ([0], [], 1),
        "mistral_swa_decode": ([], list(range(4)), None),
        "llama31_8b_long_decode": ([], [0], 1),
        "phi4_gemma2_mixed": ([0], list(range(4)), 1),
    },
    # split into (chunk or token, KV head) units over every host core: the whole Qwen3, Mistral and Llama
    # workloads, a quarter of the mixed one's chunks and decode tokens
    "allcores": {
        "tiny_prefill_fp32": ([0], [], None),
        "qwen3_8b_prefill": ([0, 1, 2, 3], [], None),
        "mistral_swa_decode": ([], list(range(64)), None),
        "llama31_8b_long_decode": ([], list(range(16)), None),
        "phi4_gemma2_mixed": ([0, 1], list(range(30)), None),
    },
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--scale", choices=["full", "profile"], default="full",
                    help="profile: the same head shapes with bounded caches (a few GB), for profiler captures")
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--kv-block", type=int, default=0,
                    help="0: contiguous caches; N > 0: a paged pool of N-position blocks in shuffled order "
                         "(da_*_paged entry points)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single", action="store_true",
                    help="time only --workload (the default run also times the decode and mixed workloads)")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)   # internal: child process
    ap.add_argument("--sample-kind", default="baseline", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and workload, if the kernel's
    source is unchanged since the capture (the summary records the source's sha256); else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if line.startswith("<!-- ") and "=" in line:
            k, v = line[5:].rstrip().rstrip("-> ").split("=", 1)
            fields[k.strip()] = v.strip()
    src = fields.get("source")
    if not src or "dram_bytes_per_launch" not in fields:
        return None
    digest = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()
    if digest != fields.get("source_sha256"):
        return None
    return int(float(fields["dram_bytes_per_launch"]))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [ln.split(", ") for ln in out.strip().splitlines() if ln.count(",") >= 8]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": "warm-up and timed steps"}


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def reduce_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def host_link_gbs(dev, nbytes=128 << 20, reps=5):
    """Host <-> device bandwidth of plain pinned copies (128 MB, best of 5 each way, CUDA events): the bound on
    `e2e`, whose steps move their inputs up and their outputs down through the same link."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            dst.copy_(src, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out[name] = nbytes / (best / 1e3) / 1e9
    del h, d
    return out


def headline(work, seconds):
    """(value, unit, tokens/s) of `work` done in `seconds`: TFLOP/s when the step has prefill, else GB/s."""
    if work["prefill_flops"] > 0:
        return (work["prefill_flops"] + work["decode_flops"]) / seconds / 1e12, "TFLOP/s", work["tokens"] / seconds
    return work["decode_bytes"] / seconds / 1e9, "GB/s", work["tokens"] / seconds


# ---------------------------------------------------------------------------------------------- oracle leg

def cpu_model():
    """The host CPU's model name (lscpu's "Model name", else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def oracle_sample_child(workload, kind, iters):
    """Runs in a fresh process: builds the workload once, times the oracle `iters` times on the bounded
    sample, prints one JSON line with the per-iteration seconds.

    kind "baseline"/"step": single-threaded, the sample run in order. kind "allcores": the sample cut into
    units of one (chunk or decode token, KV head group), run by a pool of one thread per host core (numpy
    and BLAS release the interpreter lock in their array loops; BLAS itself is held to one thread per call),
    timed from the first unit's start to the last unit's end."""
    import concurrent.futures as cf

    import torch

    from decoder_attention_gb300 import inputs, work as W
    from oracle import step as ostep
    torch.set_num_threads(1)
    chunks, dec, kvh = ORACLE_SAMPLES[kind][workload]
    num = inputs.NUMBERS[workload]
    gen_dev = "cuda" if (num in (3, 4, 5) and torch.cuda.is_available()) else "cpu"
    wl = inputs.make(num, scale="full", device=gen_dev)
    if kind == "allcores":
        hkv = wl.layers[0].num_key_value_heads
        samples = [inputs.subset(c, cs, ds, device="cpu", kv_heads=1, kv_first=g)
                   for c in wl.layers for cs, ds in [([b], []) for b in chunks] + [([], [t]) for t in dec]
                   for g in range(hkv)]
    else:
        samples = [inputs.subset(c, chunks, dec, device="cpu", kv_heads=kvh) for c in wl.layers]
    n_layers = len(wl.layers)
    del wl
    if gen_dev == "cuda":
        torch.cuda.empty_cache()
    tot = {}
    for s in samples:
        for k, v in W.layer_call_work(s).items():
            tot[k] = tot.get(k, 0) + v
    if kind == "allcores":      # each token was counted once per KV-head unit
        for k in ("tokens", "prefill_tokens", "decode_tokens"):
            tot[k] = tot.get(k, 0) // hkv
    secs = []
    cores = 1
    if kind == "allcores":
        cores = os.cpu_count() or 1
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            for _ in range(iters):
                t0 = time.perf_counter()
                list(ex.map(ostep.run_layer_call, samples))
                secs.append(time.perf_counter() - t0)
        desc = (f"{len(chunks)} prefill chunk(s) and {len(dec)} decode token(s) per layer x {n_layers} layer(s), "
                f"as {len(samples)} (chunk or token, KV head) units over {cores} threads; fp64 numpy")
    else:
        for _ in range(iters):
            t0 = time.perf_counter()
            for s in samples:
                ostep.run_layer_call(s)
            secs.append(time.perf_counter() - t0)
        heads = "all heads" if kvh is None else f"{kvh} KV head(s) and their query heads"
        desc = (f"{len(chunks)} prefill chunk(s) and {len(dec)} decode token(s), {heads}, per layer x "
                f"{n_layers} layer(s); single-threaded fp64 numpy")
    print(json.dumps({"seconds": secs, "sample": desc, "work": tot, "cores": cores}))


def run_oracle_sample(workload, kind="baseline", iters=1):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload,
                          "--sample-kind", kind, "--steps", str(iters)],
                         capture_output=True, text=True, env=env, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError(f"oracle sample failed:\n{res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


def main_reference(args):
    rank, world, _ = dist_init(args)
    if rank != 0:
        return 0
    from decoder_attention_gb300 import inputs
    r = run_oracle_sample(args.workload, "step", args.warmup + args.steps)
    sec = statistics.median(r["seconds"][args.warmup:])
    value, unit, tps = headline(r["work"], sec)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "number": inputs.NUMBERS[args.workload], "sample": r["sample"]},
            "tokens_per_s": tps,
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": r["sample"],
                             "host_cores": os.cpu_count()},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------------------------- native leg

def measure_native(args, workload, dev, world, rank, with_e2e=True):
    """Times one workload through the C ABI on `dev` (inputs resident in HBM; L2 flushed before every timed
    step, outside the step's events) and returns its record: the median step time (the mean beside it), the
    step's breakdown, the roofline of the dominant kernel (and of both halves when the step has prefill and
    decode), e2e through host buffers, launch count and clocks. The workload's tensors are freed on return."""
    import torch

    from decoder_attention_gb300 import _abi, inputs, step as S, work as W

    num = inputs.NUMBERS[workload]
    wl = inputs.make(num, scale=args.scale if num in (3, 4, 5) else "full", device=dev)
    pools = []
    if args.kv_block > 0:
        for li, c in enumerate(wl.layers):
            pools.append(inputs.paged_from_contiguous(c.k_cache, c.v_cache, args.kv_block, seed=1000 + li))

    def make_step(c, li):
        if not pools:
            return S.AttentionStep(c)
        kp, vp, table = pools[li]
        return S.PagedAttentionStep(c, kp, vp, table, args.kv_block)

    steps = [make_step(c, li) for li, c in enumerate(wl.layers)]
    work = W.workload_work(wl)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def run_step():
        for st in steps:
            st.run()

    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    clocks.mark_start()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        run_step()
    torch.cuda.synchronize()
    _abi.check_device_error()

    # ------------------------------------------------------------------ timed region
    # Whole steps with events only around each step: the kernels of a step follow one another with no event
    # in between, so a kernel may start (programmatic dependent launch) while the one before it finishes.
    n_layers = len(steps)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        sev[i][0].record(stream)
        run_step()
        sev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    _abi.check_device_error()
    step_ms = [a.elapsed_time(b) for a, b in sev]

    # Stage breakdown: a second pass of the same steps with an event after every stage (each event closes
    # the stage before it, so these stages start only when the previous one has ended).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(1 + 3 * n_layers)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        e = ev[i]
        e[0].record(stream)
        for li, st in enumerate(steps):
            # a stage with no tokens records no event (an empty event interval still costs ~2 us of the step)
            st.update()
            e[1 + 3 * li].record(stream)
            if st.call.n_prefill:
                st.prefill()
                e[2 + 3 * li].record(stream)
            if st.call.n_decode:
                st.decode()
                e[3 + 3 * li].record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    _abi.check_device_error()

    def marks(e, li):   # (after update, after prefill, after decode) of layer li; an empty stage adds no event
        a = e[1 + 3 * li]
        b = e[2 + 3 * li] if steps[li].call.n_prefill else a
        return a, b, (e[3 + 3 * li] if steps[li].call.n_decode else b)

    def interval(x, y):
        return 0.0 if x is y else x.elapsed_time(y)

    pf_ms = [sum(interval(*marks(e, li)[:2]) for li in range(n_layers)) for e in ev]
    dec_ms = [sum(interval(*marks(e, li)[1:]) for li in range(n_layers)) for e in ev]
    pre_ms = [sum((e[0] if li == 0 else marks(e, li - 1)[2]).elapsed_time(marks(e, li)[0]) for li in range(n_layers))
              for e in ev]
    ms = statistics.median(step_ms)
    ms_all = reduce_max(ms, world)
    clock_info = clocks.stop()

    value_1, unit, _ = headline(work, ms_all / 1e3)
    peaks, peak_kind = load_peaks()
    parts = {}
    if work["prefill_flops"] > 0:
        kms = statistics.median(pf_ms)
        achieved = work["prefill_flops"] / (kms / 1e3) / 1e12
        parts["prefill"] = {
            "kernel": "prefill_kernel (tcgen05)", "bound": "tensor", "achieved": achieved,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "peak_kind": f"bf16 dense burst, of {peak_kind}", "launch_ms": kms / n_layers,
            "launches_per_step": n_layers, "algorithmic_flops_per_launch": work["prefill_flops"] / n_layers,
            "traffic": None if (pools or n_layers > 1) else load_traffic("prefill_kernel", workload)}
    if work["decode_bytes"] > 0:
        kms = statistics.median(dec_ms)
        achieved = work["decode_bytes"] / (kms / 1e3) / 1e9
        parts["decode"] = {
            "kernel": "decode_kernel + merge_kernel (one da_attn_decode call)", "bound": "hbm",
            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "peak_kind": f"HBM copy, of {peak_kind}", "launch_ms": kms / n_layers, "launches_per_step": n_layers,
            "algorithmic_bytes_per_launch": work["decode_bytes"] / n_layers,
            "traffic": None if (pools or n_layers > 1) else load_traffic("decode_kernel", workload)}
    roof = parts["prefill"] if "prefill" in parts else parts["decode"]

    # ------------------------------------------------------------------ end to end (host buffers)
    # Each step uploads its inputs (new tokens' q/k/v, rows, positions, chunk offsets) from pinned host
    # memory, runs the step through the C ABI and downloads its output, as a serving loop would: uploads,
    # kernels and downloads run on three streams with two input/output buffer sets, so step i+1's upload
    # and step i-1's download overlap step i's kernels. The KV caches stay resident (they are the layer's
    # state, shared by both buffer sets).
    e2e = None
    if with_e2e:
        names = ["q", "k", "v", "tok_rows", "tok_pos", "tok_seq_len", "q_start", "pf_rows", "pf_first_pos",
                 "dec_rows", "dec_pos"]
        sets = []
        for b in range(2):
            layer_steps = []
            for li, st in enumerate(steps):
                c = st.call
                if b == 0:
                    layer_steps.append(st)
                    continue
                fields = {k: getattr(c, k) for k in c.__dataclass_fields__}
                for n in names:
                    fields[n] = getattr(c, n).clone()
                layer_steps.append(make_step(type(c)(**fields), li))
            sets.append(layer_steps)
        host_in = [[[getattr(st.call, n).cpu().pin_memory() for n in names] for st in layer_steps]
                   for layer_steps in sets]
        host_out = [[torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for st in layer_steps]
                    for layer_steps in sets]
        h2d = sum(t.numel() * t.element_size() for hs in host_in[0] for t in hs)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):                      # the events start out "done"
            ev_cmp[b].record(s_cmp)
            ev_out[b].record(s_out)

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_cmp[b])          # buffer set b's previous step has read its inputs
                for st, hs in zip(sets[b], host_in[b]):
                    for n, h in zip(names, hs):
                        getattr(st.call, n).copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[b])
                s_cmp.wait_event(ev_out[b])         # its previous output has been downloaded
                for st in sets[b]:
                    st.run(s_cmp)
                ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                for st, ho in zip(sets[b], host_out[b]):
                    ho.copy_(st.out, non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 50))
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier(world)
        _abi.check_device_error()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e_ms = reduce_max(e2e_ms, world)
        v, u, _ = headline(work, e2e_ms / 1e3)
        e2e = {"value": v * world, "unit": u, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "steps": n_e2e,
               "via": "AttentionStep.run (C ABI) with pinned host inputs/outputs; upload, kernels and download "
                      "on three streams, two buffer sets, L2 not flushed (each step moves more than L2 holds)",
               "link_gbs": host_link_gbs(dev)}
        del sets, host_in, host_out

    rec = {
        "value": value_1 * world, "unit": unit, "ms_per_step": ms_all,
        "ms_per_step_mean": statistics.mean(step_ms), "timing": (f"median of {args.steps} timed steps (events around each step only); breakdown_ms and "
                   f"roofline from a second pass of {args.steps} steps with an event after every stage"),
        "dtype": "bf16" if wl.layers[0].dtype == torch.bfloat16 else "fp32",
        "config": {"workload": workload, "number": num, "scale": args.scale, "description": wl.description,
                   "l2": "flushed (256 MB write) before every timed step, outside the step's events",
                   "kv": (f"paged pool, {args.kv_block}-position blocks in shuffled order" if pools
                          else "contiguous caches"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": work["tokens"] * world / (ms_all / 1e3),
        "breakdown_ms": {"rope_and_cache_update": statistics.median(pre_ms), "prefill": statistics.median(pf_ms),
                         "decode": statistics.median(dec_ms),
                         "wall_ms_per_step_incl_flush": wall * 1e3 / args.steps},
        "work": {k: v for k, v in work.items() if v},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": sum(st.kernel_launches() for st in steps) * args.steps,
        "clocks": clock_info,
        "peaks": dict(peaks, kind=peak_kind),
    }
    if len(parts) > 1:
        rec["roofline_parts"] = parts
        # a mixed batch's two parts share the GPU within the step (da_attn_mixed): each part's work over the whole
        # step's time, as a fraction of its own peak; the sum is how much of the two roofs the step uses at once
        pf_t = work["prefill_flops"] / (ms_all / 1e3) / 1e12
        dec_g = work["decode_bytes"] / (ms_all / 1e3) / 1e9
        rec["parts_over_step"] = {
            "prefill_tflops": pf_t, "prefill_frac": pf_t / peaks["bf16_tflops"],
            "decode_gbs": dec_g, "decode_frac": dec_g / peaks["hbm_gbs"],
            "sum_of_fracs": pf_t / peaks["bf16_tflops"] + dec_g / peaks["hbm_gbs"],
            # SMs the library's split model gives each layer's prefill (the rest run the decode; all SMs: in turn)
            "prefill_sms_per_layer": None if pools else [
                _abi.attn_mixed_prefill_sms(st.L, torch.cuda.get_device_properties(dev).multi_processor_count,
                                            st.hint_pairs, st.hint_keys) for st in steps]}
    del steps, pools, wl, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


# The workloads the default invocation times beside the headline (each as a sub-record of the same line):
# the sliding-window decode, the long-context decode and the mixed prefill + decode layer pair.
SIDE_WORKLOADS = ("mistral_swa_decode", "llama31_8b_long_decode", "phi4_gemma2_mixed")


def cpu_baselines(workload, all_cores=True):
    """The oracle on the host cores: single-threaded on the bounded sample, and (all_cores) the same kind of
    sample spread over a process pool of every core. Reported, never fatal."""
    out = {}
    try:
        r = run_oracle_sample(workload, "baseline", 1)
        v, u, _ = headline(r["work"], r["seconds"][0])
        out = {"value": v, "unit": u, "cores": 1, "kind": "oracle", "sample": r["sample"],
               "seconds": r["seconds"][0], "host_cores": os.cpu_count(), "cpu_model": cpu_model()}
    except Exception as exc:
        return {"value": None, "unit": None, "cores": 1, "kind": "oracle", "error": str(exc)[-300:]}
    if all_cores:
        try:
            r = run_oracle_sample(workload, "allcores", 1)
            v, u, _ = headline(r["work"], r["seconds"][0])
            out["all_cores"] = {"value": v, "unit": u, "cores": r["cores"], "sample": r["sample"],
                                "seconds": r["seconds"][0]}
        except Exception as exc:
            out["all_cores"] = {"value": None, "error": str(exc)[-300:]}
    return out


def main_native(args):
    import torch

    rank, world, local = dist_init(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rec = measure_native(args, args.workload, dev, world, rank, with_e2e=not args.no_e2e)
    side = {}
    if args.workload == DEFAULT_WORKLOAD and not args.single and args.kv_block == 0 and args.scale == "full":
        for w in SIDE_WORKLOADS:
            side[w] = measure_native(args, w, dev, world, rank, with_e2e=not args.no_e2e)
        # the two steps beside the attention step proper: the absorbed MLA decode and the attention block with
        # its fused projections (their records keep their own keys; the MLA one carries its own CPU baseline)
        side[MLA_WORKLOAD] = measure_mla(args, dev, world, rank)
        side[BLOCK_WORKLOAD] = measure_block(args, dev, world, rank)
    cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if rank == 0:
        line = {
            "metric": METRIC, "value": rec["value"], "unit": rec["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": rec["dtype"], "data": "synthetic",
        }
        line.update({k: v for k, v in rec.items() if k not in line})
        line["cpu_baseline"] = cpu_baselines(args.workload) if cpu else None
        if side:
            for w, r in side.items():
                r.pop("peaks", None)
                for k in ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data"):
                    r.pop(k, None)
                if w in SIDE_WORKLOADS:
                    r["cpu_baseline"] = cpu_baselines(w, all_cores=False) if cpu else None
            line["workloads"] = side
            line["gpu_launches"] += sum(r["gpu_launches"] for r in side.values())
            line["gpu_launches_note"] = "headline workload plus the side workloads' timed steps"
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------------------------- MLA decode

MLA_WORKLOAD = "deepseek_v3_mla_decode"


def mla_work(call):
    """Latent rows read (one 1152-byte row per visible key) and tensor FLOPs of one MLA decode step."""
    pos = call.positions.cpu().tolist()
    keys = sum(min(p + 1, call.window) if call.window else p + 1 for p in pos)
    h = call.num_heads
    return {"decode_keys": keys, "decode_bytes": keys * 576 * 2, "decode_flops": keys * h * (576 + 512) * 2,
            "tokens": len(pos), "prefill_flops": 0}


def mla_oracle_sample(call, seqs):
    """The oracle on the listed sequences of an MLA call (each against its own cache row only)."""
    from decoder_attention_gb300 import inputs
    from oracle import mla as OM
    cpu = call.to("cpu") if call.q.is_cuda else call
    t0 = time.perf_counter()
    keys = 0
    for s in seqs:
        sub = inputs.MlaCall(**{k: getattr(cpu, k) for k in cpu.__dataclass_fields__})
        r, p = int(cpu.rows[s]), int(cpu.positions[s])
        sub.q, sub.latent, sub.k_rope = cpu.q[s:s + 1], cpu.latent[s:s + 1], cpu.k_rope[s:s + 1]
        sub.rows = cpu.rows.new_zeros(1)
        sub.positions, sub.seq_len = cpu.positions[s:s + 1], cpu.seq_len[s:s + 1]
        sub.cache = cpu.cache[r:r + 1, :p + 1]
        OM.run_mla_call(sub)
        keys += p + 1
    sec = time.perf_counter() - t0
    return keys * 576 * 2 / sec / 1e9, sec, f"{len(seqs)} of {call.n_seqs} sequences, all heads; single-threaded fp64 numpy"


def main_native_mla(args):
    import torch

    rank, world, local = dist_init(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rec = measure_mla(args, dev, world, rank)
    if rank == 0:
        print(json.dumps(rec))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_mla(args, dev, world, rank):
    """The DeepSeek-V3-shaped MLA decode step through the C ABI on `dev`; returns its record."""
    import torch

    from decoder_attention_gb300 import _abi, inputs, step as S

    call = inputs.deepseek_v3_mla_decode("full", device=dev)
    pool = None
    if args.kv_block > 0:
        kp, _, table = inputs.paged_from_contiguous(call.cache[:, None], call.cache[:, None], args.kv_block, seed=1006)
        pool = (kp, table)
    st = S.MlaDecodeStep(call, *(pool or ()), args.kv_block) if pool else S.MlaDecodeStep(call)
    work = mla_work(call)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    clocks.mark_start()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        st.run()
    torch.cuda.synchronize()
    _abi.check_device_error()
    # whole steps (events around each step only), then a second pass with an event between the two stages
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        sev[i][0].record(stream)
        st.run()
        sev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        st.update()
        ev[i][1].record(stream)
        st.decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    _abi.check_device_error()
    ms = reduce_max(statistics.median(a.elapsed_time(b) for a, b in sev), world)
    dec_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    clock_info = clocks.stop()
    value = work["decode_bytes"] / (ms / 1e3) / 1e9 * world
    peaks, peak_kind = load_peaks()
    achieved = work["decode_bytes"] / (dec_ms / 1e3) / 1e9
    kname = "mla_pair_kernel" if call.num_heads == 128 else "mla_decode_kernel"
    roof = {"kernel": f"{kname} + mla_merge_kernel (one da_mla_decode call)", "bound": "hbm",
            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "peak_kind": f"HBM copy, of {peak_kind}", "launch_ms": dec_ms,
            "algorithmic_bytes_per_launch": work["decode_bytes"],
            "tensor_tflops": work["decode_flops"] / (dec_ms / 1e3) / 1e12,
            "traffic": load_traffic(kname, MLA_WORKLOAD) if not args.kv_block else None}
    e2e = None
    if not args.no_e2e:
        names = ["q", "latent", "k_rope", "rows", "positions", "seq_len"]
        host_in = [getattr(call, n).cpu().pin_memory() for n in names]
        host_out = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = host_out.numel() * host_out.element_size()

        def e2e_step():
            for n, h in zip(names, host_in):
                getattr(call, n).copy_(h, non_blocking=True)
            st.run()
            host_out.copy_(st.out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(e0.elapsed_time(e1) / n_e2e, world)
        e2e = {"value": work["decode_bytes"] / (e2e_ms / 1e3) / 1e9 * world, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e,
               "via": "MlaDecodeStep.run (C ABI) with pinned host inputs/outputs, one stream, L2 not flushed"}
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sec, desc = mla_oracle_sample(call, [0, 1])
        cpu_base = {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc, "seconds": sec,
                    "host_cores": os.cpu_count()}
    rec = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "timing": (f"median of {args.steps} timed steps (events around each step only); breakdown_ms and "
                   f"roofline from a second pass of {args.steps} steps with an event between the stages"),
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": MLA_WORKLOAD, "description": call.meta["description"],
                   "l2": "flushed (256 MB write) before every timed step, outside the step's events",
                   "kv": (f"paged pool, {args.kv_block}-position blocks in shuffled order" if pool
                          else "contiguous latent rows"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": work["tokens"] * world / (ms / 1e3),
        "breakdown_ms": {"rope_and_cache_update": ms - dec_ms, "decode": dec_ms},
        "work": work, "roofline": roof, "e2e": e2e, "gpu_launches": st.kernel_launches() * args.steps,
        "clocks": clock_info, "cpu_baseline": cpu_base, "peaks": dict(peaks, kind=peak_kind)}
    del st, call, pool, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def main_reference_mla(args):
    rank, world, _ = dist_init(args)
    if rank != 0:
        return 0
    from decoder_attention_gb300 import inputs
    call = inputs.deepseek_v3_mla_decode("full", device="cpu")
    secs = []
    for _ in range(args.warmup + args.steps):
        v, sec, desc = mla_oracle_sample(call, [0])
        secs.append(sec)
    sec = statistics.median(secs[args.warmup:])
    keys = int(call.positions[0]) + 1
    value = keys * 576 * 2 / sec / 1e9
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": {"workload": MLA_WORKLOAD, "sample": desc},
                      "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
                      "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
    return 0


# ---------------------------------------------------------------------------------------------- attention block

BLOCK_WORKLOAD = "qwen3_8b_attn_block"


def main_native_block(args):
    """The Qwen3-8B-shaped attention block: the fused q/k/v projection (norm, RoPE and cache write in the GEMM
    epilogue), the prefill attention and o_proj, all through the C ABI; the unfused form (a cuBLAS GEMM for
    q/k/v, then da_kv_cache_update; cuBLAS for o_proj) is timed beside it for comparison."""
    import torch

    rank, world, local = dist_init(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rec = measure_block(args, dev, world, rank)
    if rank == 0:
        print(json.dumps(rec))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_block(args, dev, world, rank):
    """The attention-block record on `dev` (see main_native_block)."""
    import math

    import torch

    from decoder_attention_gb300 import _abi, inputs, step as S, work as W

    call = inputs.make(2, scale="full", device=dev).layers[0]          # 4 x 2048 tokens, Hq 32, Hkv 8
    n, hq, hkv, hidden = call.n_tokens, call.num_attention_heads, call.num_key_value_heads, 4096
    g = torch.Generator(device=dev).manual_seed(3002)
    x = torch.randn((n, hidden), generator=g, device=dev).to(torch.bfloat16)
    w_qkv = (torch.randn(((hq + 2 * hkv) * 128, hidden), generator=g, device=dev) / math.sqrt(hidden)).to(torch.bfloat16)
    w_o = (torch.randn((hidden, hq * 128), generator=g, device=dev) / math.sqrt(hq * 128)).to(torch.bfloat16)
    st = S.AttentionStep(call)
    y = torch.empty((n, hidden), dtype=torch.bfloat16, device=dev)
    qkv = torch.empty((n, (hq + 2 * hkv) * 128), dtype=torch.bfloat16, device=dev)
    proj_flops = 2 * n * (hq + 2 * hkv) * 128 * hidden
    o_flops = 2 * n * hidden * hq * 128
    attn_flops = W.layer_call_work(call)["prefill_flops"]

    def fused():
        st.rope()
        _abi.qkv_project_update(st.L, x, w_qkv, None, n, hidden, call.tok_rows, call.tok_pos, st.cos, st.sin,
                                st.q_rot, call.k_cache, call.v_cache, call.num_rows, call.max_len)

    def unfused():
        st.rope()
        torch.matmul(x, w_qkv.t(), out=qkv)
        q = qkv[:, :hq * 128].view(n, hq, 128)
        k = qkv[:, hq * 128:(hq + hkv) * 128].view(n, hkv, 128)
        v = qkv[:, (hq + hkv) * 128:].view(n, hkv, 128)
        _abi.kv_cache_update(st.L, q.contiguous(), k.contiguous(), v.contiguous(), n, call.tok_rows, call.tok_pos,
                             st.cos, st.sin, st.q_rot, call.k_cache, call.v_cache, call.num_rows, call.max_len)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    clocks.mark_start()

    def timed(fn_parts, steps):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fn_parts) + 1)] for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            for j, fn in enumerate(fn_parts):
                fn()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize()
        return [statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(len(fn_parts))]

    def timed_whole(fn_parts, steps):   # events around each step only (kernels may overlap launches)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            for fn in fn_parts:
                fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    parts = [fused, st.prefill, lambda: _abi.linear(st.out.view(n, hq * 128), w_o, None, n, hidden, hq * 128, y)]
    timed(parts, max(args.warmup, 3))
    _abi.check_device_error()
    barrier(world)
    ms_whole = timed_whole(parts, args.steps)
    barrier(world)
    ms_parts = timed(parts, args.steps)
    clocks.mark_end()
    _abi.check_device_error()
    cmp_parts = [unfused, st.prefill, lambda: torch.matmul(st.out.view(n, hq * 128), w_o.t(), out=y)]
    timed(cmp_parts, 3)
    ms_cmp = timed(cmp_parts, max(3, min(args.steps, 20)))
    clock_info = clocks.stop()
    ms = reduce_max(ms_whole, world)
    total = proj_flops + attn_flops + o_flops
    peaks, peak_kind = load_peaks()
    achieved = proj_flops / (ms_parts[0] / 1e3) / 1e12
    rec = {
            "metric": METRIC, "value": total / (ms / 1e3) / 1e12 * world, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "timing": (f"median of {args.steps} timed blocks (events around each block only); breakdown_ms and "
                       f"roofline from a second pass of {args.steps} blocks with an event after every part"),
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init projection weights)",
            "config": {"workload": BLOCK_WORKLOAD, "description": "Qwen3-8B-shaped attention block: 4 x 2048 tokens, "
                       "hidden 4096, fused q/k/v projection + norm + RoPE + cache write, prefill attention, o_proj",
                       "l2": "flushed (256 MB write) before every timed step, outside the step's events",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "breakdown_ms": {"rope_tables_and_fused_qkv_projection": ms_parts[0], "prefill": ms_parts[1],
                             "o_proj": ms_parts[2]},
            "work": {"qkv_projection_flops": proj_flops, "attention_flops": attn_flops, "o_proj_flops": o_flops},
            "roofline": {"kernel": "gemm_kernel<EPI_QKV> (one da_qkv_project_update call)", "bound": "tensor",
                         "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "peak_kind": f"bf16 dense burst, of {peak_kind}",
                         "launch_ms": ms_parts[0], "traffic": load_traffic("gemm_kernel", BLOCK_WORKLOAD)},
            "unfused_comparison_ms": {"rope_tables_cublas_qkv_and_cache_update": ms_cmp[0], "prefill": ms_cmp[1],
                                      "cublas_o_proj": ms_cmp[2]},
            "e2e": None, "gpu_launches": 5 * args.steps, "clocks": clock_info, "cpu_baseline": None,
            "peaks": dict(peaks, kind=peak_kind)}
    del st, call, x, w_qkv, w_o, y, qkv, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_sample:
        oracle_sample_child(args.workload, args.sample_kind, args.steps)
        return 0
    if args.workload == BLOCK_WORKLOAD:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the attention-block workload has no oracle arm"}))
            return 0
        return main_native_block(args)
    if args.workload == MLA_WORKLOAD:
        return main_reference_mla(args) if args.impl == "reference" else main_native_mla(args)
    if args.impl == "reference":
        return main_reference(args)
    return main_native(args)


if __name__ == "__main__":
    sys.exit(main())
