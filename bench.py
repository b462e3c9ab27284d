"""Benchmark: batch-1 greedy decode of a Llama-style decoder on GB300.

One "step" is one decode step (one token) of the whole model: embedding, every
layer, LM head and argmax, run by the persistent megakernel through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1b]
                  [--backend megakernel|chain] [--impl ours|reference]

Default workload: Llama-3.2-1B shape, bf16 weights bf16(0.02*N(0,1)) from seed
0, a 1024-token random prompt (seed 1) prefilled through the model in one
ll_prefill call (tcgen05 GEMMs; timed on its own as ``prefill``), then K greedy
decode steps timed with CUDA events on the decode stream: one ll_decode_steps
launch in which each step takes the token the previous one chose (no host
round trip). ``single_step_launches`` times the same K positions again as K
chained single-step launches. The weights (2.47 GB) are far larger than L2 (129
MB), so every step streams them from HBM. ``e2e`` repeats K steps through
ll_decode_step with the token passed from the host and the next token read
back to host memory every step, timed by the host clock. ``batch`` times
batched handles (ll_decode_steps_batch) of 2, 4 and 8 sequences on seeded
N(0,1) caches at the same context: tokens/s of all sequences together.

``--impl reference`` times the CPU oracle (the only reference implementation
there is) on the host cores on the same workload. Under torchrun every rank
decodes its own sequence (replicas; batch-1 decode has nothing to shard).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/token & tokens/s, batch-1 Llama-3.2-1B-shape decode; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SPEC_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--workload", default="1b")
    ap.add_argument("--backend", default="megakernel", choices=["megakernel", "chain"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-batch", action="store_true", help="skip the batched-decode lines")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# bf16 terms of the activation operand per prefill GEMM (its tensor-pipe work is
# that many products of the matrix)
PREFILL_TERMS = {"wq": 3, "wk": 3, "wv": 3, "wo": 2, "wg": 2, "wu": 2, "wd": 2}


def prefill_tensor_flops(shape, n):
    """Flops the tensor pipe does in a prefill of n positions: 2 n per weight
    element and activation term, over every layer's projections."""
    per_layer = sum(PREFILL_TERMS[k] * v[0] * v[1] for k, v in shape.layer_shapes().items() if k in PREFILL_TERMS)
    return 2.0 * n * shape.n_layers * per_layer


def bf16_peak():
    """Measured dense bf16 GEMM rate (TFLOP/s, burst), else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank space (no string literal
    of these sources contains a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


# Sources that do not go into a backend's decode kernels (so changing them leaves
# that backend's recorded counters valid).
NOT_IN_BACKEND = {
    "megakernel": {"chain.cu", "prefill.cu", "static_step.cu"},
    "chain": {"megakernel.cuh", "mk_cuda_cores.cu", "mk_tensor_cores.cu", "mk_geo.cu", "prefill.cu", "static_step.cu"},
}


def kernel_sha(backend: str = "megakernel") -> str:
    """Hash of the code a backend's decode step is built from (comments and
    layout excluded), which ties recorded ncu counters to the code they were
    taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_megakernel_persistent_gb300", "csrc")
    skip = NOT_IN_BACKEND.get(backend, set())
    for name in sorted(os.listdir(csrc)):
        if name in skip:
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str, backend: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{backend}:{workload_name}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_sha") != kernel_sha(backend):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept with host timestamps."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.out = tempfile.NamedTemporaryFile(prefix="clocks", suffix=".csv", delete=False)
        self.t0 = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.marks = []

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()

    @staticmethod
    def _stamp(text: str):
        try:
            base, _, frac = text.partition(".")
            return time.mktime(time.strptime(base, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
        except ValueError:
            return None

    def summary(self):
        """Median SM clock and throttle reasons over samples taken between the
        first and the last mark (the timed regions)."""
        rows = []
        lo, hi = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0.0, float("inf"))
        try:
            with open(self.out.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    t = self._stamp(parts[0])
                    if t is not None and lo - 0.02 <= t <= hi + 0.02:
                        rows.append(parts)
        finally:
            os.unlink(self.out.name)
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------
# CPU oracle timing (rank 0 only): the cpu_baseline leg and the reference arm.

def oracle_timing(shape, ctx: int, budget_s: float, max_steps: int | None = None, weights_host=None):
    """Time oracle decode steps at positions ctx, ctx+1, ... on a seeded N(0,1) KV
    cache (a step's cost depends on its position, not on the cached values)."""
    import numpy as np

    import oracle
    from decode_megakernel_persistent_gb300 import synth
    if weights_host is None:
        weights_host = synth.weights_to_host_bits(synth.make_weights(shape, seed=0, device="cpu"))
    steps_cap = max_steps if max_steps is not None else 1 << 30
    max_seq = ctx + min(steps_cap, 4096) + 1
    orc = oracle.OracleModel(shape.as_dict(), weights_host, max_seq, prec=32)
    rng = np.random.default_rng(2)
    fill = (rng.standard_normal((shape.n_layers, shape.n_kv_heads, ctx, shape.head_dim)) * 1.0)
    bits = (fill.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    orc.k_cache[:, :, :ctx] = bits
    orc.v_cache[:, :, :ctx] = bits[:, :, ::-1]
    toks = synth.make_tokens(shape.vocab, 4096, seed=1)
    n, t_total = 0, 0.0
    while n < steps_cap and n < 4096 and (max_steps is not None or t_total < budget_s):
        t0 = time.perf_counter()
        orc.decode_step(toks[n], ctx + n)
        t_total += time.perf_counter() - t0
        n += 1
    return n, t_total, oracle.num_threads()


def bench_config(wl, steps: int, warmup: int, world: int) -> dict:
    """The workload both arms report under "config", key for key: the model and
    context, the K timed greedy steps and their positions (after W warm-up steps),
    the weight format and how ranks split the work."""
    pos0 = wl.context + warmup
    return {"workload": wl.name, "context": wl.context, "decode_steps_timed": steps,
            "positions": [pos0, pos0 + steps - 1], "weights": "bf16",
            "parallelism": f"replicas{world}" if world > 1 else "single"}


def run_reference(args):
    from decode_megakernel_persistent_gb300 import synth
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    import oracle
    oracle.build()
    from decode_megakernel_persistent_gb300 import synth as s2
    wh = s2.weights_to_host_bits(s2.make_weights(wl.shape, seed=0, device="cpu"))
    oracle_timing(wl.shape, wl.context, 0.0, max_steps=max(1, args.warmup), weights_host=wh)
    n, secs, cores = oracle_timing(wl.shape, wl.context + args.warmup, 0.0, max_steps=args.steps,
                                   weights_host=wh)
    tps = n / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": world, "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * secs / n,
        "us_per_token": 1e6 * secs / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(wl, n, args.warmup, world),
        "method": {"timed": "CPU oracle decode steps (fp32, OpenMP over rows) on a seeded KV cache"},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} full oracle decode steps at positions {wl.context + args.warmup}.."},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------

def batch_lines(shape, w, ctx, dev, K, peak):
    """Decode throughput of batched handles (2, 4, 8 sequences) at context ctx on
    seeded N(0,1) caches: one ll_decode_steps_batch launch of K steps, timed with
    CUDA events after a warm-up launch; achieved GB/s from the algorithmic bytes
    of the K steps (weights once per step, each sequence's K/V)."""
    import torch

    from decode_megakernel_persistent_gb300 import bytemodel, ll, synth
    out = {}
    for n in (2, 4, 8):
        max_seq = ctx + K + 8
        kv = [synth.make_kv(shape, max_seq, ctx, seed=2 + b, device=dev) for b in range(n)]
        dec = ll.BatchDecoder(shape, w, [x[0] for x in kv], [x[1] for x in kv], max_seq)
        toks = torch.zeros((K, n), dtype=torch.int32, device=dev)
        first = torch.tensor(synth.make_tokens(shape.vocab, n, seed=3), dtype=torch.int32, device=dev)
        dec.steps_batch(first, [ctx] * n, 4, None, toks[:4])
        dec.synchronize()
        s = torch.cuda.current_stream(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        dec.steps_batch(first, [ctx + 4] * n, K, None, toks)
        e1.record(s)
        torch.cuda.synchronize(dev)
        dec.synchronize()
        secs = e0.elapsed_time(e1) / 1e3
        nbytes = sum(bytemodel.batch_step_bytes(shape, ctx + 4 + i, n) for i in range(K))
        out[str(n)] = {"tokens_per_s": n * K / secs, "us_per_step": 1e6 * secs / K,
                       "achieved_gbs": nbytes / secs / 1e9, "frac": nbytes / secs / 1e9 / peak,
                       "kv_splits": dec.query(ll.LL_Q_ATTN_SPLITS)}
        dec.close()
        del kv
    return out


def run_ours(args):
    import torch

    from decode_megakernel_persistent_gb300 import build, bytemodel, ll, synth
    world, rank, local = dist_setup(args)
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    shape, ctx = wl.shape, wl.context
    K, W = args.steps, args.warmup
    if W < 3:
        raise SystemExit("--warmup must be at least 3")
    max_seq = ctx + W + 2 * K + 1
    backend = ll.LL_BACKEND_MEGAKERNEL if args.backend == "megakernel" else ll.LL_BACKEND_CHAIN

    w = synth.make_weights(shape, seed=0 + rank * 1000, device=dev)
    fill = ctx if wl.kv_fill == "normal" else 0
    k_cache, v_cache = synth.make_kv(shape, max_seq, fill, seed=2, device=dev)
    stream = torch.cuda.Stream(device=dev)
    dec = ll.Decoder(shape, w, k_cache, v_cache, max_seq, backend, stream=stream)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    prompt = synth.make_tokens(shape.vocab, max(ctx, 1), seed=1 + rank)
    prefill = None
    with torch.cuda.stream(stream):
        if wl.kv_fill == "prefill":
            prompt_dev = torch.tensor(prompt, dtype=torch.int32, device=dev)
            if backend == ll.LL_BACKEND_MEGAKERNEL:
                # the prompt in one pass (tcgen05 GEMMs); once untimed (the first
                # call makes its buffers), then timed
                dec.prefill(prompt_dev, 0, logits, tok)
                dec.synchronize()
                p0 = torch.cuda.Event(enable_timing=True)
                p1 = torch.cuda.Event(enable_timing=True)
                p0.record(stream)
                dec.prefill(prompt_dev, 0, logits, tok)
                p1.record(stream)
                torch.cuda.synchronize(dev)
                secs = p0.elapsed_time(p1) / 1e3
                flops = 2.0 * ctx * bytemodel.layer_weight_elements(shape)
                tflops = prefill_tensor_flops(shape, ctx)
                tpeak, tpeak_kind = bf16_peak()
                prefill = {"tokens": ctx, "ms": 1e3 * secs, "tokens_per_s": ctx / secs,
                           "tflops_algorithmic": flops / secs / 1e12,
                           "tflops_tensor": tflops / secs / 1e12,
                           "tensor_peak": tpeak, "tensor_peak_kind": tpeak_kind,
                           "tensor_frac": tflops / secs / 1e12 / tpeak,
                           "call": "ll_prefill: every projection a tcgen05 GEMM, activations as bf16 terms "
                                   "(3 for Q/K/V, 2 for O, gate/up, down)"}
            else:
                for pos in range(ctx):
                    dec.step_async(prompt_dev[pos:pos + 1], pos, logits, tok)
        else:
            tok.fill_(prompt[0])
        dec.synchronize()
        pos = ctx
        for _ in range(W):
            dec.step_async(tok, pos, logits, tok)
            pos += 1
        dec.synchronize()

        clocks = ClockSampler(local) if rank == 0 else None
        if clocks:
            time.sleep(1.0)  # let nvidia-smi start sampling
        barrier(world)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        pos0 = pos
        if clocks:
            clocks.mark()
        # timed: K greedy steps in one launch of the persistent kernel (each step
        # fed the previous one's token on the device), logits of every step kept
        logits_k = torch.empty((K, shape.vocab), dtype=torch.float32, device=dev)
        toks_k = torch.zeros(K, dtype=torch.int32, device=dev)
        e0.record(stream)
        dec.steps(tok, pos0, K, logits_k, toks_k)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        dec.synchronize()
        dev_ms = e0.elapsed_time(e1)
        t_dev = max_over_ranks(dev_ms / 1e3, world, dev)
        # the same K positions again as K single-step launches chained on the
        # device (the cache rows they rewrite are read back the same way)
        tok.copy_(toks_k[:1])
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for i in range(K):
            dec.step_async(tok, pos0 + i, logits, tok)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        dec.synchronize()
        t_single = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        tok.copy_(toks_k[-1:])
        pos = pos0 + K

        # end to end through the C ABI with host buffers
        host_tok = int(tok.item())
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(K):
            host_tok = dec.step(host_tok, pos, logits)
            pos += 1
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        if clocks:
            clocks.mark()
        barrier(world)
        if clocks:
            clocks.stop()
    # kernels launched in the timed region: one persistent launch (the chain
    # backend runs its per-operation kernels for every step)
    launches = 1 if backend == ll.LL_BACKEND_MEGAKERNEL else dec.query(ll.LL_Q_LAUNCHES_PER_STEP) * K

    if rank != 0:
        dec.close()
        return

    bytes_per_step = statistics.mean(bytemodel.step_bytes(shape, p) for p in range(pos0, pos0 + K))
    achieved = bytes_per_step * K / t_dev / 1e9  # the launch's algorithmic bytes over its duration
    traffic_step = recorded_traffic(wl.name, args.backend)
    peak, peak_kind = peaks()
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        wh = synth.weights_to_host_bits(w)
        n, secs, cores = oracle_timing(shape, ctx, args.cpu_seconds, weights_host=wh)
        cpu = {"value": n / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} full oracle decode steps (fp32, OpenMP over rows) at positions "
                         f"{ctx}..{ctx + n - 1} on a seeded KV cache, {secs:.1f} s"}
        # the same on one thread, a smaller sample
        import oracle
        oracle.set_threads(1)
        n1, secs1, _ = oracle_timing(shape, ctx, args.cpu_seconds / 2, weights_host=wh)
        oracle.set_threads(cores)
        cpu["single_thread"] = {"value": n1 / secs1, "unit": "tokens/s", "cores": 1,
                                "sample": f"{n1} full oracle decode steps on one thread at positions "
                                          f"{ctx}..{ctx + n1 - 1}, {secs1:.1f} s"}
    batch = None
    if not args.no_batch and backend == ll.LL_BACKEND_MEGAKERNEL and shape.hidden % 1024 == 0:
        batch = batch_lines(shape, w, ctx, dev, K, peak)
    line = {
        "metric": METRIC,
        "value": world * K / t_dev,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": 1e3 * t_dev / K,
        "us_per_token": 1e6 * t_dev / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": bench_config(wl, K, W, world),
        "method": {"backend": args.backend,
                   "l2": "inputs larger than L2: every step streams all weights from HBM",
                   "timed": "one ll_decode_steps launch of K greedy steps" if backend == ll.LL_BACKEND_MEGAKERNEL
                   else "ll_decode_steps: K steps of per-operation launches"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_8000": achieved / SPEC_HBM_GBS,
                     "bytes_per_launch": bytes_per_step * K, "bytes_per_step": bytes_per_step,
                     # ncu DRAM bytes of a single-step launch (same kernel sources) times the K steps
                     "traffic": traffic_step * K if traffic_step else None},
        "single_step_launches": {"us_per_token": 1e6 * t_single / K, "value": world * K / t_single,
                                 "unit": "tokens/s", "launches": K},
        "e2e": {"value": world * K / t_e2e, "unit": "tokens/s", "us_per_token": 1e6 * t_e2e / K,
                "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 8},
        "gpu_launches": launches,
        "prefill": prefill,
        "batch": batch,
        "cpu_baseline": cpu,
        "clocks": clocks.summary() if clocks else None,
    }
    dec.close()
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
