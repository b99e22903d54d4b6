"""Benchmark of the Qwen2 decoder forward on GB300 (one JSON line on stdout).

Headline workload: Qwen2.5-0.5B-shaped model (24 layers, hidden 896, 14/2
heads, vocab 151936, tied head), seeded synthetic f16 weights, batch 1: a
128-token prompt is prefilled once (untimed), then each timed step is one
greedy generation of 256 tokens at positions 128..383 through
qwen2_decode_steps (one persistent launch per token, ids fed back on the
device).  The default run also measures the other workloads the metric
names and reports them under "workloads": long-context batch-1 decode
(positions 4000..4095), the 8 x 512 tensor-core prefill, and batched decode
of 32 ragged sequences on Q8_0 weights.  Every workload's weights (988 MB
f16, 525 MB Q8_0) exceed the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME]

Under torchrun (N > 1) every rank runs an independent replica (the forward
has no exchange step); value = tokens of all ranks / max rank time.
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tokens/s (batch 1 and 32) and prefill tok/s; % of HBM/tensor roofline"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc, self.lines = gpu, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class Replicas:
    """Coordination of N independent replicas, one process per GPU (the
    forward has no exchange step, so the only collectives are the timing
    barrier and the max over ranks).  backend "nccl" with a CUDA device on
    the GPU box; "gloo" with device None runs the same logic on the CPU."""

    def __init__(self, world: int, backend: str = "nccl", device=None):
        self.world, self.device, self.dist = world, device, None
        if world > 1:
            import torch.distributed as dist
            kw = {"device_id": device} if backend == "nccl" else {}
            dist.init_process_group(backend, **kw)
            self.dist = dist

    def barrier(self):
        import torch
        if self.dist:
            self.dist.barrier()
        if self.device is not None:
            torch.cuda.synchronize()

    def max(self, x: float) -> float:
        """The largest of every rank's x (the slowest replica's time)."""
        if not self.dist:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()
            self.dist = None


def decode_bytes_per_step(shape, positions, q8: bool = False) -> float:
    """Algorithmic HBM bytes of one decode step of B sequences at positions
    p_b: the weights once (f16: 2 bytes an element; Q8_0: 1 byte plus a
    2-byte scale per 32) + f32 biases and norms + B embedding rows + per
    sequence the KV read of positions 0..p_b and the KV write of p_b."""
    H, I, V, L = shape.hidden, shape.intermediate, shape.vocab, shape.n_layer
    nq, nkv = shape.n_head * shape.head_dim, shape.n_kv_head * shape.head_dim
    per_elem = 1 + 2 / 32 if q8 else 2
    elems = V * H + L * ((nq + 2 * nkv) * H + H * nq + 2 * I * H + H * I)
    small = 4 * (L * (nq + 2 * nkv + 2 * H) + H)
    p = np.asarray(positions, dtype=np.float64)
    kv_pos = L * 2 * nkv * 4
    return float(elems * per_elem + small + len(p) * H * per_elem + kv_pos * np.sum(p + 2))


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum of
# the 21st launch, a position near 150 of the 0.5b-decode-b1 workload) from
# an ncu capture of those two counters on the persistent decode kernel
# (profiles/decode_persistent_0p5b_b1_launches.md), valid only
# for that workload and only while the kernel's sources -- their code, with
# // comments and blank lines left out -- hash to `src`.
TRAFFIC = {"k_decode_persistent": {"workload": "0.5b-decode-b1", "src": "45812fb3f0393c9d", "bytes": 1003649792.0}}
KERNEL_SOURCES = ("persistent.cu", "persistent.h", "rowdot.cuh", "common.cuh", "attn.cuh", "ctx.h", "sm100.cuh")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "qwen2_decoder_forward_gb300", "csrc", f), "rb") as fh:
            text = fh.read().decode("utf-8", errors="replace")  # the same on any locale
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def kernel_traffic(name: str, workload: str):
    rec = TRAFFIC.get(name)
    if rec is None or rec.get("workload") != workload:
        return None
    return rec["bytes"] if kernel_source_hash() == rec["src"] else None


def prefill_flops(shape, lens, n_keep: int) -> float:
    """Algorithmic FLOPs of one prefill with the tail cut: every row through
    the first L-1 layers and the last layer's Q/K/V product; causal GQA
    attention of every row in the first L-1 layers and of the kept rows in
    the last; o_proj and the FFN of the kept rows in the last layer; the LM
    head on the kept rows (2 flops per multiply-add)."""
    H, I, V, L = shape.hidden, shape.intermediate, shape.vocab, shape.n_layer
    nq, nkv = shape.n_head * shape.head_dim, shape.n_kv_head * shape.head_dim
    qkv = 2 * (nq + 2 * nkv) * H
    rest = 2 * (H * nq + 2 * I * H + H * I)
    lens = [int(n) for n in lens]
    rows = sum(lens)
    per_key = 4 * shape.n_head * shape.head_dim          # q.k and p.v, all heads
    att_all = sum(n * (n + 1) // 2 for n in lens) * per_key
    kept_keys = sum(sum(n - k for k in range(n_keep)) for n in lens)
    att_kept = kept_keys * per_key
    return float((L - 1) * rows * (qkv + rest) + rows * qkv + len(lens) * n_keep * rest
                 + (L - 1) * att_all + att_kept + 2 * len(lens) * n_keep * V * H)


@contextlib.contextmanager
def blas_threads(n: int):
    """Limit the BLAS pool the oracle's numpy calls use to ``n`` threads
    inside the block (threadpoolctl when present, else numpy's bundled
    OpenBLAS through its own thread-count entry points)."""
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    if threadpool_limits is not None:
        with threadpool_limits(limits=n, user_api="blas"):
            yield
        return
    import ctypes
    lib, getter, setter = None, None, None
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ln.split()[-1].startswith("/")})
        for path in paths:
            cand = ctypes.CDLL(path)
            for suffix in ("64_", ""):
                for pre in ("scipy_openblas_", "openblas_"):
                    if hasattr(cand, f"{pre}set_num_threads{suffix}"):
                        lib = cand
                        setter = getattr(cand, f"{pre}set_num_threads{suffix}")
                        getter = getattr(cand, f"{pre}get_num_threads{suffix}")
                        break
                if lib:
                    break
            if lib:
                break
    except Exception:
        lib = None
    if lib is None:
        yield
        return
    old = int(getter())
    setter(int(n))
    try:
        yield
    finally:
        setter(old)


def cpu_threads() -> int:
    """Threads of the BLAS pool the oracle's products run on."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


class OracleTimer:
    """Bounded samples of a workload run by the oracle on the host cores.

    Decode samples are single-token forwards at the workload's positions
    over a key/value cache filled with seeded random values up to that
    position: the oracle's work per token (every weight once, attention
    over positions 0..p) is the same as after a real prefill, without the
    prefill itself (a 4000-token float64 prefill alone takes minutes)."""

    def __init__(self, shape, weights):
        self.shape, self.weights, self._orc = shape, weights, {}

    def oracle(self, weight_format: str):
        if weight_format not in self._orc:
            import oracle
            self._orc[weight_format] = oracle.build_oracle(self.shape, self.weights, 4096,
                                                           weight_format=weight_format)
        return self._orc[weight_format]

    def decode(self, wl, budget_s: float, max_tokens: int):
        """(tokens/s, tokens, seconds, what) of greedy decode tokens at the
        workload's positions, round-robin over its sequences."""
        orc = self.oracle(wl.weight_format)
        lens = [int(n) for n in wl.prompt_lengths()]
        rng = np.random.Generator(np.random.PCG64(77))
        cache = orc.new_cache()
        filled = 0
        tok = 17
        t_total, done = 0.0, 0
        while done < max_tokens and (done == 0 or t_total < budget_s):
            s = done % len(lens)
            pos = lens[s] + (done // len(lens)) % max(1, wl.decode_steps)
            if pos > filled:
                cache.K[:, filled:pos] = 0.1 * rng.standard_normal(cache.K[:, filled:pos].shape)
                cache.V[:, filled:pos] = 0.1 * rng.standard_normal(cache.V[:, filled:pos].shape)
                filled = pos
            t0 = time.perf_counter()
            r = orc.forward(cache, [tok], [pos])
            t_total += time.perf_counter() - t0
            tok = int(r["ids"][0])
            done += 1
        what = (f"{done} greedy decode tokens at the workload's positions "
                f"({'sequences round-robin, ' if len(lens) > 1 else ''}first at {lens[0]}; "
                f"cache filled with seeded random keys/values up to each position), "
                f"{wl.weight_format} weights")
        return done / t_total, done, t_total, what

    def prefill(self, wl, budget_s: float, n_rows: int):
        """(tokens/s, tokens, seconds, what) of prefills of the first
        ``n_rows`` tokens of the workload's first sequence."""
        orc = self.oracle(wl.weight_format)
        prompt = wl.prompts(self.shape.vocab)[0][:n_rows]
        t_total, done = 0.0, 0
        while done == 0 or t_total < budget_s / 3:
            t0 = time.perf_counter()
            orc.prefill(orc.new_cache(), prompt)
            t_total += time.perf_counter() - t0
            done += len(prompt)
            if t_total > budget_s:
                break
        what = f"{done // len(prompt)} causal prefill(s) of one {len(prompt)}-token sequence (tail cut)"
        return done / t_total, done, t_total, what

    def baseline(self, wl, budget_s: float = 8.0):
        """The cpu_baseline record: the oracle on every core of the BLAS pool,
        and on one thread."""
        cores = cpu_threads()
        if wl.decode_steps == 0:
            rate, _, _, what = self.prefill(wl, budget_s, wl.prompt_len)
            with blas_threads(1):
                r1, _, _, what1 = self.prefill(wl, budget_s, min(wl.prompt_len, 64))
        else:
            rate, _, _, what = self.decode(wl, budget_s, 256)
            with blas_threads(1):
                r1, _, _, what1 = self.decode(wl, budget_s, 64)
        return {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": what,
                "single_thread": {"value": r1, "unit": "tokens/s", "cores": 1, "sample": what1}}


def workload_config(wl, shape, world: int) -> dict:
    lens = [int(n) for n in wl.prompt_lengths()]
    if wl.decode_steps == 0:
        return {"workload": f"{wl.name}: {shape.name} shape, {wl.n_seq} sequences x {wl.prompt_len} tokens, "
                            f"causal prefill with the tail cut (last row of each sequence to the LM head), "
                            f"{'tensor-core f16 operands' if wl.prefill == 'tensor' else 'f32 CUDA cores'}, "
                            f"f32 accumulation and KV, n_ctx {wl.n_ctx}",
                "global_batch": wl.n_seq * world, "seq_len": wl.prompt_len, "parallelism": f"replicas x{world}",
                "l2": "weights (988 MB) exceed L2 (129 MB): no flush between steps"}
    q8 = wl.weight_format == "q8_0"
    ragged = len(set(lens)) > 1
    return {"workload": f"{wl.name}: {shape.name} shape, batch {wl.n_seq}, "
                        + (f"ragged prompts U{{{wl.ragged_lo}..{wl.ragged_hi}}} (mean {np.mean(lens):.0f})"
                           if ragged else f"prompt {lens[0]}")
                        + f", {wl.decode_steps} greedy decode steps per timed step, "
                        + ("Q8_0" if q8 else "f16") + f" weights, f32 KV, n_ctx {wl.n_ctx}",
            "global_batch": wl.n_seq * world, "seq_len": int(max(lens)) + wl.decode_steps,
            "parallelism": f"replicas x{world}",
            "l2": "weights (" + ("525" if q8 else "988") + " MB) and KV exceed L2 (129 MB): no flush between steps"}


def reference_line(args, wl, shape, weights, world: int) -> dict:
    """The reference arm: the oracle as it stands on the host cores, K timed
    steps after W warm-up steps, each step a bounded sample of the workload
    (at most 32 decode tokens, or one prefill of at most 128 tokens)."""
    timer = OracleTimer(shape, weights)
    if wl.decode_steps == 0:
        n_rows = min(wl.prompt_len, 128)
        sample = lambda: timer.prefill(wl, 0.0, n_rows)  # noqa: E731  (one prefill per step)
    else:
        n_tok = min(wl.decode_steps * wl.n_seq, 32)
        sample = lambda: timer.decode(wl, 1e9, n_tok)  # noqa: E731
    for _ in range(max(0, args.warmup)):
        sample()
    secs, toks, what = 0.0, 0, ""
    for _ in range(max(1, args.steps)):
        _, done, dt, what = sample()
        secs += dt
        toks += done
    rate = toks / secs
    return {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            # the measured time of one reference step (one bounded sample)
            "ms_per_step": secs / max(1, args.steps) * 1e3, "tokens_per_step": toks // max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random weights)", "config": workload_config(wl, shape, world),
            "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"each step: {what}"},
            "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_prefill(args, wl, shape, weights, reps, world):
    """Prefill workloads: a step is one qwen2_prefill of all the workload's
    sequences through the tail cut (one kept row per sequence, greedy ids
    out).  Tokens are host arrays (the C ABI copies them, 4 bytes a token)."""
    import torch
    import qwen2_decoder_forward_gb300 as q2
    prompts = wl.prompts(shape.vocab)
    lens = [len(p) for p in prompts]
    n_tok = sum(lens)
    flops = prefill_flops(shape, lens, 1)
    mode = q2.PREFILL_TENSOR if wl.prefill == "tensor" else q2.PREFILL_F32
    model = q2.Qwen2Model(shape, weights, n_ctx=wl.n_ctx, max_seqs=wl.n_seq, max_tokens=n_tok,
                          prefill_mode=mode, flags=args.flags)
    seqs = list(range(wl.n_seq))
    ids = torch.empty((wl.n_seq,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(out):
        model.prefill(seqs, prompts, n_out=1, want_logits=False, ids_out=out)

    for _ in range(max(3, args.warmup)):
        step(ids)
    model.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps.barrier()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            step(ids)
        end.record(stream)
        torch.cuda.synchronize()
    reps.barrier()
    ms = reps.max(start.elapsed_time(end))
    model.synchronize()
    value = args.steps * n_tok * world / (ms / 1e3)
    # End to end: host token arrays in, ids read back into host memory.
    host_ids = np.empty((wl.n_seq,), dtype=np.int32)
    reps.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(host_ids)
    e2e_s = reps.max(time.perf_counter() - t0)
    hbm, tflops, src = peaks()
    achieved = flops / (ms / 1e3 / args.steps) / 1e12
    tensor = bool(model.features & q2.FEATURE_TENSOR_PREFILL)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "traffic": None,
                "kernel": "one whole prefill (all kernels; tcgen05 GEMMs dominate)" if tensor else
                          "one whole prefill (f32 CUDA-core kernels)",
                "peak_source": src + " bf16 dense burst (f16 has the same tensor rate)",
                "flops_per_launch": flops}
    # Launches per step: embed; per layer norm, QKV, attention, O, norm, GU,
    # down (the last layer: norm, QKV, 4 gathers, attention, 3 GEMVs); LM
    # head.  (The tensor path's attention-operand conversion runs only for
    # keys an earlier call stored: none here.)
    launches = 1 + (shape.n_layer - 1) * 7 + 2 + 4 + 1 + 3 + 1
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16 tensor-core operands (activations of Q/K/V, o_proj and gate/up as f16 hi/lo pairs, "
                     "down's as f16; attention q, k, p in f16 and v as an f16 hi/lo pair; the kept rows' LM "
                     "head as f16 hi/lo rows against the f16 embedding), f32 accumulation, f32 "
                     "residual/softmax/KV" if tensor else "f32",
            "data": "synthetic (seeded random weights of the Qwen2.5-0.5B shape, uniform-random tokens)",
            "config": workload_config(wl, shape, world), "clocks": clocks.summary(),
            "e2e": {"value": args.steps * n_tok * world / e2e_s, "unit": "tokens/s",
                    # token, position and slot per row, kept-row indices, and
                    # the (first row, row count) plan of the 16-row blocks
                    "h2d_bytes_per_step": int(12 * n_tok + 4 * wl.n_seq
                                              + 8 * (sum((n + 15) // 16 for n in lens) + wl.n_seq)),
                    "d2h_bytes_per_step": int(host_ids.nbytes)},
            "roofline": roofline, "gpu_launches": launches * args.steps}
    model.close()
    return line


def run_decode(args, wl, shape, weights, reps, world):
    """Decode workloads: the prompts are prefilled once (untimed); a step is
    one qwen2_decode_steps call of decode_steps greedy tokens for every
    sequence (one CUDA-graph replay, or one persistent launch, per token;
    ids fed back on the device)."""
    import torch
    import qwen2_decoder_forward_gb300 as q2
    prompts = wl.prompts(shape.vocab)
    lens = [len(p) for p in prompts]
    q8 = wl.weight_format == "q8_0"
    B = wl.n_seq
    n_steps = args.tokens_per_step or wl.decode_steps
    model = q2.Qwen2Model(shape, weights, n_ctx=wl.n_ctx, max_seqs=B, max_tokens=sum(lens),
                          weight_format=q2.WEIGHTS_Q8_0 if q8 else q2.WEIGHTS_F16, flags=args.flags)
    seqs = list(range(B))
    _, ids = model.prefill(seqs, prompts)
    first = [int(t) for t in ids.cpu().numpy()]
    out = torch.empty((n_steps, B), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(dst):
        model.decode_steps(seqs, first, lens, n_steps, ids_out=dst)

    for _ in range(max(3, args.warmup)):
        step(out)
    model.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps.barrier()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            step(out)
        end.record(stream)
        torch.cuda.synchronize()
    reps.barrier()
    ms = reps.max(start.elapsed_time(end))
    model.synchronize()
    tokens = args.steps * n_steps * B * world
    value = tokens / (ms / 1e3)

    # End to end through the public API with host buffers: host token,
    # position and sequence-id inputs, ids read back into host memory.
    host_ids = np.empty((n_steps, B), dtype=np.int32)
    reps.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(host_ids)
    e2e_s = reps.max(time.perf_counter() - t0)
    e2e = {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 3 * 4 * B,
           "d2h_bytes_per_step": int(host_ids.nbytes)}

    persistent = B == 1 and bool(model.features & q2.FEATURE_PERSISTENT_DECODE) and not (
        args.flags & (q2.FLAG_NO_MEGAKERNEL | q2.FLAG_NO_FUSE_QKV | q2.FLAG_NO_FUSE_FFN))
    hbm, tflops, src = peaks()
    step_bytes = float(np.mean([decode_bytes_per_step(shape, [n + i for n in lens], q8) for i in range(n_steps)]))
    per_dec_s = (ms / 1e3) / (args.steps * n_steps)
    achieved = step_bytes / per_dec_s / 1e9
    if persistent:
        kname = "one decode token: k_decode_persistent (one launch per token)"
        launches = 1
    elif q8:
        kname = f"one decode step of {B} sequences: all kernels of the step graph (Q8_0 warp-MMA products, " \
                "TF32 flash-decoding attention + merge)"
        launches = 1 + shape.n_layer * 6 + 2
    else:
        kname = f"one decode step of {B} sequences: all kernels of the step graph"
        launches = 2 + shape.n_layer * 5
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": kernel_traffic("k_decode_persistent", wl.name) if persistent else None,
                "kernel": kname, "peak_source": src, "bytes_per_launch": step_bytes}
    dtype = ("f32 activations, Q8_0 weights (exact f32 dequantisation). Products: activations as f16 hi/lo "
             "MMA operand pairs, the LM head's as f16 only; attention: q, k and p rounded to TF32, v as a "
             "TF32 hi/lo pair; f32 accumulation, softmax and KV" if q8 else
             "f32 activations and accumulation, f16 weights, f32 KV")
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded random weights of the Qwen2.5-0.5B shape, uniform-random tokens)",
            "config": workload_config(wl, shape, world), "clocks": clocks.summary(), "e2e": e2e,
            "roofline": roofline, "gpu_launches": launches * n_steps * args.steps,
            "decode_kernel": "persistent" if persistent else "per-step"}
    model.close()
    return line


HEADLINE = "0.5b-decode-b1"
# The other workloads the metric names, measured by the default run and
# reported under "workloads" of the headline's line.
OTHERS = ("0.5b-decode-b1-long", "0.5b-prefill-8x512", "0.5b-decode-b32-q8")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(synth.WORKLOADS),
                    help="one workload alone (default: the batch-1 decode line, with the other 0.5B "
                         "workloads under 'workloads')")
    ap.add_argument("--tokens-per-step", type=int, default=0,
                    help="override the decode tokens of one timed step (profiling runs only)")
    ap.add_argument("--skip-cpu-baseline", action="store_true", help="profiling runs: no oracle timing")
    ap.add_argument("--flags", type=int, default=0, help="QWEN2_FLAG_* bits for the context")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    name = args.workload or HEADLINE
    wl = synth.WORKLOADS[name]
    shape = synth.SHAPES[wl.shape]
    if args.impl == "reference":
        if rank != 0:
            return  # the oracle arm runs on rank 0 alone; other ranks exit 0 without work
        weights = synth.make_weights(shape, wl.weight_seed)
        print(json.dumps(reference_line(args, wl, shape, weights, args.gpus)), flush=True)
        return

    import torch
    torch.cuda.set_device(local)
    reps = Replicas(world, "nccl", torch.device("cuda", local))
    weights = synth.make_weights(shape, wl.weight_seed)
    run = lambda w: (run_prefill if w.decode_steps == 0 else run_decode)(  # noqa: E731
        args, w, synth.SHAPES[w.shape], synth.make_weights(synth.SHAPES[w.shape], w.weight_seed), reps, world)
    line = run(wl)
    extra = {}
    if args.workload is None:
        for other in OTHERS:
            extra[other] = run(synth.WORKLOADS[other])
    if rank == 0 and not args.skip_cpu_baseline:
        timer = OracleTimer(shape, weights)
        line["cpu_baseline"] = timer.baseline(wl)
        for other, rec in extra.items():
            rec["cpu_baseline"] = timer.baseline(synth.WORKLOADS[other])
    if extra:
        keep = ("value", "unit", "ms_per_step", "steps", "dtype", "config", "roofline", "e2e", "clocks",
                "gpu_launches", "cpu_baseline", "decode_kernel")
        line["workloads"] = {k: {f: v[f] for f in keep if f in v} for k, v in extra.items()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    reps.close()


if __name__ == "__main__":
    main()
