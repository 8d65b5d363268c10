"""Benchmark: MoE decode tokens/s per layer stack, and the kernels' rooflines.

Default workload (the metric's configuration): a 48-layer MoE-only stack,
each layer of Qwen3.8-Flash-Next shape (H 2048, 512 routed experts top-10 +
1 shared, I 512, 4-bit block-32 weights with fp16 scales, Zipf(1.1) router
bias; 0.91 GB of packed experts per layer, 43.5 GB in all), residual +
RMSNorm (eps 1e-6) between layers, batch 1.  Every layer's VRAM slot pool
holds 128 of its 512 experts (25 %, LRU); misses come from the layer's
pinned host master copy after the in-kernel hit check rings the host
doorbell.  One step = the configuration's measured window: the pools start
empty, 64 warm-up tokens run untimed, then 256 decode tokens are timed,
each token one CUDA-graph replay of the 48 layer calls.

  value         tokens/s of the 25 % pool stack, inputs resident in HBM
  resident      the same stack with every expert resident (bit-identical
                output required); its decode kernel gives the roofline line
  roofline      HBM: algorithmic bytes of one layer-token (router fp32 + 11
                experts) per decode-kernel launch / mean launch time, against
                the measured HBM copy bandwidth
  pool          25 % pool: misses, host-link GB/s against the measured
                host -> device copy bandwidth
  miss_heavy    16-slot pools (3 %): the host link is the bound; host-link
                GB/s against the measured host -> device copy bandwidth
  pool_copy_engine  25 % pool with the host copy server serving misses
  e2e           the pooled stack through the public API: each token's x
                copied host -> device and the stack output device -> host
  cpu_baseline  the CPU oracle (binary64, single-threaded, as written) on a
                sample of the same stack, one core and every host core
  c2_layer, c3_batched, c5_prefill   the single-layer, batched-decode and
                prefill configurations, each with its own roofline

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas; the layer does not shard across GPUs here) and rank 0 prints the
aggregate.  --impl reference times the CPU oracle instead (rank 0 only).
--workload decode|batched|prefill runs one secondary configuration alone.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE decode tokens/s per layer stack; expert-weight HBM GB/s vs 8 TB/s peak"
UNIT = "tokens/s"
H, E, K, I = 2048, 512, 10, 512
EXPERT_BYTES = 1_769_472
ROUTER_BYTES = E * H * 4
STEP_BYTES_PER_TOKEN = ROUTER_BYTES + (K + 1) * EXPERT_BYTES  # 23,658,496 per layer-token
N_LAYERS = 48
POOL_SLOTS = 128        # 25 % of 512
HEAVY_SLOTS = 16        # 3 %: misses dominate
WARM_TOKENS = 64        # untimed tokens before each measured window
WINDOW_TOKENS = 256     # measured tokens per step
HEAVY_WINDOW = 64       # measured tokens per miss-heavy step
C2_TOKENS = 1000
C2_REPLICAS = 8
PREFILL_T = 4096
PREFILL_PAIRS = PREFILL_T * (K + 1)                   # routed pairs + shared-expert rows
PREFILL_FLOPS = 2 * PREFILL_PAIRS * 3 * H * I         # gate, up, down: 283.5 GFLOP on the tensor cores
STACK_WORKLOAD = (f"{N_LAYERS}-layer page-scale MoE stack (H 2048, 512 routed experts top-10 + 1 shared, I 512, "
                  "4-bit block-32 fp16-scale weights, Zipf(1.1) router bias), residual + RMSNorm eps 1e-6 between "
                  f"layers, batch 1; {POOL_SLOTS}-slot (25 %) LRU expert pool per layer, misses from pinned host "
                  f"RAM after the host doorbell; per step the pools start empty, {WARM_TOKENS} warm-up tokens, then "
                  f"{WINDOW_TOKENS} timed decode tokens")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, pg=None, device="cpu"):
    """Elementwise max of per-rank figures (the slowest rank sets the job's
    time); the values themselves on one rank."""
    if pg is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, world_size, ms):
    """Units all ranks processed per second of the slowest rank's time."""
    return units_per_rank * world_size / (ms * 1e-3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "kind": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "kind": "fallback"}


def source_hash():
    """Hash of the decode kernel's sources: a recorded traffic figure is used
    only while the kernel it was measured on is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_expert_ffn_gemv_gb300", "csrc")
    for f in ("moe_decode.cu", "moe_internal.h", "moe_mma.cuh", "moe_route.cuh", "moe_norm.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram bytes per decode launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        d = json.load(open(p))
        if d.get("source_hash") == source_hash():
            return d["dram_bytes_per_token"]
    except Exception:
        pass
    return None


def spread(per_token_ms):
    """median, p10, p90 of per-token times (ms) as tokens/s figures."""
    a = np.asarray(per_token_ms, np.float64)
    return {"per_token_us_median": float(np.median(a) * 1e3), "per_token_us_p10": float(np.percentile(a, 10) * 1e3),
            "per_token_us_p90": float(np.percentile(a, 90) * 1e3), "samples": int(a.size),
            "tokens_per_s_median": float(1e3 / np.median(a))}


class ClockSampler:
    def __init__(self, path):
        self.path = path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # the timed region starts once the sampler is running (its first row
        # is written), so that even a short region is sampled
        t_end = time.time() + 2.0
        while self.proc and time.time() < t_end:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.01)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self, gpu_index):
        try:
            rows = [r.split(", ") for r in open(self.path).read().strip().splitlines()]
        except Exception:
            return None
        rows = [r for r in rows if len(r) >= 9 and r[0].strip() == str(gpu_index)]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6), ("sw_thermal_slowdown", 7),
                              ("sw_power_cap", 8)):
                if r[col].strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows)}


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_stack_rate(sample_layers, calls, threads):
    """Stack tokens/s of the CPU oracle, as written, from `calls` layer-token
    calls spread over the sample layers (token-parallel on `threads` threads:
    the C oracle is reentrant and ctypes releases the GIL during a call).
    A stack token is N_LAYERS layer calls, so the rate is calls / time / N_LAYERS."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from quantized_expert_ffn_gemv_gb300 import synth
    x = synth.activations(synth.PAGE, 1000, 0, max(calls, 1), stream=9)

    def one(i):
        L = sample_layers[i % len(sample_layers)]
        oracle.moe_forward(H, I, E, K, L.W_r, L.bias, L.experts, L.shared, x[i:i + 1])

    if threads == 1:
        t0 = time.perf_counter()
        for i in range(calls):
            one(i)
        dt = time.perf_counter() - t0
    else:
        with ThreadPoolExecutor(max_workers=threads) as pool:
            list(pool.map(one, range(threads)))  # threads up
            t0 = time.perf_counter()
            list(pool.map(one, range(calls)))
            dt = time.perf_counter() - t0
    return calls / dt / N_LAYERS


def cpu_baseline(sample_layers):
    cores = host_cores()
    one = oracle_stack_rate(sample_layers, 48, 1)
    line = {"value": one, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"48 layer-token calls (one token through {len(sample_layers)} of the stack's layers in turn), "
                      f"single-threaded binary64 C oracle; stack tokens/s = calls/s / {N_LAYERS}"}
    if cores > 1:
        line["all_cores"] = {"value": oracle_stack_rate(sample_layers, 16 * cores, cores), "unit": UNIT,
                             "cores": cores, "sample": f"{16 * cores} layer-token calls on {cores} threads"}
    return line


def run_reference(args):
    """The CPU oracle on the default workload's metric: stack tokens/s, each
    step one decode token through two of the stack's layers on every host
    core (one token per core), scaled to the 48-layer stack."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from quantized_expert_ffn_gemv_gb300 import synth
    sample = [synth.make_layer(synth.PAGE, layer=l) for l in range(2)]
    cores = host_cores()
    times = []
    for s in range(args.warmup + args.steps):
        v = oracle_stack_rate(sample, 2 * cores, cores)
        if s >= args.warmup:
            times.append(v)
    value = float(np.mean(times))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * 2 * cores / (value * N_LAYERS), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": STACK_WORKLOAD, "sample_per_step": f"{cores} tokens x 2 layers (of {N_LAYERS}), "
                                                                     "stack tokens/s scaled by 2/48"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"per step {2 * cores} layer-token calls of two stack layers, one token per "
                                       f"core, single-threaded binary64 C oracle on each of {cores} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def h2d_peak_gbs(torch, nbytes, reps):
    src = torch.empty(nbytes * 4, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes * 4, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(4):
            dst[i * nbytes:(i + 1) * nbytes].copy_(src[i * nbytes:(i + 1) * nbytes], non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for r in range(reps):
            i = r % 4
            dst[i * nbytes:(i + 1) * nbytes].copy_(src[i * nbytes:(i + 1) * nbytes], non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    return nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9


# ---------------------------------------------------------------------------- the stack


class StackBench:
    """The 48 layer objects, their CUDA graph of one token, and timed windows."""

    def __init__(self, torch, layers):
        from quantized_expert_ffn_gemv_gb300.stack import MoeStack
        self.torch = torch
        self.layers = layers

        class _Stack(MoeStack):
            def __init__(s, objs):
                s.layers, s.eps, s.H, s.k = objs, 1e-6, H, K
                s.device = torch.device("cuda", torch.cuda.current_device())

        self.st = _Stack(layers)
        self.st.link()  # each layer warms L2 with the next layer's router rows and shared expert
        self.stream = torch.cuda.Stream()
        self.xin = torch.empty((1, H), dtype=torch.bfloat16, device="cuda")
        self.bufs = self.st.buffers(1)
        self.graph = None

    def hot_lists(self, x_dev, n_tok, n_hot):
        """Each layer's n_hot most-selected experts over n_tok tokens of an
        eager, every-expert-resident pass (a hot-expert profile)."""
        torch = self.torch
        self.configure(E, 1)
        rec = self.st.buffers(1, record=True)
        counts = torch.zeros((len(self.layers), E), dtype=torch.int64, device="cuda")
        ones = torch.ones((len(self.layers), K), dtype=torch.int64, device="cuda")
        with torch.cuda.stream(self.stream):
            for t in range(n_tok):
                self.xin.copy_(x_dev[t:t + 1], non_blocking=True)
                self.st.forward(self.xin, rec, self.stream)
                counts.scatter_add_(1, rec["idx"].reshape(len(self.layers), -1).long(), ones)
        torch.cuda.synchronize()
        return [np.argsort(-c, kind="stable")[:n_hot].astype(np.int32).tolist() for c in counts.cpu().numpy()]

    def configure(self, n_slots, service=1):
        for layer in self.layers:
            layer.configure(n_slots)
            layer.set_miss_service(service)

    def capture(self):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            self.st.forward(self.xin, self.bufs, self.stream)  # first call: host-side set-up
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.out = self.st.forward(self.xin, self.bufs, self.stream)
        torch.cuda.synchronize()

    def totals(self):
        ss = [l.stats() for l in self.layers]
        return (sum(s["misses"] for s, _ in ss), sum(s["h2d_bytes"] for s, _ in ss), [c for _, c in ss])

    def window(self, x_src, t0, warm, n, reset, outs=None, host_out=None):
        """One measured window: pools reset (reconfigured) if `reset`, `warm`
        untimed tokens, then `n` timed tokens with an event before each.
        x_src: device (resident inputs) or pinned host tensor [tokens, H];
        host_out: pinned host [n, H] for the end-to-end variant (each token's
        output copied back inside the timed region).  Returns per-token ms,
        total ms, misses and host-link bytes of the timed tokens."""
        torch = self.torch
        if reset is not None:
            self.configure(*reset)
        s = self.stream
        with torch.cuda.stream(s):
            for t in range(warm):
                self.xin.copy_(x_src[t0 + t:t0 + t + 1], non_blocking=True)
                self.graph.replay()
        torch.cuda.synchronize()
        m0, b0, _ = self.totals()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(s):
            for t in range(n):
                ev[t].record(s)
                i = t0 + warm + t
                self.xin.copy_(x_src[i:i + 1], non_blocking=True)
                self.graph.replay()
                if outs is not None:
                    outs[i:i + 1].copy_(self.out, non_blocking=True)
                if host_out is not None:
                    host_out[t:t + 1].copy_(self.out, non_blocking=True)
            ev[n].record(s)
        torch.cuda.synchronize()
        m1, b1, codes = self.totals()
        if any(codes):
            raise RuntimeError(f"layer errors {codes}")
        per = [ev[t].elapsed_time(ev[t + 1]) for t in range(n)]
        return per, ev[0].elapsed_time(ev[n]), m1 - m0, b1 - b0

    def run(self, x_dev, n_slots, service, steps, warmup, warm, n, outs=None):
        """warmup + steps windows (each from empty pools); the timed steps'
        per-token times, total ms, misses and host-link bytes."""
        self.configure(n_slots, service)
        self.capture()
        per, tot, miss, byt = [], 0.0, 0, 0
        for s in range(warmup + steps):
            p, ms, m, b = self.window(x_dev, 0, warm, n, (n_slots, service), outs if s == warmup else None)
            if s >= warmup:
                per += p
                tot += ms
                miss += m
                byt += b
        return per, tot, miss, byt


def decode_launch_time(torch, layers, x_dev, tokens):
    """Mean device time of one decode-kernel launch (one layer-token), from
    CUDA events around a graph of single-token calls on the launching stream:
    resident layers round-robin (inputs > L2), one fused kernel per call."""
    stream = torch.cuda.Stream()
    y = torch.empty((tokens, H), dtype=torch.bfloat16, device="cuda")
    for i, layer in enumerate(layers):  # the call after layer i's is layer i + 1's
        layer.set_next(layers[(i + 1) % len(layers)])

    def step():
        for t in range(tokens):
            layers[t % len(layers)].forward(x_dev[t:t + 1], y[t:t + 1], stream=stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    with torch.cuda.stream(stream):
        for i in range(5):
            ev[i].record(stream)
            g.replay()
        ev[5].record(stream)
    torch.cuda.synchronize()
    per_call = [ev[i].elapsed_time(ev[i + 1]) / tokens for i in range(5)]
    return statistics.median(per_call), g, stream, y


def c3_batched(torch, layers, T, x_dev):
    """Calls of T independent tokens through the page-scale layer, layer
    objects round-robin (all experts resident); bytes of a call = W_r + its
    distinct routed experts (from the call's routing output) + the shared
    expert."""
    pk = peaks()
    calls = (C2_TOKENS + T - 1) // T
    ntok = calls * T
    xd = x_dev[:ntok]
    yd = torch.empty_like(xd)
    idx = torch.empty((ntok, K), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        for c in range(calls):
            sl = slice(c * T, (c + 1) * T)
            layers[c % len(layers)].forward(xd[sl], yd[sl], idx[sl], stream=stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    routed = idx.cpu().numpy().reshape(calls, T * K)
    distinct = [len(np.unique(r)) for r in routed]
    step_bytes = sum(ROUTER_BYTES + (d + 1) * EXPERT_BYTES for d in distinct)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(11)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        for i in range(10):
            ev[i].record(stream)
            g.replay()
        ev[10].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(10)]
    ms = statistics.median(per)
    achieved = step_bytes / (ms * 1e-3) / 1e9
    return {"tokens_per_s": ntok / (ms * 1e-3), "batch": T, "calls_per_step": calls, "layers_round_robin": len(layers),
            "path": "fused decode kernel" if T <= 8 else "route_kernel + gateup_kernel + down_kernel",
            "ms_per_step_median": ms, "ms_per_step_p10": float(np.percentile(per, 10)),
            "ms_per_step_p90": float(np.percentile(per, 90)),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "peak_kind": pk["kind"],
                         "bytes_per_call": step_bytes / calls, "distinct_experts_per_call": sum(distinct) / calls}}


def c5_prefill(torch, layer, x_dev):
    """One 4,096-token chunk per step (grouped GEMMs on the tensor cores).
    Algorithmic bytes: the experts the call's routing touched (from its
    output) + the shared expert + W_r + x in and y out."""
    pk = peaks()
    xd = x_dev[:PREFILL_T]
    yd = torch.empty_like(xd)
    idx = torch.empty((PREFILL_T, K), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(3):
            layer.forward(xd, yd, idx, stream=stream)
    torch.cuda.synchronize()
    touched = len(np.unique(idx.cpu().numpy()))
    st0, _ = layer.stats()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(11)]
    with torch.cuda.stream(stream):
        for i in range(10):
            ev[i].record(stream)
            layer.forward(xd, yd, stream=stream)
        ev[10].record(stream)
    torch.cuda.synchronize()
    st1, code = layer.stats()
    if code:
        raise RuntimeError(f"prefill error {code}")
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(10)]
    ms = statistics.median(per)
    tflops = PREFILL_FLOPS / (ms * 1e-3) / 1e12
    nbytes = (touched + 1) * EXPERT_BYTES + ROUTER_BYTES + 2 * 2 * PREFILL_T * H
    return {"tokens_per_s": PREFILL_T / (ms * 1e-3), "ms_per_chunk_median": ms,
            "ms_per_chunk_p10": float(np.percentile(per, 10)), "ms_per_chunk_p90": float(np.percentile(per, 90)),
            "roofline": {"bound": "tensor", "kernel": "whole moe_forward call", "achieved": tflops,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": tflops / pk["bf16_tflops"],
                         "peak_kind": f"{pk['kind']} bf16 burst (f16 runs at the bf16 rate)",
                         "flops_per_chunk": PREFILL_FLOPS},
            "hbm": {"algorithmic_bytes": nbytes, "touched_experts": touched,
                    "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
                    "frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
            "exact_rechecks_per_chunk": (st1["rechecks"] - st0["rechecks"]) / 10}


def run_default(args):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_expert_ffn_gemv_gb300 import moe, synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    pk = peaks()

    # ---- the 48 layers (weights generated, repacked, pinned; all resident first)
    t_setup = time.time()
    layers, keep = [], {}
    for l in range(N_LAYERS):
        L = synth.make_layer(synth.PAGE, layer=l)
        layers.append(moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=1, device=local))
        if l < 4:
            keep[l] = L
        del L
    # prefill- and batch-capable objects of layers 0..3 (a pooled layer must take T <= 12)
    wide = [moe.MoeLayer(keep[l].shape, keep[l].W_r, keep[l].bias, keep[l].experts, keep[l].shared,
                         max_tokens=PREFILL_T, device=local) for l in range(4)]
    setup_s = time.time() - t_setup
    sample = [keep[0], keep[1]]
    for l in (2, 3):
        del keep[l]

    ntok = WARM_TOKENS + WINDOW_TOKENS
    x_host = synth.activations(synth.PAGE, 1000, 0, max(ntok, PREFILL_T), stream=9)
    x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    x_dev = x_pin.to("cuda")
    sb = StackBench(torch, layers)
    if args.hot > 0:
        # each layer also warms the next layer's hot experts (profile of the warm-up tokens)
        sb.st.link(sb.hot_lists(x_dev, WARM_TOKENS, args.hot))

    def barrier():
        if pg:
            pg.barrier()
        torch.cuda.synchronize()

    # ---- resident stack: bit-identity reference and the roofline
    out_res = torch.empty((ntok, H), dtype=torch.bfloat16, device="cuda")
    barrier()
    per_res, ms_res, _, _ = sb.run(x_dev, E, 1, args.steps, args.warmup, WARM_TOKENS, WINDOW_TOKENS, out_res)
    # ---- the configuration: 25 % pools, misses read by the kernel from pinned host RAM
    out_pool = torch.empty((ntok, H), dtype=torch.bfloat16, device="cuda")
    barrier()
    clocks = ClockSampler(os.path.join(tempfile.gettempdir(), f"bench_clocks_{rank}.csv"))
    with clocks:
        per_pool, ms_pool, miss_pool, h2d_pool = sb.run(x_dev, POOL_SLOTS, 1, args.steps, args.warmup, WARM_TOKENS,
                                                        WINDOW_TOKENS, out_pool)
        barrier()
    identical = bool(torch.equal(out_pool.view(torch.int16), out_res.view(torch.int16)))
    # ---- end to end: x from pinned host memory, the stack output back to it, per token
    host_out = torch.empty((WINDOW_TOKENS, H), dtype=torch.bfloat16).pin_memory()
    e2e_ms = 0.0
    for s in range(args.warmup + args.steps):
        _, ms, _, _ = sb.window(x_pin, 0, WARM_TOKENS, WINDOW_TOKENS, (POOL_SLOTS, 1), host_out=host_out)
        if s >= args.warmup:
            e2e_ms += ms
    # ---- miss-heavy pools: the host link is the bound
    per_heavy, ms_heavy, miss_heavy, h2d_heavy = sb.run(x_dev, HEAVY_SLOTS, 1, max(3, args.steps // 4), 1, 16,
                                                        HEAVY_WINDOW)
    # ---- 25 % pools with the host copy server serving the misses
    try:
        out_copy = torch.empty((ntok, H), dtype=torch.bfloat16, device="cuda")
        per_copy, ms_copy, miss_copy, h2d_copy = sb.run(x_dev, POOL_SLOTS, 0, max(3, args.steps // 4), 1,
                                                        WARM_TOKENS, WINDOW_TOKENS, out_copy)
        n_copy = max(3, args.steps // 4) * WINDOW_TOKENS
        copy_line = {"tokens_per_s": n_copy / (ms_copy * 1e-3), "misses": miss_copy,
                     "h2d_gbs": h2d_copy / (ms_copy * 1e-3) / 1e9, **spread(per_copy),
                     "bit_identical_vs_resident": bool(torch.equal(out_copy.view(torch.int16),
                                                                   out_res.view(torch.int16)))}
    except (moe.MoeError, RuntimeError) as e:
        copy_line = {"error": str(e)}
    sb.configure(E, 1)
    h2d_small = h2d_peak_gbs(torch, EXPERT_BYTES, 256)
    h2d_large = h2d_peak_gbs(torch, 64 << 20, 16)
    h2d_peak = max(h2d_small, h2d_large)

    # ---- the decode kernel alone: mean launch time over resident layers round-robin
    launch_ms, _, _, _ = decode_launch_time(torch, layers[:C2_REPLICAS], x_dev, C2_TOKENS)
    # ---- secondary configurations
    c2_tps = 1e3 / launch_ms
    c2 = {"tokens_per_s": c2_tps, "workload": f"one page-scale layer, {C2_TOKENS} independent decode tokens "
                                              f"(batch 1) per step over {C2_REPLICAS} distinct resident layers "
                                              "round-robin (inputs > L2), one fused kernel per token",
          "roofline": {"bound": "hbm", "achieved": STEP_BYTES_PER_TOKEN * c2_tps / 1e9, "peak": pk["hbm_gbs"],
                       "unit": "GB/s", "frac": STEP_BYTES_PER_TOKEN * c2_tps / 1e9 / pk["hbm_gbs"],
                       "peak_kind": pk["kind"], "bytes_per_token": STEP_BYTES_PER_TOKEN}}
    c3 = {f"T{T}": c3_batched(torch, wide, T, x_dev) for T in (8, 64)}
    c5 = c5_prefill(torch, wide[0], x_dev)

    ms_res, ms_pool, e2e_ms = max_over_ranks([ms_res, ms_pool, e2e_ms], pg, device="cuda")
    if rank != 0:
        for l in layers:
            l.set_next(None)
        for l in layers + wide:
            l.close()
        pg.destroy_process_group() if pg else None
        return
    n_timed = args.steps * WINDOW_TOKENS
    value = whole_job_rate(n_timed, ws, ms_pool)
    res_tps = n_timed / (ms_res * 1e-3)
    launches_per_token = N_LAYERS + 1  # 48 decode kernels + the closing residual add
    res_launch_s = ms_res * 1e-3 / n_timed / N_LAYERS
    achieved = STEP_BYTES_PER_TOKEN / res_launch_s / 1e9
    heavy_n = max(3, args.steps // 4) * HEAVY_WINDOW
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_pool / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 x f16 MMA, f32 accumulate, 4-bit weights; h stored f16; router compensated f32",
        "data": "synthetic",
        "config": {"workload": STACK_WORKLOAD, "layers": N_LAYERS, "slots_per_layer": POOL_SLOTS,
                   "tokens_per_step": WINDOW_TOKENS, "warmup_tokens_per_step": WARM_TOKENS,
                   "l2": "inputs larger than L2 (43.5 GB of expert weights)", "parallelism": f"replicas x{ws}",
                   "next_layer_l2_warmup": "router rows + shared expert" + (f" + {args.hot} hot experts from a "
                                                                            "64-token profile" if args.hot else "")},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (fused router + top-k + hit check + gate/up + down), "
                                               "resident stack", "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "peak_kind": pk["kind"],
                     "bytes_per_launch": STEP_BYTES_PER_TOKEN, "unit_of_work": "layer-token (one launch)",
                     "traffic": recorded_traffic()},
        "timing": spread(per_pool),
        "resident": {"tokens_per_s": res_tps, **spread(per_res),
                     "hbm_gbs": N_LAYERS * STEP_BYTES_PER_TOKEN * res_tps / 1e9,
                     "hbm_frac": N_LAYERS * STEP_BYTES_PER_TOKEN * res_tps / 1e9 / pk["hbm_gbs"]},
        "pool": {"tokens_per_s": value, "misses": miss_pool, "misses_per_layer_token": miss_pool / n_timed / N_LAYERS,
                 "h2d_bytes_per_token": h2d_pool / n_timed, "h2d_gbs": h2d_pool / (ms_pool * 1e-3) / 1e9,
                 "h2d_frac": h2d_pool / (ms_pool * 1e-3) / 1e9 / h2d_peak,
                 "service": "kernel reads misses from pinned host RAM (after the host doorbell)"},
        "miss_heavy": {"slots_per_layer": HEAVY_SLOTS, "tokens_per_s": heavy_n / (ms_heavy * 1e-3),
                       "misses": miss_heavy, "misses_per_layer_token": miss_heavy / heavy_n / N_LAYERS,
                       "h2d_gbs": h2d_heavy / (ms_heavy * 1e-3) / 1e9,
                       "h2d_frac": h2d_heavy / (ms_heavy * 1e-3) / 1e9 / h2d_peak, **spread(per_heavy),
                       "window": f"16 warm-up + {HEAVY_WINDOW} timed tokens per step from empty pools"},
        "h2d_peak": {"gbs": h2d_peak, "expert_copies_gbs": h2d_small, "copies_64MB_gbs": h2d_large,
                     "how": "pinned cudaMemcpyAsync host -> device, CUDA events"},
        "pool_copy_engine": copy_line,
        "bit_identical_pool_vs_resident": identical,
        "e2e": {"value": whole_job_rate(n_timed, ws, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": WINDOW_TOKENS * H * 2,
                "d2h_bytes_per_step": WINDOW_TOKENS * H * 2},
        "gpu_launches": n_timed * launches_per_token,
        "clocks": clocks.summary(local),
        "c2_layer": c2,
        "c3_batched": c3,
        "c5_prefill": c5,
        "decode_launch_us": launch_ms * 1e3,
        "setup_s": setup_s,
    }
    if ws == 1 and args.cpu_sample:
        line["cpu_baseline"] = cpu_baseline(sample)
    print(json.dumps(line), flush=True)
    for l in layers:
        l.set_next(None)
    for l in layers + wide:
        l.close()
    if pg:
        pg.destroy_process_group()


def run_single(args):
    """One secondary configuration alone (quick iteration)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_expert_ffn_gemv_gb300 import moe, synth
    torch.cuda.set_device(0)
    n = (args.replicas or C2_REPLICAS) if args.workload == "decode" else 4
    mt = 1 if args.workload == "decode" else PREFILL_T
    layers = []
    for l in range(n):
        L = synth.make_layer(synth.PAGE, layer=l)
        layers.append(moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=mt))
        del L
    x_host = synth.activations(synth.PAGE, 1000, 0, PREFILL_T, stream=9)
    x_dev = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).cuda()
    if args.workload == "decode":
        ms, _, _, _ = decode_launch_time(torch, layers, x_dev, args.tokens or C2_TOKENS)
        pk = peaks()
        out = {"workload": "c2 decode", "tokens_per_s": 1e3 / ms, "us_per_token": ms * 1e3,
               "frac": STEP_BYTES_PER_TOKEN / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    elif args.workload == "batched":
        out = c3_batched(torch, layers, args.batch, x_dev)
    else:
        out = c5_prefill(torch, layers[0], x_dev)
    print(json.dumps(out), flush=True)
    for l in layers:
        l.set_next(None)
    for l in layers:
        l.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=1, help="0: skip the cpu_baseline timing")
    ap.add_argument("--workload", default="stack", choices=["stack", "decode", "prefill", "batched"],
                    help="stack: the 48-layer stack with every configuration (default); decode: one page-scale "
                         "layer, batch 1; prefill: one 4096-token chunk; batched: calls of --batch tokens")
    ap.add_argument("--batch", type=int, default=8, help="tokens per call for --workload batched (2..64)")
    ap.add_argument("--hot", type=int, default=0, help="hot experts per layer the previous layer warms in L2")
    ap.add_argument("--replicas", type=int, default=0, help="--workload decode: layer replicas (default 8; 1 for a "
                                                              "small profiling case)")
    ap.add_argument("--tokens", type=int, default=0, help="--workload decode: tokens per graph (default 1000)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "stack":
        return run_default(args)
    return run_single(args)


if __name__ == "__main__":
    main()
