"""Benchmark: MoE decode tokens/s of the page-scale quantized expert-FFN layer.

Workload (one "step"): 1,000 decode tokens, batch 1, through the MoE layer of
Qwen3.8-Flash-Next shape (H 2048, 512 routed experts top-10 + 1 shared,
I 512, 4-bit block-32 weights, Zipf(1.1) router bias), cycling round-robin
over 8 byte-identical layer replicas (8 x 0.91 GB of expert weights > L2),
all experts resident.  Each token is one moe_forward call (one fused
kernel); the 1,000 calls are replayed as one CUDA graph.

  value  tokens/s with inputs resident in HBM (CUDA events on the stream)
  e2e    the same through the public API with the step's activations copied
         host -> device and the outputs device -> host inside the timed region
  roofline  algorithmic bytes of one decode step (router fp32 + 11 experts)
         per token / time per token, against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle (single-threaded binary64) on a bounded sample

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas; the layer does not shard across GPUs here) and rank 0 prints the
aggregate.  --impl reference times the CPU oracle instead (rank 0 only).

Other workloads (one JSON line each, same keys):
  --workload stack    48 page-scale layers, residual + RMSNorm, 25% slot pool
  --workload prefill  one 4,096-token prefill chunk through the page-scale
                      layer (grouped GEMMs on the tensor cores)
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
TOKENS_PER_STEP = 1000
REPLICAS = 8
H, E, K, I = 2048, 512, 10, 512
EXPERT_BYTES = 1_769_472
ROUTER_BYTES = E * H * 4
STEP_BYTES_PER_TOKEN = ROUTER_BYTES + (K + 1) * EXPERT_BYTES  # 23,658,496
WORKLOAD = ("page-scale MoE layer decode, batch 1: H 2048, 512 routed experts top-10 + 1 shared, I 512, "
            "4-bit block-32 fp16-scale weights, Zipf(1.1) router bias; {tokens} tokens per step over {replicas} "
            "identical layer replicas round-robin, all experts resident")


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


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_hash():
    """Hash of the decode kernel's sources: a recorded traffic figure is used
    only while the kernel it was measured on is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_expert_ffn_gemv_gb300", "csrc")
    for f in ("moe_decode.cu", "moe_internal.h", "moe_mma.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram bytes per token from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        d = json.load(open(p))
        if d.get("source_hash") == source_hash():
            return d["dram_bytes_per_token"]
    except Exception:
        pass
    return None


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


def cpu_baseline(L, tokens):
    """Time the oracle, as written, on `tokens` decode tokens on one core;
    then the same calls token-parallel on every host core (threads: the C
    oracle is reentrant and ctypes releases the GIL during the call)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    x = L_tokens(L, 0, tokens)
    one = lambda t: oracle.moe_forward(H, I, E, K, L.W_r, L.bias, L.experts, L.shared, x[t:t + 1])
    t0 = time.perf_counter()
    for t in range(tokens):
        one(t)
    dt = time.perf_counter() - t0
    line = {"value": tokens / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{tokens} decode tokens (batch 1) of the page-scale layer, single-threaded binary64 C oracle"}
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    if cores > 1 and tokens > 0:
        n = max(tokens, 2 * cores)
        x = L_tokens(L, 0, n)
        with ThreadPoolExecutor(max_workers=cores) as pool:
            list(pool.map(one, range(min(n, cores))))  # threads up
            t0 = time.perf_counter()
            list(pool.map(one, range(n)))
            dt = time.perf_counter() - t0
        line["all_cores"] = {"value": n / dt, "unit": UNIT, "cores": cores,
                             "sample": f"{n} decode tokens, one per task, on {cores} threads"}
    return line


def L_tokens(L, t0, n):
    from quantized_expert_ffn_gemv_gb300 import synth
    return synth.activations(L.shape, L.index, t0, n, stream=7)


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from quantized_expert_ffn_gemv_gb300 import synth
    import oracle
    L = synth.make_layer(synth.PAGE, layer=0)
    per_step = 4
    x = L_tokens(L, 0, per_step * (args.steps + args.warmup))
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for t in range(per_step):
            i = s * per_step + t
            oracle.moe_forward(H, I, E, K, L.W_r, L.bias, L.experts, L.shared, x[i:i + 1])
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = per_step * args.steps / tot
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD.format(tokens=args.tokens, replicas=args.replicas),
                       "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{per_step} decode tokens per step, single-threaded binary64 C oracle"},
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


def run_stack(args):
    """48 distinct page-scale layers, residual + RMSNorm between them, each
    layer's VRAM slot pool capped at 128 of 512 experts (LRU, misses read
    from pinned host RAM by the kernel after the host doorbell); 64 warm-up
    then 256 measured decode tokens, batch 1.  The same stack also runs with
    every expert resident (outputs must be bit-identical; that run gives the
    HBM roofline figure), with tiered per-layer budgets and profile-seeded
    pools, and with the host copy engine serving the misses."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_expert_ffn_gemv_gb300 import moe, synth
    from quantized_expert_ffn_gemv_gb300.stack import MoeStack
    torch.cuda.set_device(0)
    n_layers, slots = args.layers, 128
    warm = max(args.warmup, 64)
    meas = args.steps
    t0 = time.time()
    layer_objs = []
    for l in range(n_layers):
        L = synth.make_layer(synth.PAGE, layer=l)
        layer_objs.append(moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=1, n_slots=slots))
        del L
    setup_s = time.time() - t0

    class _Stack(MoeStack):
        def __init__(self, layers):
            self.layers, self.eps, self.H, self.k = layers, 1e-6, synth.PAGE.H, synth.PAGE.k
            self.device = torch.device("cuda", 0)

    st = _Stack(layer_objs)
    ntok = warm + meas
    x = synth.activations(synth.PAGE, 1000, 0, ntok, stream=9)
    x_pin = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    xin = torch.empty((1, synth.PAGE.H), dtype=torch.bfloat16, device="cuda")
    bufs = st.buffers(1)
    stream = torch.cuda.Stream()

    def totals():
        ss = [l.stats() for l in st.layers]
        return (sum(s["misses"] for s, _ in ss), sum(s["h2d_bytes"] for s, _ in ss), [c for _, c in ss],
                sum(s["wait_ns"] for s, _ in ss))

    def configure(n_slots, seeds):
        budgets = n_slots if isinstance(n_slots, list) else [n_slots] * n_layers
        for l, layer in enumerate(st.layers):
            layer.configure(budgets[l])
            if seeds is not None and budgets[l] < synth.PAGE.E:
                layer.seed(seeds[l][:budgets[l]])

    def run(n_slots, service=1, seeds=None, fused=True):
        configure(n_slots, seeds)
        for l in st.layers:
            l.set_miss_service(service)
        st.fused = fused
        outs = torch.empty((ntok, synth.PAGE.H), dtype=torch.bfloat16, device="cuda")
        with torch.cuda.stream(stream):
            xin.copy_(x_pin[0:1], non_blocking=True)
            st.forward(xin, bufs, stream)  # first call: host-side set-up
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            o = st.forward(xin, bufs, stream)
        configure(n_slots, seeds)  # start every pool as it was again
        with torch.cuda.stream(stream):
            for t in range(warm):
                xin.copy_(x_pin[t:t + 1], non_blocking=True)
                graph.replay()
                outs[t:t + 1].copy_(o)
        torch.cuda.synchronize()
        m0, b0, _, w0 = totals()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for t in range(warm, ntok):
                xin.copy_(x_pin[t:t + 1], non_blocking=True)
                graph.replay()
                outs[t:t + 1].copy_(o)
            ev[1].record(stream)
        torch.cuda.synchronize()
        m1, b1, codes, w1 = totals()
        return ev[0].elapsed_time(ev[1]), outs, m1 - m0, b1 - b0, codes, w1 - w0

    # every expert resident; then the default miss service (the kernel reads
    # misses from pinned host RAM), uniform and tiered + seeded; last the
    # host copy engine behind the doorbell (a bounded-wait error there leaves
    # the layers' sticky error set)
    ms_res, out_res, _, _, codes_res, _ = run(synth.PAGE.E)
    # the same, with the residual + RMSNorm as a kernel of its own between layers
    ms_split, out_split, _, _, _, _ = run(synth.PAGE.E, fused=False)
    st.fused = True
    ms_pool, out_pool, misses, h2d_bytes, codes, _ = run(slots, service=1)
    identical = bool(torch.equal(out_pool.view(torch.int16), out_res.view(torch.int16)))
    # per-layer budgets (early layers more, late fewer) and pools seeded from
    # a profile: each layer's most-selected experts over the warm-up tokens of
    # a resident profiling pass
    tiers = [240 if 3 * l < n_layers else (92 if 3 * l < 2 * n_layers else 60) for l in range(n_layers)]
    configure(synth.PAGE.E, None)
    prof = st.buffers(1, record=True)
    with torch.cuda.stream(stream):
        counts = torch.zeros((n_layers, synth.PAGE.E), dtype=torch.int64, device="cuda")
        for t in range(warm):
            xin.copy_(x_pin[t:t + 1], non_blocking=True)
            st.forward(xin, prof, stream)
            counts.scatter_add_(1, prof["idx"].reshape(n_layers, -1).long(),
                                torch.ones((n_layers, synth.PAGE.k), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    seeds = [np.argsort(-c, kind="stable").astype(np.int32).tolist() for c in counts.cpu().numpy()]
    ms_ts, out_ts, misses_ts, h2d_ts, codes_ts, _ = run(tiers, service=1, seeds=seeds)
    tiered_line = {"tokens_per_s": meas / (ms_ts * 1e-3), "misses": misses_ts, "status": codes_ts,
                   "slots": f"{tiers[0]}/{tiers[n_layers // 2]}/{tiers[-1]} by thirds of the stack "
                            f"({sum(tiers)} in all, uniform {slots * n_layers})",
                   "seed": "each layer's most-selected experts over the warm-up tokens, resident profiling pass",
                   "bit_identical_vs_resident": bool(torch.equal(out_ts.view(torch.int16),
                                                                 out_res.view(torch.int16)))}
    try:
        ms_copy, out_copy, misses_copy, h2d_copy, codes_copy, wait_ns = run(slots, service=0)
        copy_line = {"tokens_per_s": meas / (ms_copy * 1e-3), "misses": misses_copy, "status": codes_copy,
                     "h2d_gbs": h2d_copy / (ms_copy * 1e-3) / 1e9,
                     "kernel_wait_us_per_miss": wait_ns / 1e3 / max(1, misses_copy),
                     "bit_identical_vs_resident": bool(torch.equal(out_copy.view(torch.int16),
                                                                   out_res.view(torch.int16)))}
    except moe.MoeError as e:
        copy_line = {"error": str(e), "status": [l.stats()[1] for l in st.layers]}
    peak_small = h2d_peak_gbs(torch, synth.PAGE.expert_bytes, 256)
    peak_large = h2d_peak_gbs(torch, 64 << 20, 16)
    hbm_peak, peak_kind = measured_peak()
    step_bytes = n_layers * STEP_BYTES_PER_TOKEN
    res_tps = meas / (ms_res * 1e-3)
    pool_tps = meas / (ms_pool * 1e-3)
    h2d_gbs = h2d_bytes / (ms_pool * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": pool_tps, "unit": UNIT, "n_gpus": 1, "steps": meas, "warmup": warm,
        "ms_per_step": ms_pool / meas, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16+f32 (4-bit weights)", "data": "synthetic",
        "config": {"workload": f"{n_layers}-layer page-scale MoE stack, residual + RMSNorm, 128-slot (25%) "
                               "LRU pool per layer, misses read from pinned host RAM by the kernel after the "
                               "host doorbell; 64 warm-up tokens, then the timed tokens, batch 1",
                   "layers": n_layers, "slots_per_layer": slots},
        "pool": {"tokens_per_s": pool_tps, "service": "sm_pull", "misses": misses, "h2d_bytes": h2d_bytes,
                 "h2d_bytes_per_token": h2d_bytes / meas, "h2d_gbs": h2d_gbs,
                 "h2d_peak_gbs_expert_copies": peak_small, "h2d_peak_gbs_64MB_copies": peak_large,
                 "h2d_frac_of_expert_copy_peak": h2d_gbs / peak_small, "status": codes},
        "pool_tiered_seeded": tiered_line,
        "pool_copy_engine": copy_line,
        "resident_norm_kernel_between_layers": {
            "tokens_per_s": meas / (ms_split * 1e-3),
            "bit_identical_vs_fused": bool(torch.equal(out_split.view(torch.int16), out_res.view(torch.int16)))},
        "resident": {"tokens_per_s": res_tps, "status": codes_res, "roofline": {
            "bound": "hbm", "achieved": step_bytes * res_tps / 1e9, "peak": hbm_peak, "unit": "GB/s",
            "frac": step_bytes * res_tps / 1e9 / hbm_peak, "peak_kind": peak_kind, "bytes_per_token": step_bytes}},
        "bit_identical_pool_vs_resident": identical,
        "setup_s": setup_s,
    }
    print(json.dumps(line), flush=True)
    st.close()

def run_batched(args):
    """Batched decode: calls of T independent tokens (T <= 8: the fused
    kernel; 9..64: route + gate/up + down kernels) through the page-scale
    layer, all experts resident, about 1,000 tokens per step over 8 layer
    replicas round-robin.  Algorithmic bytes of a call: W_r plus the
    distinct experts its T tokens select (counted from the call's routing
    output) plus the shared expert."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_expert_ffn_gemv_gb300 import moe, synth
    T = args.batch
    if not 2 <= T <= 64:
        raise SystemExit("--batch must be 2..64")
    torch.cuda.set_device(0)
    L = synth.make_layer(synth.PAGE, layer=0)
    layers = [moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=T) for _ in range(args.replicas)]
    calls = (args.tokens + T - 1) // T
    ntok = calls * T
    x_host = L_tokens(L, 0, ntok)
    x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_pin = torch.empty_like(x_pin).pin_memory()
    xd = x_pin.to("cuda")
    yd = torch.empty_like(xd)
    idx = torch.empty((ntok, K), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        for c in range(calls):
            sl = slice(c * T, (c + 1) * T)
            layers[c % len(layers)].forward(xd[sl], yd[sl], idx[sl])

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    routed = idx.cpu().numpy().reshape(calls, T * K)
    distinct = [len(np.unique(r)) for r in routed]
    step_bytes = sum(ROUTER_BYTES + (d + 1) * EXPERT_BYTES for d in distinct)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(os.path.join(tempfile.gettempdir(), "bench_batched_clocks.csv"))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with clocks:
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev[1].record(stream)
        torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1])
    with torch.cuda.stream(stream):
        ev[2].record(stream)
        for _ in range(args.steps):
            xd.copy_(x_pin, non_blocking=True)
            graph.replay()
            y_pin.copy_(yd, non_blocking=True)
        ev[3].record(stream)
    torch.cuda.synchronize()
    ms_e2e = ev[2].elapsed_time(ev[3])
    for l in layers:
        _, code = l.stats()
        if code != 0:
            raise RuntimeError(f"layer error {code}")
    peak, peak_kind = measured_peak()
    step_s = ms * 1e-3 / args.steps
    achieved = step_bytes / step_s / 1e9
    fused = T <= 8
    line = {
        "metric": METRIC, "value": ntok / step_s, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16xf16+f32 (4-bit weights)", "data": "synthetic",
        "config": {"workload": f"page-scale MoE layer, batched decode: {calls} calls of {T} independent tokens per "
                               f"step over {len(layers)} layer replicas round-robin, all experts resident",
                   "batch": T, "calls_per_step": calls, "replicas": len(layers),
                   "l2": "inputs larger than L2 (layer replicas round-robin)", "parallelism": "replicas x1"},
        "roofline": {"bound": "hbm", "kernel": "moe_decode_kernel" if fused else "route_kernel + gateup_kernel + "
                     "down_kernel", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "bytes_per_unit": step_bytes / calls, "unit_of_work": "call",
                     "distinct_experts_per_call": sum(distinct) / calls, "traffic": None},
        "e2e": {"value": ntok / (ms_e2e * 1e-3 / args.steps), "unit": UNIT,
                "h2d_bytes_per_step": int(x_pin.numel() * 2), "d2h_bytes_per_step": int(y_pin.numel() * 2)},
        "gpu_launches": calls * (1 if fused else 3) * args.steps,
        "clocks": clocks.summary(0),
    }
    print(json.dumps(line), flush=True)
    for l in layers:
        l.close()


PREFILL_T = 4096
PREFILL_PAIRS = PREFILL_T * (K + 1)                   # routed pairs + shared-expert rows
PREFILL_FLOPS = 2 * PREFILL_PAIRS * 3 * H * I         # gate, up, down: 283.5 GFLOP on the tensor cores
PREFILL_WEIGHT_BYTES = (E + 1) * EXPERT_BYTES + ROUTER_BYTES


def run_prefill(args):
    """One 4,096-token chunk through the page-scale layer per step: router,
    top-k, grouping, gate/up and down grouped GEMMs (tcgen05), combine.
    All experts resident; 0.91 GB of weights per step (> L2)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_expert_ffn_gemv_gb300 import moe, synth
    torch.cuda.set_device(0)
    L = synth.make_layer(synth.PAGE, layer=0)
    layer = moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=PREFILL_T)
    x_host = synth.activations(L.shape, L.index, 0, PREFILL_T, stream=11)
    x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_pin = torch.empty_like(x_pin).pin_memory()
    xd = x_pin.to("cuda")
    yd = torch.empty_like(xd)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            layer.forward(xd, yd, stream=stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(os.path.join(tempfile.gettempdir(), "bench_prefill_clocks.csv"))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with clocks:
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for _ in range(args.steps):
                layer.forward(xd, yd, stream=stream)
            ev[1].record(stream)
        torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1])
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        e[0].record(stream)
        for _ in range(args.steps):
            xd.copy_(x_pin, non_blocking=True)
            layer.forward(xd, yd, stream=stream)
            y_pin.copy_(yd, non_blocking=True)
        e[1].record(stream)
    torch.cuda.synchronize()
    ms_e2e = e[0].elapsed_time(e[1])
    st, code = layer.stats()
    if code != 0:
        raise RuntimeError(f"layer error {code}")
    per_call = ms * 1e-3 / args.steps
    tflops = PREFILL_FLOPS / per_call / 1e12
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    tpeak = float(peaks.get("bf16_tflops", 1900.0))
    hbm_peak, peak_kind = measured_peak()
    line = {
        "metric": "MoE prefill tokens/s (one 4096-token chunk per step); tensor-pipe fraction",
        "value": PREFILL_T * args.steps / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16xf16+f32 (4-bit weights dequantized to f16)", "data": "synthetic",
        "config": {"workload": "page-scale MoE layer prefill chunk: 4096 tokens, H 2048, 512 routed experts "
                               "top-10 + 1 shared, I 512, Zipf(1.1) router bias, all experts resident",
                   "l2": "inputs larger than L2 (0.91 GB of expert weights per step)"},
        "roofline": {"bound": "tensor", "kernel": "whole moe_forward call (11 kernels)", "achieved": tflops,
                     "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                     "peak_kind": "measured bf16 burst (f16 runs at the bf16 rate)",
                     "flops_per_unit": PREFILL_FLOPS, "unit_of_work": "4096-token chunk", "traffic": None,
                     "hbm_frac": PREFILL_WEIGHT_BYTES / per_call / 1e9 / hbm_peak},
        "e2e": {"value": PREFILL_T * args.steps / (ms_e2e * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_pin.numel() * 2), "d2h_bytes_per_step": int(y_pin.numel() * 2)},
        "gpu_launches": 11 * args.steps,  # prep, router, top-k, prefix, scan, pairs, 2 small-chunk + 2 tensor-core GEMMs, combine
        "clocks": clocks.summary(0),
    }
    if args.cpu_sample > 0:
        import oracle
        n = min(args.cpu_sample, 16)
        t0 = time.perf_counter()
        oracle.moe_forward(H, I, E, K, L.W_r, L.bias, L.experts, L.shared, x_host[:n])
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} prefill tokens of the page-scale layer, single-threaded binary64"}
    print(json.dumps(line), flush=True)
    layer.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=32, help="oracle tokens timed for cpu_baseline")
    ap.add_argument("--tokens", type=int, default=TOKENS_PER_STEP)
    ap.add_argument("--workload", default="decode", choices=["decode", "stack", "prefill", "batched"],
                    help="decode: one page-scale layer, batch 1 (default); stack: 48-layer stack with a 25%% "
                         "pool; prefill: one 4096-token chunk; batched: calls of --batch tokens")
    ap.add_argument("--batch", type=int, default=8, help="tokens per call for --workload batched (2..64)")
    ap.add_argument("--layers", type=int, default=48, help="stack depth for --workload stack")
    ap.add_argument("--replicas", type=int, default=REPLICAS,
                    help="decode: identical layer copies cycled round-robin (8 keeps every reuse out of L2)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 256 if args.workload == "stack" else 10
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "stack":
        return run_stack(args)
    if args.workload == "prefill":
        return run_prefill(args)
    if args.workload == "batched":
        return run_batched(args)

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

    L = synth.make_layer(synth.PAGE, layer=0)
    layers = [moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=1, device=local)
              for _ in range(args.replicas)]
    ntok = args.tokens
    x_host = L_tokens(L, 0, ntok)
    x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_pin = torch.empty_like(x_pin).pin_memory()
    xd = x_pin.to("cuda")
    yd = torch.empty_like(xd)
    stream = torch.cuda.Stream()

    def step():
        for t in range(ntok):
            layers[t % len(layers)].forward(xd[t:t + 1], yd[t:t + 1])

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()

    def barrier():
        if pg:
            pg.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    barrier()
    clocks = ClockSampler(os.path.join(tempfile.gettempdir(), f"bench_clocks_{rank}.csv"))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clocks:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        barrier()
    ms = ev0.elapsed_time(ev1)
    # ---- end to end through the public API: H2D x, the forwards, D2H y
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            xd.copy_(x_pin, non_blocking=True)
            graph.replay()
            y_pin.copy_(yd, non_blocking=True)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            xd.copy_(x_pin, non_blocking=True)
            graph.replay()
            y_pin.copy_(yd, non_blocking=True)
        e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    for l in layers:
        s, code = l.stats()
        if code != 0:
            raise RuntimeError(f"layer error {code}")
    ms, ms_e2e = max_over_ranks([ms, ms_e2e], pg, device="cuda")
    if rank != 0:
        pg.destroy_process_group() if pg else None
        return
    tokens = ntok * args.steps * ws
    value = whole_job_rate(ntok * args.steps, ws, ms)
    per_token_s = (ms * 1e-3) / (ntok * args.steps)
    peak, peak_kind = measured_peak()
    achieved = STEP_BYTES_PER_TOKEN / per_token_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16+f32 (4-bit weights)", "data": "synthetic",
        "config": {"workload": WORKLOAD.format(tokens=ntok, replicas=len(layers)), "tokens_per_step": ntok,
                   "replicas": len(layers),
                   "l2": f"inputs larger than L2 ({len(layers)} layer replicas, "
                         f"{len(layers) * E * EXPERT_BYTES / 2**30:.2f} GiB of expert weights, round-robin)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "kernel": "moe_decode_kernel (fused route + hit check + gate/up + down)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "bytes_per_unit": STEP_BYTES_PER_TOKEN, "unit_of_work": "token",
                     "traffic": recorded_traffic()},
        "e2e": {"value": whole_job_rate(ntok * args.steps, ws, ms_e2e), "unit": UNIT,
                "h2d_bytes_per_step": int(x_pin.numel() * 2),
                "d2h_bytes_per_step": int(y_pin.numel() * 2)},
        "gpu_launches": ntok * args.steps,  # one fused kernel per token (T = 1)
        "clocks": clocks.summary(local),
    }
    if ws == 1 and args.cpu_sample > 0:
        line["cpu_baseline"] = cpu_baseline(L, args.cpu_sample)
    print(json.dumps(line), flush=True)
    for l in layers:
        l.close()
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
