#!/usr/bin/env python
"""Benchmark of the MoE expert-layer hot path on one or more GPUs (one process per GPU).

Default run: the headline workload -- prefill with token-dimension bucketing: the W4A16
MXFP4 layer (hidden 2880, intermediate 2880, 128 experts, top-4, bf16 biases) over 16
requests of 3277..4096 tokens (58,879 tokens, padded to the bucket of 61,440 rows) -- timed
for exactly --steps steps, and after it every other workload, each with its own line in the
``workloads`` map: the tiny layer, the 64-token decode layer, the tiny-M bf16 decode layer
at M = 1, 7, 14, 21, 28, the MXFP8 grouped GEMMs + weight gradients, the MXFP8 layer and the
per-token FP8 grouped GEMM.  One step of a layer workload = bucket padding of the token
dimension (W4A16 only), routing + alignment, grouped GEMM1 + bias + SwiGLU, grouped GEMM2 +
bias * routing weight, and the top-k combine, through the C ABI.

Prints one JSON line.  value = tokens/s over all ranks with inputs resident in HBM;
e2e = the same metric with the step's inputs copied from pinned host memory and the
output copied back inside the timed region; roofline = the dominant kernel's algorithmic
bytes (or flops) / its CUDA-event time against the measured HBM copy bandwidth (or bf16
tensor peak); cpu_baseline = the float64 oracle timed on a bounded sample on this host, with
every core available to its BLAS and with one thread.

``--workload NAME`` runs one workload alone (smaller cases for profiling: --tokens,
--experts).  ``--impl reference`` times the oracle alone (the reference arm), on rank 0.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer useful TFLOP/s & tokens/s; % of GB300 block-scaled TC / HBM roofline"
L2_BYTES = 129 * 1024 * 1024

# DRAM traffic (read + write bytes) of one launch of the dominant kernel (for the weight
# gradient: every launch of one moe_wgrad call), from an ncu capture of the same command,
# valid while the kernel source hashes the same; otherwise reported as null.
TRAFFIC = {
    "decode_tc.cu:gemm1@decode_mxfp4": {
        "src": "dfafccfa25145f06", "bytes": 1024535552 + 5261568},
    # both launches of the call: the main pass and the (empty) exact-scale pass
    "prefill_ts.cu:gemm1@prefill_mxfp4": {
        "src": "40b9e45121f051d6", "bytes": 2599493120 + 1443217152 + 68608},
    # the dW1 call: the two slot-order copies, the expert ranges and the tensor-core kernel
    "wgrad_tc.cu:wgrad_dW1@mxfp8_wgrad": {
        "src": "76867c344737658b", "bytes": 37354372864},
}


def e2e_pipelined(L, T, xh, lh, yh, x, lg, y, stream, n):
    """n layer steps with the inputs copied in from pinned host memory and the output copied
    out every step, overlapped: inputs of step i + 1 (copy-in stream) and the output of step
    i - 1 (copy-out stream) move while step i computes; two device buffers of each.  Returns
    the milliseconds from before the first copy to after the last output copy."""
    import torch

    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    xd = [torch.empty_like(x), torch.empty_like(x)]
    ld = [torch.empty_like(lg), torch.empty_like(lg)]
    yd = [torch.empty_like(y), torch.empty_like(y)]
    ev = lambda: torch.cuda.Event()
    ready, done, out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(count):
        for i in range(count):
            b = i % 2
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(done[b])       # step i - 2 has read this input buffer
                xd[b].copy_(xh, non_blocking=True)
                ld[b].copy_(lh, non_blocking=True)
                ready[b].record(cin)
            stream.wait_event(ready[b])
            if i >= 2:
                stream.wait_event(out[b])         # step i - 2's output has left this buffer
            L.step(xd[b], ld[b], T, yd[b])
            done[b].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(done[b])
                yh.copy_(yd[b], non_blocking=True)
                out[b].record(cout)
        stream.wait_stream(cout)

    run(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cin.wait_stream(stream)
    run(n)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    choices=["all", "decode_mxfp4", "decode_bf16", "prefill_mxfp4", "tiny", "mxfp8_wgrad",
                             "pertoken_fp8", "mxfp8_layer"],
                    help="all (default): the prefill headline plus every other workload")
    ap.add_argument("--m", type=int, default=28, help="tokens for decode_bf16")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the token count (smaller cases for profiling)")
    ap.add_argument("--experts", type=int, default=None,
                    help="experts of the mxfp8_wgrad workload (a smaller case for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-dir", default=None,
                    help="directory for the raw clock samples of the timed region")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of replays of the step's CUDA graph")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sample-tokens", type=int, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


HEADLINE = "prefill_mxfp4"
# the other workloads of the default run, each with its own entry of the ``workloads`` map
MAP_WORKLOADS = ["tiny", "decode_mxfp4"] + [f"decode_bf16_M{m}" for m in (1, 7, 14, 21, 28)] + \
    ["mxfp8_wgrad", "mxfp8_layer", "pertoken_fp8"]
# workloads whose expert weights would fit twice in the 129 MB L2: a 512 MB buffer is written
# between their steps, outside the timed intervals
L2_FLUSHED = {"tiny", "decode_bf16_M1"}
DEFAULT_STEPS = {"decode_mxfp4": (2000, 50), "decode_bf16": (4000, 100),
                 "prefill_mxfp4": (10, 3), "tiny": (4000, 100), "mxfp8_wgrad": (3, 3),
                 "pertoken_fp8": (20, 3), "mxfp8_layer": (5, 3)}
ORACLE_SAMPLE = {"decode_mxfp4": 8, "decode_bf16": 28, "prefill_mxfp4": 24, "tiny": 64,
                 "mxfp8_wgrad": 512, "pertoken_fp8": 8192, "mxfp8_layer": 4096}
# The per-token FP8 grouped GEMM workload: the GEMM1 shape of the MXFP8 workload (256 experts,
# K = 7168 -> N = 4096, T = 8192 tokens at top-8, Zipf(1.1) routing), rows grouped by expert.
PERTOKEN = {"T": 8192, "E": 256, "N": 4096, "K": 7168, "k": 8, "seed": 9}


def workload(name, m):
    import synth
    if name == "decode_mxfp4":
        return synth.DECODE_MXFP4
    if name == "decode_bf16":
        return synth.decode_bf16_workload(m)
    if name == "prefill_mxfp4":
        return synth.prefill_workload()
    return synth.TINY


def describe(w, rows):
    d = {"workload": f"{w.name}: T={w.T} tokens, hidden {w.K}, intermediate {w.I}, "
                     f"{w.E} experts, top-{w.k}, {w.quant}{', bf16 biases' if w.bias else ''}",
         "T": w.T, "T_rows": rows, "hidden": w.K, "intermediate": w.I, "experts": w.E,
         "top_k": w.k, "quant": w.quant, "block_m": 128}
    return d


def useful_flops(w):
    P = w.T * w.k
    return 2.0 * P * w.K * 2 * w.I + 2.0 * P * w.I * w.K


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "mixture_experts_grouped_align_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------------------ ranks

def barrier(world):
    """Every rank reaches this point (one process per GPU; nothing to do alone)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """The largest of every rank's x (the slowest rank's time); x itself when alone."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world, units_per_rank, ms):
    """Whole-job rate: the units every rank processed over the slowest rank's time (per s)."""
    return world * units_per_rank / (ms * 1e-3)


# ------------------------------------------------------------------------------ oracle

def oracle_sample_mxfp8(n_tok):
    """The oracle on a bounded sample of the MXFP8 GEMM + wgrad workload: n_tok tokens of
    top-8 routing over 2 experts' worth of freshly drawn weights (same shapes and
    recipe), both grouped GEMMs and both weight gradients of those experts."""
    import numpy as np
    import synth
    from oracle import formats, layer, wgrad
    w = synth.MXFP8_WGRAD
    rng = np.random.default_rng(4)
    E, K, I, k = 2, w.K, w.I, 1
    T = n_tok
    ids = (np.arange(T) % E).astype(np.int32)[:, None]
    se = synth.scale_exp_for_std(w.weight_std)
    xc, xs = synth.gen_mx_e4m3(rng, (T, K))
    ac, as_ = synth.gen_mx_e4m3(rng, (T, I))
    w1c, w1s = synth.gen_mx_e4m3(rng, (E, 2 * I, K), se)
    w2c, w2s = synth.gen_mx_e4m3(rng, (E, K, I), se)
    g1 = synth.to_bf16_bits(rng.standard_normal((T, 2 * I)).astype(np.float32))
    g2 = synth.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    xb = synth.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    hb = synth.to_bf16_bits(rng.standard_normal((T, I)).astype(np.float32))
    t0 = time.perf_counter()
    A1 = formats.dequant_mxfp8(xc, xs)
    A2 = formats.dequant_mxfp8(ac, as_)
    layer.grouped_gemm(A1, ids, lambda e: (formats.dequant_mxfp8(w1c[e], w1s[e]), None), False)
    layer.grouped_gemm(A2, ids, lambda e: (formats.dequant_mxfp8(w2c[e], w2s[e]), None), True)
    wgrad.moe_wgrad(formats.bf16_decode(g1), formats.bf16_decode(xb), ids, E, False)
    wgrad.moe_wgrad(formats.bf16_decode(g2), formats.bf16_decode(hb), ids, E, True)
    # the full workload has 8 pairs per token
    return time.perf_counter() - t0, T / 8.0


def oracle_sample_pertoken(n_rows):
    """The oracle on a bounded sample of the per-token FP8 workload: n_rows rows of one
    expert (freshly drawn E4M3 codes and scales of the same shapes).  Returns seconds and
    the tokens the rows stand for (top-8: 8 rows per token)."""
    import numpy as np
    from oracle import per_token
    c = PERTOKEN
    rng = np.random.default_rng(c["seed"])
    a = rng.integers(0, 126, size=(n_rows, c["K"]), dtype=np.uint8) | (rng.integers(0, 2, size=(n_rows, c["K"]), dtype=np.uint8) << 7)
    w = rng.integers(0, 126, size=(1, c["N"], c["K"]), dtype=np.uint8) | (rng.integers(0, 2, size=(1, c["N"], c["K"]), dtype=np.uint8) << 7)
    sa = rng.uniform(2.0 ** -10, 2.0 ** -8, n_rows)
    sw = rng.uniform(2.0 ** -10, 2.0 ** -8, 1)
    t0 = time.perf_counter()
    per_token.gemm_per_token(a, sa, w, sw, None, np.array([n_rows]))
    return time.perf_counter() - t0, n_rows / float(c["k"])


def oracle_sample_mxfp8_layer(n_pairs):
    """The oracle MXFP8 layer on a bounded sample: n_pairs token-expert pairs over 2 experts'
    worth of freshly drawn weights of the workload's shapes (top-1 here; the workload has 8
    pairs per token)."""
    import numpy as np
    import synth
    from oracle import formats, layer
    w = synth.MXFP8_WGRAD
    rng = np.random.default_rng(5)
    E, K, I = 2, w.K, w.I
    se = synth.scale_exp_for_std(w.weight_std)
    xc, xs = synth.gen_mx_e4m3(rng, (n_pairs, K))
    w1c, w1s = synth.gen_mx_e4m3(rng, (E, 2 * I, K), se)
    w2c, w2s = synth.gen_mx_e4m3(rng, (E, K, I), se)
    ids = (np.arange(n_pairs) % E).astype(np.int32)[:, None]
    wt = np.ones((n_pairs, 1), dtype=np.float32)
    t0 = time.perf_counter()
    W = layer.ExpertWeights("mxfp8", w1c, w1s, None, w2c, w2s, None)
    layer.moe_layer(formats.dequant_mxfp8(xc, xs), ids, wt, W)
    return time.perf_counter() - t0, n_pairs / 8.0


def oracle_sample(name, m, n_tok):
    """Times the float64 oracle on the first n_tok tokens of the workload (this process
    was started with one BLAS / OpenMP thread).  Returns seconds."""
    if name == "mxfp8_layer":
        return oracle_sample_mxfp8_layer(n_tok)
    if name == "mxfp8_wgrad":
        return oracle_sample_mxfp8(n_tok)
    if name == "pertoken_fp8":
        return oracle_sample_pertoken(n_tok)
    import synth
    from oracle import formats, layer, route
    w = workload(name, m)
    lay = synth.make_layer(w, T=w.T if name != "prefill_mxfp4" else 4096)
    W = layer.ExpertWeights(w.quant, lay["w1"], lay["w1_scale"], lay["b1"], lay["w2"],
                            lay["w2_scale"], lay["b2"])
    n = min(n_tok, lay["x"].shape[0])
    t0 = time.perf_counter()
    x = formats.bf16_decode(lay["x"][:n])
    ids, wt = route.route(lay["logits"][:n], w.k)
    layer.moe_layer(x, ids, wt, W)
    return time.perf_counter() - t0, n


def run_oracle_subprocess(name, m, n_tok, threads=1, timeout=900):
    """Runs oracle_sample in a fresh process whose BLAS / OpenMP pools have ``threads``
    threads (and no GPU); returns {"seconds", "tokens"}."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", name,
           "--m", str(m), "--sample-tokens", str(n_tok)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:  # pragma: no cover
        return os.cpu_count() or 1


def workload_name(base, m):
    return f"decode_bf16_M{m}" if base == "decode_bf16" else base


def layer_config(w, rows, world, flush):
    """The ``config`` of a layer workload: its shapes and how the L2 is kept cold (the same
    dict for both arms of the benchmark)."""
    return dict(describe(w, rows),
                l2=("L2 flushed between steps (a 512 MB buffer written outside the timed intervals): the "
                    "step's expert weights would fit in the 129 MB L2" if flush else
                    "inputs larger than L2: the expert weights streamed per step exceed the 129 MB L2"),
                parallelism=f"replicas x{world}")


# ------------------------------------------------------------------------------ clocks

def clocks_csv(args, rank):
    """Where the raw nvidia-smi samples of the timed region go (--clocks-dir, else the
    system temporary directory); the JSON line carries their summary."""
    d = args.clocks_dir or tempfile.gettempdir()
    os.makedirs(d, exist_ok=True)
    return os.path.join(d, f"clocks_rank{rank}.csv")


class ClockSampler:
    def __init__(self, path):
        self.path = path
        self.proc = None

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, dev_index):
        if not self.proc:
            return {"samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            rows = [[p.strip() for p in line.split(",")] for line in f]
        rows = [r for r in rows if len(r) >= 9]
        idx = {r[0] for r in rows}
        want = str(dev_index) if str(dev_index) in idx else (sorted(idx)[0] if idx else None)
        if True:
            for parts in rows:
                if parts[0] != want:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, v in zip(names[1:], parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return {"samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ ours

def bench_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import mixture_experts_grouped_align_gb300 as moe
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    import synth

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    moe.build()
    moe.load()
    w = workload(args.workload, args.m)
    if args.tokens:
        import dataclasses
        w = dataclasses.replace(w, T=args.tokens, name=f"{w.name}_T{args.tokens}")
    steps, warmup = DEFAULT_STEPS[args.workload]
    steps = args.steps if args.steps is not None else steps
    warmup = max(3, args.warmup if args.warmup is not None else warmup)
    lay = synth.make_layer(w)

    def d(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    L = DeviceLayer(w.quant, w.E, w.K, w.I, w.k, d(lay["w1"]), d(lay["w1_scale"]), d(lay["b1"]),
                    d(lay["w2"]), d(lay["w2_scale"]), d(lay["b2"]), max_rows=w.T, device=dev)
    T = w.T
    x = d(lay["x"])
    lg = d(lay["logits"])
    y = torch.empty((T, w.K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    # one step to learn the routing (same every step) for the byte counts
    rows = L.step(x, lg, T, y)
    torch.cuda.synchronize()
    if int(L.status[0]) != 0:
        raise RuntimeError(f"device status {int(L.status[0])}")
    eoff = L.expert_offsets[:w.E + 1].cpu().numpy()
    touched = int(np.count_nonzero(np.diff(eoff)))
    P_rows = rows * w.k

    def wbytes(N, Kin):
        if w.quant == "mxfp4":
            return N * Kin // 2 + N * Kin // 32
        return N * Kin * 2
    bias_b = (2 * w.I * 2) if w.bias else 0
    gemm1_bytes = touched * (wbytes(2 * w.I, w.K) + bias_b) + rows * w.K * 2 + P_rows * w.I * 2
    gemm2_bytes = touched * (wbytes(w.K, w.I) + (w.K * 2 if w.bias else 0)) + P_rows * w.I * 2 + P_rows * w.K * 4
    step_weight_bytes = touched * (wbytes(2 * w.I, w.K) + wbytes(w.K, w.I))

    def step(evs=None):
        return L.step(x, lg, T, y, events=evs)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # per-kernel split: eager steps with the library's CUDA events around its launches
    n_ev = max(1, min(steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]
    for es in evs:  # torch creates the CUDA event on its first record
        for e in es:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(n_ev):
        step(evs[i])
    torch.cuda.synchronize()
    g1 = sum(e[0].elapsed_time(e[1]) for e in evs) / n_ev
    g2 = sum(e[1].elapsed_time(e[2]) for e in evs) / n_ev
    cb = sum(e[2].elapsed_time(e[3]) for e in evs) / n_ev
    # the timed region: the whole step (every kernel, every step) replayed from one CUDA graph,
    # which removes the host launch gaps between its kernels; --no-graph launches eagerly
    graph = None
    if not args.no_graph:
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            L.step(x, lg, T, y, stream=cs)
        stream.wait_stream(cs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            L.step(x, lg, T, y, stream=cs)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(clocks_csv(args, rank))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    cur = torch.cuda.current_stream()
    # a step whose weights fit twice in L2 would be served from L2 by the previous step: such
    # workloads write a 512 MB buffer between steps, outside the timed intervals
    flush = workload_name(args.workload, args.m) in L2_FLUSHED and not args.tokens
    if flush:
        scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            scrub.fill_(i & 0xff)
            pairs[i][0].record(cur)
            if graph is not None:
                graph.replay()
            else:
                step()
            pairs[i][1].record(cur)
        torch.cuda.synchronize()
    else:
        t_start.record(cur)
        for i in range(steps):
            if graph is not None:
                graph.replay()
            else:
                step()
        t_end.record(cur)
        torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop(local_rank)
    ms = sum(a.elapsed_time(b) for a, b in pairs) if flush else t_start.elapsed_time(t_end)
    if int(L.status[0]) != 0:
        raise RuntimeError(f"device status {int(L.status[0])}")
    ms = max_over_ranks(ms, world, dev)

    # end to end: pinned host inputs in, output back out, inside the timed region.  As a
    # serving loop would run it: the next step's inputs go up on a copy stream and the last
    # step's output comes down on another while this step computes (two buffers each).
    xh = torch.empty_like(x, device="cpu").pin_memory()
    xh.copy_(x.cpu())
    lh = torch.empty_like(lg, device="cpu").pin_memory()
    lh.copy_(lg.cpu())
    yh = torch.empty_like(y, device="cpu").pin_memory()
    e2e_steps = max(1, min(steps, 500))
    e2e_ms = e2e_pipelined(L, T, xh, lh, yh, x, lg, y, stream, e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    if rank != 0:
        return None
    hbm, bf16, src = peaks()
    dominant = "gemm1" if g1 >= g2 else "gemm2"
    dom_bytes, dom_ms = (gemm1_bytes, g1) if dominant == "gemm1" else (gemm2_bytes, g2)
    tensor_path = rows > 256  # row counts above the bucket value 256 run the tcgen05 kernels
    # the W4A16 layer above 256 rows runs the kernel with the decoded weights in tensor memory;
    # up to 256 rows the MXFP4 SwiGLU layer runs the block-scaled kernel that reads the E2M1
    # codes as stored (K and I multiples of 64, at most 3072), other layers weight streaming
    block_scaled = (not tensor_path and w.quant == "mxfp4" and w.activation == "swiglu"
                    and w.K % 64 == 0 and w.I % 64 == 0 and w.K <= 3072 and w.I <= 3072)
    if tensor_path:
        kernel_file = "prefill_ts.cu" if w.quant == "mxfp4" else "prefill_gemm.cu"
    else:
        kernel_file = "decode_tc.cu" if block_scaled else "decode_gemm.cu"
    kernel_name = kernel_file[:-3] + f" ({dominant})"
    key = f"{kernel_file}:{dominant}@{w.name}"
    tr = TRAFFIC.get(key)
    traffic = tr["bytes"] if tr and tr.get("src") == src_hash(kernel_file) else None
    if tensor_path:
        # useful (unpadded) flops of the dominant GEMM against the dense f16/bf16 peak
        # (f16 and bf16 tensor rates are equal)
        P_real = w.T * w.k
        dom_flops = 2.0 * P_real * w.K * 2 * w.I if dominant == "gemm1" else 2.0 * P_real * w.I * w.K
        achieved = dom_flops / (dom_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": kernel_name, "achieved": achieved, "peak": bf16,
                    "unit": "TFLOP/s", "frac": achieved / bf16, "traffic": traffic,
                    "algorithmic_flops": dom_flops, "peak_source": f"{src} (bf16_tflops)"}
    else:
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": achieved, "peak": hbm,
                    "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                    "algorithmic_bytes": dom_bytes, "peak_source": f"{src} (hbm_gbs)"}
    ms_step = ms / steps
    line = {
        "metric": METRIC,
        "value": aggregate_rate(world, T * steps, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f16 tcgen05 mma -> f32" if tensor_path else
                  ("e2m1 x e2m1 digit planes, block-scaled tcgen05 mma -> f32" if block_scaled else "f16 mma -> f32"))
                 if w.quant != "bf16" else "bf16 mma -> f32",
        "data": "synthetic (seeded PCG64 inputs, random-init weights)",
        "config": layer_config(w, rows, world, flush),
        "timing": ("replays of one CUDA graph of the whole step (every kernel of the step runs each replay); "
                   "the per-kernel split comes from eager steps with the library's CUDA events"
                   if graph is not None else "eager launches"),
        "useful_tflops": world * useful_flops(w) * steps / (ms * 1e-3) / 1e12,
        "layer_latency_us": ms_step * 1e3,
        "kernel_ms": {"gemm1_swiglu": g1, "gemm2_weighted": g2, "combine": cb,
                      "route_align_pad_x16_and_gaps": ms_step - g1 - g2 - cb},
        "experts_touched": touched,
        "roofline": roofline,
        "step_roofline": {"bytes": step_weight_bytes, "achieved_gbs": step_weight_bytes / (ms_step * 1e-3) / 1e9,
                          "frac": step_weight_bytes / (ms_step * 1e-3) / 1e9 / hbm},
        "e2e": {"value": aggregate_rate(world, T * e2e_steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * 2 + lg.numel() * 4,
                "d2h_bytes_per_step": y.numel() * 2, "steps": e2e_steps},
        "gpu_launches": steps * launches_per_step(w, rows),
        "clocks": ck,
    }
    return line


def bench_mxfp8_wgrad(args, rank, world, local_rank):
    """256 experts, hidden 7168, intermediate 2048, top-8, T=8192, Zipf routing: MXFP8
    grouped GEMM1 (per token, K=7168 -> 4096) and GEMM2 (per pair, K=2048 -> 7168), then
    the deterministic weight gradients dW1 [256, 4096, 7168] and dW2 [256, 7168, 2048]."""
    import numpy as np
    import torch

    import mixture_experts_grouped_align_gb300 as moe
    import synth

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    moe.build()
    moe.load()
    steps, warmup = DEFAULT_STEPS["mxfp8_wgrad"]
    steps = args.steps if args.steps is not None else steps
    warmup = max(3, args.warmup if args.warmup is not None else warmup)
    kw = {} if not args.tokens else {"T": args.tokens}
    if args.experts:
        kw["E"] = args.experts
    g = synth.make_mxfp8_gemm_wgrad(device=dev, **kw)
    T, E, K, I, k, P = g["T"], g["E"], g["K"], g["I"], g["k"], g["P"]
    bm = 128
    cap, capb = moe.moe_align_capacity(P, E, bm)
    ids = torch.from_numpy(g["topk_ids"]).to(dev)
    srt = torch.empty(cap, dtype=torch.int32, device=dev)
    eid = torch.empty(capb, dtype=torch.int32, device=dev)
    ntpp = torch.empty(4, dtype=torch.int32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    moe.moe_align(None, ids, None, T, k, E, bm, srt, cap, eid, ntpp, None, moe.Ctx(dev_status=status))
    out1 = torch.empty((P, 2 * I), dtype=torch.bfloat16, device=dev)
    out2 = torch.empty((P, K), dtype=torch.bfloat16, device=dev)
    dW1 = torch.empty((E, 2 * I, K), dtype=torch.float32, device=dev)
    dW2 = torch.empty((E, K, I), dtype=torch.float32, device=dev)
    # the weight gradients' slot-ordered copies of grad and input (one workspace, used in turn)
    wg_ws = torch.empty(max(moe.moe_wgrad_workspace_size(E, 2 * I, K, bm, cap, 0),
                            moe.moe_wgrad_workspace_size(E, K, I, bm, cap, 0), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    def step(evs=None):
        c = [moe.Ctx(dev_status=status, events=None if evs is None else evs[i], workspace=wg_ws if i >= 2 else None)
             for i in range(4)]
        moe.moe_grouped_gemm("mxfp8", E, 2 * I, K, g["x_codes"], g["x_scale"], 0, g["w1"], g["w1_scale"],
                             None, T, k, srt, eid, ntpp, bm, cap, out1, c[0])
        moe.moe_grouped_gemm("mxfp8", E, K, I, g["a2_codes"], g["a2_scale"], 1, g["w2"], g["w2_scale"],
                             None, T, k, srt, eid, ntpp, bm, cap, out2, c[1])
        moe.moe_wgrad(g["grad1"], g["x_bf16"], 0, T, k, E, 2 * I, K, srt, eid, ntpp, bm, cap, dW1, 0, c[2])
        moe.moe_wgrad(g["grad2"], g["h_bf16"], 1, T, k, E, K, I, srt, eid, ntpp, bm, cap, dW2, 0, c[3])

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if int(status[0]) != 0:
        raise RuntimeError(f"device status {int(status[0])}")
    evs = [[[ev(), ev()] for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(clocks_csv(args, rank))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop(local_rank)
    ms = t0.elapsed_time(t1)
    kms = [sum(e[j][0].elapsed_time(e[j][1]) for e in evs) / steps for j in range(4)]
    ms = max_over_ranks(ms, world, dev)
    # end to end: the step's activations and output gradients from pinned host memory,
    # the GEMM outputs back to the host; weights and dW stay resident
    ins = ["x_codes", "x_scale", "a2_codes", "a2_scale", "grad1", "grad2", "x_bf16", "h_bf16"]
    host = {n: torch.empty_like(g[n], device="cpu").pin_memory() for n in ins}
    for n in ins:
        host[n].copy_(g[n].cpu())
    o1h = torch.empty_like(out1, device="cpu").pin_memory()
    o2h = torch.empty_like(out2, device="cpu").pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(steps, 3))
    e0.record(stream)
    for _ in range(e2e_steps):
        for n in ins:
            g[n].copy_(host[n], non_blocking=True)
        step()
        o1h.copy_(out1, non_blocking=True)
        o2h.copy_(out2, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return None
    hbm, bf16, src = peaks()
    f_gemm1 = 2.0 * P * K * 2 * I
    f_gemm2 = 2.0 * P * I * K
    names = ["gemm1_mxfp8", "gemm2_mxfp8", "wgrad_dW1", "wgrad_dW2"]
    dw_bytes = [None, None, E * 2 * I * K * 4 + P * 2 * I * 2 + T * K * 2, E * K * I * 4 + P * K * 2 + P * I * 2]
    dom = int(np.argmax(kms))
    if dom >= 2:
        achieved = dw_bytes[dom] / (kms[dom] * 1e-3) / 1e9
        tr = TRAFFIC.get(f"wgrad_tc.cu:{names[dom]}@mxfp8_wgrad")
        traffic = tr["bytes"] if tr and tr.get("src") == src_hash("wgrad_tc.cu", "elementwise.cu") else None
        roofline = {"bound": "hbm", "kernel": f"wgrad ({names[dom]})", "achieved": achieved, "peak": hbm,
                    "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                    "algorithmic_bytes": dw_bytes[dom], "peak_source": f"{src} (hbm_gbs)"}
    else:
        # E4M3 x E4M3 block-scaled MMA: the measured bf16 peak times the nominal 2x of fp8
        fl = f_gemm1 if dom == 0 else f_gemm2
        achieved = fl / (kms[dom] * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": f"mx8_gemm ({names[dom]})", "achieved": achieved,
                    "peak": 2 * bf16, "unit": "TFLOP/s", "frac": achieved / (2 * bf16), "traffic": None,
                    "algorithmic_flops": fl,
                    "peak_source": f"{src} (bf16_tflops x 2, the nominal fp8/bf16 dense ratio)"}
    h2d = sum(host[n].numel() * host[n].element_size() for n in ins)
    line = {
        "metric": METRIC, "value": aggregate_rate(world, T * steps, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 block-scaled tcgen05 mma (GEMMs), bf16 tcgen05 mma (wgrad) -> f32",
        "data": "synthetic (seeded inputs drawn on the device, random-init weights)",
        "config": {"workload": f"mxfp8_wgrad: T={T} tokens, hidden {K}, intermediate {I}, {E} experts, "
                               f"top-{k}, Zipf(1.1) routing, MXFP8 GEMM1+GEMM2, dW1+dW2 fp32",
                   "T": T, "experts": E, "hidden": K, "intermediate": I, "top_k": k, "block_m": bm,
                   "l2": "inputs larger than L2: 11.3 GB of MXFP8 weights and 45 GB of dW per step",
                   "parallelism": f"replicas x{world}"},
        "useful_tflops": world * 2 * (f_gemm1 + f_gemm2) * steps / (ms * 1e-3) / 1e12,
        "kernel_ms": dict(zip(names, kms)),
        "roofline": roofline,
        "e2e": {"value": aggregate_rate(world, T * e2e_steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out1.numel() * 2 + out2.numel() * 2,
                "steps": e2e_steps},
        "gpu_launches": steps * 4,
        "clocks": ck,
    }
    return line


def bench_pertoken(args, rank, world, local_rank):
    """One per-token FP8 grouped GEMM over group sizes: 256 experts, K = 7168 -> N = 4096,
    65,536 rows (8192 tokens at top-8, Zipf(1.1) routing with cold experts), E4M3 operands
    with one scale per row and one per expert."""
    import numpy as np
    import torch

    import mixture_experts_grouped_align_gb300 as moe
    import synth

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    moe.build()
    moe.load()
    c = PERTOKEN
    steps, warmup = DEFAULT_STEPS["pertoken_fp8"]
    steps = args.steps if args.steps is not None else steps
    warmup = max(3, args.warmup if args.warmup is not None else warmup)
    T = args.tokens or c["T"]
    E, N, K, k = (args.experts or c["E"]), c["N"], c["K"], c["k"]
    rng = np.random.default_rng(c["seed"])
    ids, _ = synth.zipf_topk_ids(rng, T, E, k, n_cold=min(16, E // 4))
    gs = np.bincount(ids.reshape(-1), minlength=E).astype(np.int32)
    M = int(gs.sum())
    # E4M3 codes of N(0, 64^2) values (truncated at 448) for activations and weights, with one
    # scale per row drawn uniformly in [2^-7, 2^-5] and one per expert in [2^-13, 2^-11]
    # (input preparation, outside the timed region)
    gen = torch.Generator(device=dev)
    gen.manual_seed(c["seed"])

    def codes(shape):
        v = torch.randn(shape, device=dev, generator=gen) * 64.0
        return v.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)

    a = codes((M, K))
    a_scale = torch.rand(M, device=dev, generator=gen) * (2.0 ** -5 - 2.0 ** -7) + 2.0 ** -7
    w = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
    for e0 in range(0, E, 16):
        w[e0:e0 + 16] = codes((min(16, E - e0), N, K))
    w_scale = (torch.rand(E, device=dev, generator=gen) * (2.0 ** -11 - 2.0 ** -13) + 2.0 ** -13).float()
    a_scale = a_scale.float().contiguous()
    gsd = torch.from_numpy(gs).to(dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        moe.moe_gemm_per_token(E, N, K, a, a_scale, w, w_scale, None, gsd, M, out,
                               moe.Ctx(dev_status=status, events=evs))

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if int(status[0]) != 0:
        raise RuntimeError(f"device status {int(status[0])}")
    evs = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(steps)]
    for pair in evs:  # a torch event has a CUDA event only once it has been recorded
        for e_ in pair:
            e_.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(clocks_csv(args, rank))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop(local_rank)
    ms = t0.elapsed_time(t1)
    kms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    ms = max_over_ranks(ms, world, dev)
    # end to end: activations, their scales and the group sizes from pinned host memory, the
    # output back to the host; weights stay resident
    ins = [a, a_scale, gsd]
    host = [t.cpu().pin_memory() for t in ins]
    oh = torch.empty_like(out, device="cpu").pin_memory()
    e2e_steps = max(1, min(steps, 3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for d_, h_ in zip(ins, host):
            d_.copy_(h_, non_blocking=True)
        step()
        oh.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return None
    hbm, bf16, src = peaks()
    fl = 2.0 * M * N * K
    achieved = fl / (kms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "pertoken_gemm", "achieved": achieved, "peak": 2 * bf16,
                "unit": "TFLOP/s", "frac": achieved / (2 * bf16), "traffic": None, "algorithmic_flops": fl,
                "peak_source": f"{src} (bf16_tflops x 2, the nominal fp8/bf16 dense ratio)"}
    h2d = sum(t.numel() * t.element_size() for t in host)
    return {
        "metric": METRIC, "value": aggregate_rate(world, T * steps, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 tcgen05 mma -> f32, scales after the dot",
        "data": "synthetic (per-token E4M3 quantisation of N(0,1) activations drawn on the device, "
                "random-init weights)",
        "config": {"workload": f"pertoken_fp8: T={T} tokens, top-{k}, {M} rows grouped by expert, "
                               f"{E} experts, K={K} -> N={N}, Zipf(1.1) routing",
                   "T": T, "rows": M, "experts": E, "N": N, "K": K, "top_k": k,
                   "l2": f"inputs larger than L2: {E * N * K / 1e9:.1f} GB of E4M3 weights and "
                         f"{M * K / 1e9:.2f} GB of activations per step",
                   "parallelism": f"replicas x{world}"},
        "useful_tflops": world * fl * steps / (ms * 1e-3) / 1e12,
        "kernel_ms": {"gemm_per_token": kms},
        "roofline": roofline,
        "e2e": {"value": aggregate_rate(world, T * e2e_steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out.numel() * 2, "steps": e2e_steps},
        "gpu_launches": steps,
        "clocks": ck,
    }


def bench_mxfp8_layer(args, rank, world, local_rank):
    """The whole MXFP8 layer through moe_forward on the MXFP8 workload's shapes (256 experts,
    hidden 7168, intermediate 2048, top-8, T = 8192, Zipf(1.1) routing with the routing
    weights uniform 1/8): GEMM1 + SwiGLU with h quantised to MXFP8 in the epilogue, GEMM2,
    combine."""
    import numpy as np
    import torch

    import mixture_experts_grouped_align_gb300 as moe
    import synth

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    moe.build()
    moe.load()
    steps, warmup = DEFAULT_STEPS["mxfp8_layer"]
    steps = args.steps if args.steps is not None else steps
    warmup = max(3, args.warmup if args.warmup is not None else warmup)
    kw = {} if not args.tokens else {"T": args.tokens}
    if args.experts:
        kw["E"] = args.experts
    g = synth.make_mxfp8_gemm_wgrad(device=dev, **kw)
    T, E, K, I, k, P = g["T"], g["E"], g["K"], g["I"], g["k"], g["P"]
    for n in ("grad1", "grad2", "x_bf16", "h_bf16", "a2_codes", "a2_scale"):
        g.pop(n, None)
    torch.cuda.empty_cache()
    bm = 128
    cap, capb = moe.moe_align_capacity(P, E, bm)
    ids = torch.from_numpy(g["topk_ids"]).to(dev)
    topk_w = torch.full((T, k), 1.0 / k, dtype=torch.float32, device=dev)
    srt = torch.empty(cap, dtype=torch.int32, device=dev)
    eid = torch.empty(capb, dtype=torch.int32, device=dev)
    ntpp = torch.empty(4, dtype=torch.int32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    moe.moe_align(None, ids, None, T, k, E, bm, srt, cap, eid, ntpp, None, moe.Ctx(dev_status=status))
    ws = torch.empty(moe.moe_forward_workspace_size(T, k, K, I, cap), dtype=torch.uint8, device=dev)
    y = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        moe.moe_forward("mxfp8", E, K, I, g["w1"], g["w1_scale"], None, g["w2"], g["w2_scale"], None,
                        g["x_codes"], g["x_scale"], T, T, k, topk_w, srt, eid, ntpp, None, bm, cap, y,
                        moe.Ctx(workspace=ws, dev_status=status, events=evs))

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if int(status[0]) != 0:
        raise RuntimeError(f"device status {int(status[0])}")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for quad in evs:  # a torch event has a CUDA event only once it has been recorded
        for e_ in quad:
            e_.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(clocks_csv(args, rank))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop(local_rank)
    ms = t0.elapsed_time(t1)
    g1 = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    g2 = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    cb = sum(e[2].elapsed_time(e[3]) for e in evs) / steps
    ms = max_over_ranks(ms, world, dev)
    # end to end: the step's activation codes and scales from pinned host memory, y back
    ins = [g["x_codes"], g["x_scale"]]
    host = [t.cpu().pin_memory() for t in ins]
    yh = torch.empty_like(y, device="cpu").pin_memory()
    e2e_steps = max(1, min(steps, 3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for d_, h_ in zip(ins, host):
            d_.copy_(h_, non_blocking=True)
        step()
        yh.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return None
    hbm, bf16, src = peaks()
    f1, f2 = 2.0 * P * K * 2 * I, 2.0 * P * I * K
    dom, fl, dms = ("gemm1", f1, g1) if g1 >= g2 else ("gemm2", f2, g2)
    achieved = fl / (dms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": f"mx8_gemm ({dom})", "achieved": achieved, "peak": 2 * bf16,
                "unit": "TFLOP/s", "frac": achieved / (2 * bf16), "traffic": None, "algorithmic_flops": fl,
                "peak_source": f"{src} (bf16_tflops x 2, the nominal fp8/bf16 dense ratio)"}
    return {
        "metric": METRIC, "value": aggregate_rate(world, T * steps, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 block-scaled tcgen05 mma -> f32, h quantised to MXFP8 between the GEMMs",
        "data": "synthetic (seeded inputs drawn on the device, random-init weights)",
        "config": {"workload": f"mxfp8_layer: T={T} tokens, hidden {K}, intermediate {I}, {E} experts, top-{k}, "
                               f"Zipf(1.1) routing, uniform routing weights, MXFP8 layer forward",
                   "T": T, "experts": E, "hidden": K, "intermediate": I, "top_k": k, "block_m": bm,
                   "l2": "inputs larger than L2: 11.3 GB of MXFP8 weights per step",
                   "parallelism": f"replicas x{world}"},
        "useful_tflops": world * (f1 + f2) * steps / (ms * 1e-3) / 1e12,
        "kernel_ms": {"gemm1_swiglu_quant": g1, "gemm2_weighted": g2, "combine": cb},
        "roofline": roofline,
        "e2e": {"value": aggregate_rate(world, T * e2e_steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host),
                "d2h_bytes_per_step": y.numel() * 2, "steps": e2e_steps},
        "gpu_launches": steps * 3,
        "clocks": ck,
    }


def launches_per_step(w, rows):
    n = 3  # GEMM1, GEMM2, combine
    n += 1  # align (routing fused for rows <= 512)
    if w.quant == "mxfp4":
        n += 1  # x -> f16 (or gathered into slot order; or, up to 256 rows, x planes + unit list)
    if rows > 512:
        n += 1  # separate routing kernel
    if w.quant == "mxfp4":
        n += 2  # pad x, pad logits
    return n


def sample_text(name, n, r):
    if name == "mxfp8_layer":
        return f"the MXFP8 layer for {n} token-expert pairs over 2 experts ({r['tokens']:g} tokens at top-8)"
    if name == "pertoken_fp8":
        return f"{n} rows of one expert of the per-token FP8 GEMM ({r['tokens']:g} tokens at top-8)"
    if name == "mxfp8_wgrad":
        return (f"both MXFP8 grouped GEMMs and both weight gradients for {n} token-expert pairs of 2 "
                f"experts ({r['tokens']:g} tokens at top-8)")
    return f"the first {r['tokens']} tokens of the workload"


def cpu_baseline(name, m, n=None):
    """The float64 oracle on a bounded sample of the workload, timed twice on this host:
    with every core available to its BLAS / OpenMP pools, and with one thread."""
    base = "decode_bf16" if name.startswith("decode_bf16_M") else name
    n = n or ORACLE_SAMPLE[base]
    cores = host_cores()
    r_all = run_oracle_subprocess(base, m, n, threads=cores)
    r_one = run_oracle_subprocess(base, m, n, threads=1)
    return {"value": r_all["tokens"] / r_all["seconds"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"float64 oracle: {sample_text(base, n, r_all)}; {r_all['seconds']:.2f} s with "
                      f"{cores} BLAS threads, {r_one['seconds']:.2f} s with one; input generation untimed",
            "one_thread": {"value": r_one["tokens"] / r_one["seconds"], "cores": 1}}


def run_workload(args, name, rank, world, local_rank, steps=None, warmup=None):
    """One workload of the benchmark, by name (decode_bf16_M<m> for the tiny-M bf16 layer)."""
    a = argparse.Namespace(**vars(args))
    a.steps, a.warmup = steps, warmup
    if name.startswith("decode_bf16_M"):
        a.workload, a.m = "decode_bf16", int(name[len("decode_bf16_M"):])
    else:
        a.workload = name
    if a.workload == "mxfp8_wgrad":
        return bench_mxfp8_wgrad(a, rank, world, local_rank)
    if a.workload == "pertoken_fp8":
        return bench_pertoken(a, rank, world, local_rank)
    if a.workload == "mxfp8_layer":
        return bench_mxfp8_layer(a, rank, world, local_rank)
    return bench_ours(a, rank, world, local_rank)


# keys of a workload's own line that its entry in the ``workloads`` map keeps
MAP_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "layer_latency_us",
            "useful_tflops", "kernel_ms", "experts_touched", "roofline", "step_roofline", "e2e",
            "gpu_launches", "clocks", "timing")


def free_device_memory():
    import gc
    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def main():
    args = parse()
    if args.oracle_sample:
        s, n = oracle_sample(args.workload, args.m, args.sample_tokens or ORACLE_SAMPLE[args.workload])
        print(json.dumps({"seconds": s, "tokens": n}))
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        if rank == 0:
            bench_reference(args, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    single = args.workload != "all"
    head = args.workload if single else HEADLINE
    line = run_workload(args, workload_name(head, args.m), rank, world, local_rank, args.steps, args.warmup)
    workloads = {}
    if not single:
        for name in MAP_WORKLOADS:
            free_device_memory()
            sub = run_workload(args, name, rank, world, local_rank)
            if rank == 0:
                workloads[name] = {k: sub[k] for k in MAP_KEYS if k in sub}
    if rank == 0:
        if not args.no_cpu_baseline:
            for name, entry in [(workload_name(head, args.m), line)] + list(workloads.items()):
                try:
                    entry["cpu_baseline"] = cpu_baseline(name, args.m, args.sample_tokens if single else None)
                except Exception as e:  # reported, not fatal
                    entry["cpu_baseline"] = {"error": str(e)[:300]}
        if workloads:
            line["workloads"] = workloads
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_reference(args, world):
    """The reference arm: the float64 CPU oracle as it stands, on the headline workload (or
    --workload), one bounded sample of that workload per step, every core available to its
    BLAS."""
    base = HEADLINE if args.workload == "all" else args.workload
    w = workload(base, args.m)
    steps, warmup = (args.steps if args.steps is not None else 3), max(3, args.warmup or 3)
    n = 8 if base == "tiny" else 1
    cores = host_cores()
    for _ in range(min(warmup, 1)):
        run_oracle_subprocess(base, args.m, n, threads=cores)
    secs, toks = 0.0, 0
    t_wall = time.perf_counter()
    for _ in range(steps):
        r = run_oracle_subprocess(base, args.m, n, threads=cores)
        secs += r["seconds"]
        toks += r["tokens"]
    wall = time.perf_counter() - t_wall
    v = toks / secs
    if w is not None and base not in ("mxfp8_wgrad", "pertoken_fp8", "mxfp8_layer"):
        rows = w.T
        if w.quant == "mxfp4":
            from oracle import bucket as obucket   # the padded row count the GPU arm reports
            rows = obucket.bucket(w.T)
        config = layer_config(w, rows, world, workload_name(base, args.m) in L2_FLUSHED)
    else:
        config = {"workload": base, "parallelism": f"replicas x{world}"}
    # one host process ran it (n_gpus 1); the config is the GPU arm's at this world size
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1, "steps": steps,
            "warmup": warmup, "ms_per_step": secs / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config, "impl": "reference",
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} token(s) of the workload per step (float64 oracle, {cores} BLAS "
                                       f"threads; input generation untimed; wall {wall:.1f} s)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
