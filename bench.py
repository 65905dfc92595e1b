"""Benchmark of the quantized linear layer on GB300.

One step = one pass of the whole hot path over the 28-layer decoder stack
(hidden 3584, intermediate 18944, k/v 512; q,k,o,gate,up,down Q4_K, v Q6_K):

  * decode pass: the 28 x 7 linears at M = 1 token as 4 calls per layer
    (rq_linear_group for q/k/v and gate/up, which share their input;
    rq_linear for o and down), routed to the Q4_K / Q6_K GEMV, replayed
    from a CUDA graph captured once;
  * prefill pass: the same calls at M = 2048 tokens (FP8 path: weight-cache
    hit, activation absmax + E4M3 once per shared input, one tcgen05 FP8
    GEMM per call), launched eagerly.

Headline `value`: FP8 prefill TFLOP/s at M = 2048 (2*M*N*K summed over the
28 x 7 linears / device time of the prefill pass, quantization included).  The
GEMV HBM GB/s of the decode pass at M = 1 is reported in `gemv`.  `roofline`
is for the dominant kernel (the FP8 GEMM): its algorithmic FLOPs / its
device time from CUDA events around each GEMM launch, in K passes run right
after the timed ones (events between kernels would slow the timed passes).
`--sweep` prints the other configurations (GEMV at M = 1, 4, 8 over the
decoder shapes; FP8 GEMM at M = 512; the prefill stack at M = 16 .. 4096).
`e2e` repeats the measurement through the public API
with host buffers (stack input copied in from pinned memory, last output
copied back) each step.  `cpu_baseline` times the CPU oracle on a bounded
sample.  `--impl reference` times the oracle alone as the reference arm.
Inputs are larger than L2 (3.68 GB of packed weights, 6.5 GB of FP8
weights, 6.8 GB of activations), so no flush is needed between steps.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = ("Q4_K/Q6_K GEMV HBM GB/s at M=1; FP8 prefill GEMM TFLOP/s at M=2048")
SEED = 0x5EED
M_DECODE = 1
M_PREFILL = 2048
# per layer: which activation feeds each linear
SOURCE = {"q": "x", "k": "x", "v": "x", "o": "a", "gate": "h", "up": "h", "down": "g"}
# linears that share an input are one rq_linear_group call
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
ACT_K = {"x": synthetic.HIDDEN, "a": synthetic.HIDDEN, "h": synthetic.HIDDEN,
         "g": synthetic.INTERMEDIATE}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0,
            "source": "fallback"}


def stack_flops(M):
    per_tok = sum(2 * N * K for _, _, N, K in synthetic.LAYER_LINEARS)
    return per_tok * M * synthetic.N_LAYERS


def measure_fp8_peak(torch, dev):
    """Dense FP8 throughput of this GPU in this run: torch._scaled_mm, E4M3 x
    E4M3 -> bf16 at 8192^3, best of 10 single calls (burst) and calls back to
    back for about 1.5 s (sustained).  -> dict, or None if unavailable."""
    n = 8192
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()  # column-major
        one = torch.ones((), device=dev, dtype=torch.float32)

        def f():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            f()
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        calls = max(1, int(1500.0 / best))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(calls):
            f()
        e1.record()
        torch.cuda.synchronize()
        flop = 2.0 * n ** 3
        res = {"burst": flop / best / 1e9, "sustained": flop * calls / e0.elapsed_time(e1) / 1e9,
               "how": "torch._scaled_mm E4M3 x E4M3 -> bf16, 8192^3: best of 10 (burst), "
                      "%d calls back to back (sustained)" % calls}
        del a, b
        torch.cuda.empty_cache()
        return res
    except Exception as e:  # an old torch without _scaled_mm on this GPU
        return {"error": repr(e)[:200]}


def packed_bytes(qtype, N, K):
    return N * (K // 256) * (144 if qtype == synthetic.Q4K else 210)


def decode_bytes(M):
    """Algorithmic bytes of the decode pass: packed weights + x + y."""
    tot = 0
    for _, qt, N, K in synthetic.LAYER_LINEARS:
        tot += packed_bytes(qt, N, K) + 4 * M * N
    for kind in ("x", "a", "h", "g"):
        tot += 4 * M * ACT_K[kind]  # each distinct input read once
    return tot * synthetic.N_LAYERS


# ------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- distributed ----

def dist_setup():
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
    return world, rank, local


def dist_max(value, world):
    """Max of a per-rank float over all ranks (host-side timing exchange)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------- CPU oracle leg ----

class OracleSample:
    """The CPU oracle on a bounded sample of the prefill workload: `rows`
    token rows through the seven linears of layer 0.  The FP8 weight cache is
    built once (one-time work, untimed, as on the GPU); each run times the
    activation absmax + E4M3 quantization and the exact FP8 dot products."""

    def __init__(self, rows=16, seed=SEED):
        import oracle
        self.oracle = oracle
        self.rows = rows
        self.acts = {kind: synthetic.activation(synthetic.substream(seed, 500 + j), rows, K,
                                                outlier_frac=1e-3)
                     for j, (kind, K) in enumerate(ACT_K.items())}
        self.wcache = []
        for i, (name, qt, N, K) in enumerate(synthetic.LAYER_LINEARS):
            W = synthetic.weight_matrix(synthetic.layer_seed(seed, 0, i), qt, N, K)
            self.wcache.append((name, N, K) + oracle.fp8_weight_cache(qt, W, N, K))

    def run(self):
        """-> (flops, seconds) of one pass over the sample."""
        orc, rows = self.oracle, self.rows
        flops = 0
        t0 = time.perf_counter()
        for name, N, K, wb, wd in self.wcache:
            x = self.acts[SOURCE[name]]
            xb, xd = orc.quant_e4m3(x, orc.absmax_bits(x))
            ms = np.repeat(np.arange(rows), N)
            ns = np.tile(np.arange(N), rows)
            orc.fp8_gemm_pairs(xb, xd, wb, wd, ms, ns)
            flops += 2 * rows * N * K
        return flops, time.perf_counter() - t0


def oracle_gemv_sample(seed=SEED):
    """The CPU oracle's fp64 GEMV over one decoder layer at M = 1."""
    import oracle
    nbytes = 0
    t_total = 0.0
    for i, (name, qt, N, K) in enumerate(synthetic.LAYER_LINEARS):
        W = synthetic.weight_matrix(synthetic.layer_seed(seed, 0, i), qt, N, K)
        x = synthetic.activation(synthetic.substream(seed, 600 + i), 1, K)
        t0 = time.perf_counter()
        oracle.gemv(qt, W, x, N, K)
        t_total += time.perf_counter() - t0
        nbytes += packed_bytes(qt, N, K) + 4 * K + 4 * N
    return nbytes, t_total


# All-core oracle sample: one process per host core (spawn, so that no
# worker inherits a CUDA context), each running its own `rows` token rows of
# the same prefill sample; a worker builds its weight cache once (untimed).
_POOL_SAMPLE = None


def _pool_init(rows, seed):
    global _POOL_SAMPLE
    _POOL_SAMPLE = OracleSample(rows, seed)


def _pool_run(_):
    return _POOL_SAMPLE.run()


def oracle_all_cores(rows_per_core, seed=SEED):
    """-> (flops, wall seconds, workers) of the prefill sample run on every
    host core at once."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(cores, initializer=_pool_init,
                                      initargs=(rows_per_core, seed)) as pool:
        # warm-up (and wait for every worker's setup); a worker that cannot
        # start makes the pool respawn it forever, hence the time limits
        pool.map_async(_pool_run, range(cores), chunksize=1).get(timeout=600)
        t0 = time.perf_counter()
        res = pool.map_async(_pool_run, range(cores), chunksize=1).get(timeout=600)
        wall = time.perf_counter() - t0
    return sum(f for f, _ in res), wall, cores


def oracle_config_numbers(sample, seed=SEED):
    """One-core oracle figures per workload configuration (bounded samples):
    C1 the 1 x 512 x 1024 Q4_K GEMV, C2 absmax + E4M3 of 512 x 3584, C3 one
    decoder layer at M = 1 (x28 for the stack, extrapolated), C4 the FP8
    GEMM on the four prefill shapes at M = 512 (8 sampled token rows)."""
    import oracle
    out = {}
    W = synthetic.q4k_matrix(synthetic.substream(seed, 1), 512, 1024)
    x = synthetic.activation(synthetic.substream(seed, 2), 1, 1024)
    reps = 50
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.gemv(synthetic.Q4K, W, x, 512, 1024)
    t = (time.perf_counter() - t0) / reps
    out["C1_q4k_gemv_1x512x1024"] = {"ms": t * 1e3, "GB/s": (W.size + 4 * (1024 + 512)) / t / 1e9}
    x = synthetic.activation(synthetic.substream(seed, 3), 512, 3584, outlier_frac=1e-3)
    reps = 10
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.quant_e4m3(x, oracle.absmax_bits(x))
    t = (time.perf_counter() - t0) / reps
    out["C2_absmax_quant_512x3584"] = {"ms": t * 1e3, "GB/s": 5 * x.size / t / 1e9}
    nb, sg = oracle_gemv_sample(seed)
    out["C3_gemv_one_layer_M1"] = {"ms": sg * 1e3, "GB/s": nb / sg / 1e9,
                                   "stack_ms_extrapolated_x28": 28 * sg * 1e3}
    rows = 8
    xq = synthetic.activation(synthetic.substream(seed, 4), rows, 3584, outlier_frac=1e-3)
    xg = synthetic.activation(synthetic.substream(seed, 5), rows, 18944, outlier_frac=1e-3)
    flops = 0
    t0 = time.perf_counter()
    for name, N, K, wb, wd in sample.wcache:
        if name not in ("q", "k", "gate", "down"):
            continue
        x = xg if K == 18944 else xq
        xb, xd = oracle.quant_e4m3(x, oracle.absmax_bits(x))
        ms = np.repeat(np.arange(rows), N)
        ns = np.tile(np.arange(N), rows)
        oracle.fp8_gemm_pairs(xb, xd, wb, wd, ms, ns)
        flops += 2 * rows * N * K
    t = time.perf_counter() - t0
    out["C4_fp8_gemm_M512_four_shapes"] = {"sampled_token_rows": rows, "s": t,
                                           "GFLOP/s": flops / t / 1e9}
    return out


def workload_config(world):
    """The workload both arms report: the 28-layer stack's shapes and passes."""
    return {
        "workload": "28-layer decoder linear stack (7 linears per layer; q/k/v and "
                    "gate/up as grouped calls): decode pass M=1 (GEMV, graph replay) "
                    "+ prefill pass M=2048 (FP8, eager)",
        "hidden": synthetic.HIDDEN, "intermediate": synthetic.INTERMEDIATE,
        "kv_dim": synthetic.KV_DIM, "layers": synthetic.N_LAYERS,
        "M_decode": M_DECODE, "M_prefill": M_PREFILL, "gemm_threshold": 4,
        "parallelism": "replicas" if world > 1 else "single-gpu",
        "l2": "inputs larger than L2 (no flush needed)"}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle as it stands, on every host core (one
    process per core, each running `--ref-rows` token rows per step)."""
    if rank != 0:
        return
    import multiprocessing as mp
    rows = args.ref_rows
    cores = os.cpu_count() or 1
    flops = 0
    secs = 0.0
    with mp.get_context("spawn").Pool(cores, initializer=_pool_init,
                                      initargs=(rows, SEED)) as pool:
        # a worker that cannot start makes the pool respawn it forever, hence
        # the time limits
        for _ in range(args.warmup):
            pool.map_async(_pool_run, range(cores), chunksize=1).get(timeout=600)
        for _ in range(args.steps):
            t0 = time.perf_counter()
            res = pool.map_async(_pool_run, range(cores), chunksize=1).get(timeout=600)
            secs += time.perf_counter() - t0
            flops += sum(f for f, _ in res)
    value = flops / secs / 1e12
    desc = ("%d token rows of the M=2048 prefill through the 7 linears of one layer "
            "(activation absmax + E4M3 + exact FP8 dot products) per step on each of %d "
            "host cores (one process per core)" % (rows, cores))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ GPU leg ----

class Stack:
    """Device-resident 28-layer workload."""

    def __init__(self, rq, torch, dev, seed=SEED, Ms=(M_DECODE, M_PREFILL)):
        self.rq, self.torch, self.dev = rq, torch, dev
        self.ctx = rq.Context()
        L = synthetic.N_LAYERS
        self.weights = []  # [layer][linear] -> (name, qtype, N, K, tensor)
        for layer in range(L):
            row = []
            for i, (name, qt, N, K) in enumerate(synthetic.LAYER_LINEARS):
                W = synthetic.weight_matrix(synthetic.layer_seed(seed, layer, i), qt, N, K)
                row.append((name, qt, N, K, torch.from_numpy(W).to(dev)))
            self.weights.append(row)
        # activations: one seeded set per kind, copied into per-layer buffers
        self.acts = {}
        for M in Ms:
            base = {}
            for j, (kind, K) in enumerate(ACT_K.items()):
                frac = 1e-3 if M > 8 else 0.0
                a = synthetic.activation(synthetic.substream(seed, 700 + 10 * M + j), M, K,
                                         outlier_frac=frac)
                base[kind] = torch.from_numpy(a).to(dev)
            self.acts[M] = [{k: v.clone() for k, v in base.items()} for _ in range(L)]
        self.out = {M: {name: torch.empty(M, N, device=dev)
                        for name, _, N, _ in synthetic.LAYER_LINEARS}
                    for M in Ms}
        torch.cuda.synchronize()

    def run_pass(self, M, stream=None, acts=None):
        acts = acts if acts is not None else self.acts[M]
        ctx = self.ctx
        for layer in range(synthetic.N_LAYERS):
            a = acts[layer]
            lin = {name: (qt, N, K, W) for name, qt, N, K, W in self.weights[layer]}
            for grp in GROUPS:
                x = a[SOURCE[grp[0]]]
                K = lin[grp[0]][2]
                if len(grp) == 1:
                    qt, N, _, W = lin[grp[0]]
                    ctx.rq_linear(qt, W, x, self.out[M][grp[0]], M, N, K, stream)
                else:
                    ctx.rq_linear_group([lin[n][0] for n in grp], [lin[n][3] for n in grp], x,
                                        [self.out[M][n] for n in grp], [lin[n][1] for n in grp],
                                        M, K, stream)

    @staticmethod
    def decode_launches_per_pass():
        """GEMV launches of the one-token pass: a group's Q4_K members are
        one launch, joined by its Q6_K member when it has exactly one (unless
        RQ_GEMV_NO_DUAL is set); its other members one each."""
        per_layer = 0
        qtypes = {name: qt for name, qt, _, _ in synthetic.LAYER_LINEARS}
        dual = os.environ.get("RQ_GEMV_NO_DUAL") is None
        for grp in GROUPS:
            q4 = sum(1 for n in grp if qtypes[n] == synthetic.Q4K)
            q6 = len(grp) - q4
            if len(grp) >= 2 and dual and q4 >= 1 and q6 == 1:
                per_layer += 1
            else:
                per_layer += (1 if q4 >= 2 else q4) + q6
        return per_layer * synthetic.N_LAYERS


def decode_shape_rates(torch, dev, st, hbm_peak):
    """Each call type of the decode pass timed on its own: one CUDA graph
    of that call for all 28 layers (each layer's own weights, so every
    launch reads HBM), replayed three times.  -> {call: figures}."""
    res = {}
    M = M_DECODE
    ctx = st.ctx
    for grp in GROUPS:
        calls = []
        nbytes = 0
        for layer in range(synthetic.N_LAYERS):
            a = st.acts[M][layer]
            lin = {name: (qt, N, K, W) for name, qt, N, K, W in st.weights[layer]}
            x = a[SOURCE[grp[0]]]
            K = lin[grp[0]][2]
            if len(grp) == 1:
                qt, N, _, W = lin[grp[0]]
                calls.append(lambda qt=qt, W=W, x=x, N=N, K=K, n=grp[0]:
                             ctx.rq_linear(qt, W, x, st.out[M][n], M, N, K))
            else:
                calls.append(lambda x=x, K=K, lin=lin, grp=grp: ctx.rq_linear_group(
                    [lin[n][0] for n in grp], [lin[n][3] for n in grp], x,
                    [st.out[M][n] for n in grp], [lin[n][1] for n in grp], M, K))
            nbytes += sum(packed_bytes(lin[n][0], lin[n][1], K) + 4 * M * lin[n][1]
                          for n in grp) + 4 * M * K
        ms = graph_time_ms(torch, dev, calls, reps=3)
        gbs = nbytes / len(calls) / ms / 1e6
        res["+".join(grp)] = {"us_per_launch": ms * 1e3, "MB_per_launch":
                              nbytes / len(calls) / 1e6, "GB/s": gbs, "frac": gbs / hbm_peak}
    return res


def run_gpu(args, world, rank, local):
    import torch
    import quantized_linear_layers_gb300 as rq

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    t_setup = time.perf_counter()
    fp8 = measure_fp8_peak(torch, dev)
    st = Stack(rq, torch, dev)
    stream = torch.cuda.current_stream(dev)

    # one-time FP8 weight-cache build (first prefill pass) + warm-up
    st.run_pass(M_PREFILL)
    torch.cuda.synchronize()
    for _ in range(max(1, args.warmup)):
        st.run_pass(M_DECODE)
        st.run_pass(M_PREFILL)
    torch.cuda.synchronize()
    status = rq.rq_get_device_status()
    if status != 0:
        raise RuntimeError("device status %d after warm-up" % status)
    rq.rq_gemv_exact_outputs()  # count the timed decode passes' exact-path outputs only

    # capture the decode pass (launch-bound: short kernels) in a graph
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        st.run_pass(M_DECODE, cap_stream)  # warm the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=cap_stream):
            st.run_pass(M_DECODE, cap_stream)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    # ------------------------------------------------------ timed region --
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    dec_ms, pre_ms, step_ms = [], [], []
    gemm_ms = gemv_calls = 0
    gemm_n = 0
    traced = {}
    sampler = ClockSampler(local)
    dist_barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_wall = time.perf_counter()
    # The timed steps carry no per-kernel events: an event between two
    # kernels keeps them from overlapping (programmatic dependent launch),
    # which slowed the prefill pass by about 9% even with only the GEMMs
    # traced.
    events = []
    for _ in range(args.steps):
        torch.cuda.nvtx.range_push("timed_step")
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        st.run_pass(M_PREFILL, stream)
        e2.record(stream)
        torch.cuda.nvtx.range_pop()
        events.append((e0, e1, e2))
    torch.cuda.synchronize()
    for e0, e1, e2 in events:
        dec_ms.append(e0.elapsed_time(e1))
        pre_ms.append(e1.elapsed_time(e2))
        step_ms.append(e0.elapsed_time(e2))
    wall_s = time.perf_counter() - t_wall
    dist_barrier(world)
    status = rq.rq_get_device_status()
    if status != 0:
        raise RuntimeError("device status %d in timed region" % status)
    exact_outputs = rq.rq_gemv_exact_outputs()

    # Roofline of the GEMM: the same K prefill passes again, right after the
    # timed steps (clocks still sampled), with CUDA events around each of
    # the GEMM launches (4 per layer) on the launching stream.
    st.ctx.rq_ctx_trace_kinds(["gemm"])
    traced_pre_ms = []
    for _ in range(args.steps):
        e1, e2 = ev(), ev()
        e1.record(stream)
        st.ctx.rq_ctx_trace_begin(1024)
        st.run_pass(M_PREFILL, stream)
        e2.record(stream)
        tr = st.ctx.rq_ctx_trace_end()  # waits for the pass's events
        traced_pre_ms.append(e1.elapsed_time(e2))
        for k, (n, ms) in tr.items():
            c = traced.setdefault(k, [0, 0.0])
            c[0] += n
            c[1] += ms
    torch.cuda.synchronize()
    clocks = sampler.stop()

    # per-kind breakdown of the prefill pass, from two fully traced passes
    # (informational: tracing every kernel slows the pass)
    st.ctx.rq_ctx_trace_kinds(list(st.ctx.TRACE_KINDS))
    breakdown = {}
    for _ in range(2):
        st.ctx.rq_ctx_trace_begin(1024)
        st.run_pass(M_PREFILL, stream)
        for k, (n, ms) in st.ctx.rq_ctx_trace_end().items():
            c = breakdown.setdefault(k, [0, 0.0])
            c[0] += n
            c[1] += ms / 2

    K = args.steps
    pre_s = dist_max(sum(pre_ms) / 1e3, world)
    dec_s = dist_max(sum(dec_ms) / 1e3, world)
    tot_s = dist_max(sum(step_ms) / 1e3, world)
    flops = stack_flops(M_PREFILL)
    value = world * flops * K / pre_s / 1e12
    gemv_gbs = world * decode_bytes(M_DECODE) * K / dec_s / 1e9
    gemm_calls, gemm_trace_ms = traced.get("gemm", (0, 0.0))
    gemm_achieved = flops * K / (gemm_trace_ms / 1e3) / 1e12 if gemm_trace_ms else None
    # The GEMM's denominator: the FP8 peak measured above, in the regime the
    # run was in (sustained if the clocks hit the power cap while timed,
    # burst otherwise); 2 x the measured bf16 peak if it could not be taken.
    capped = clocks is not None and "sw_power_cap" in clocks.get("reasons", [])
    regime = "sustained" if capped else "burst"
    if fp8 and "burst" in fp8:
        fp8_peak = fp8[regime]
        peak_source = "measured fp8 (%s, %s)" % (regime, fp8["how"])
    else:
        fp8_peak = 2.0 * (pk["bf16_sustained"] if capped else pk["bf16"])
        peak_source = "2 x bf16_tflops%s of %s (fp8/bf16 nominal ratio 2)" % (
            "_sustained" if capped else "", pk["source"])
    traffic = gemm_traffic_per_launch()
    shapes = decode_shape_rates(torch, dev, st, pk["hbm_gbs"])
    # the same prefill pass captured once in a CUDA graph and replayed
    # (informational; the headline value is the eager pass above)
    pre_graph_ms = pass_graph_ms(torch, dev, st, M_PREFILL, reps=max(3, min(K, 10)))

    # ----------------------------------------------------------- e2e leg --
    e2e = None if args.no_e2e else run_e2e(args, st, torch, rq, dev, stream, world)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": tot_s / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 (prefill); f32 x q4k/q6k -> f32 (decode)",
        "data": "synthetic",
        "config": workload_config(world),
        "prefill_ms": pre_s / K * 1e3, "decode_ms": dec_s / K * 1e3,
        "prefill_graph": {"ms_per_pass": pre_graph_ms,
                          "TFLOP/s": flops / (pre_graph_ms / 1e3) / 1e12,
                          "note": "the prefill pass replayed from one CUDA graph"},
        "gemv": {"value": gemv_gbs, "unit": "GB/s", "M": M_DECODE,
                 "bytes_per_pass": decode_bytes(M_DECODE),
                 "roofline": {"bound": "hbm", "achieved": gemv_gbs / world,
                              "peak": pk["hbm_gbs"], "unit": "GB/s",
                              "frac": gemv_gbs / world / pk["hbm_gbs"],
                              "note": "decode pass time incl. launch gaps"},
                 "exact_path_outputs_in_decode_passes": exact_outputs,
                 "per_call": shapes},
        "roofline": {"bound": "tensor",
                     "kernel": "FP8 GEMM: fp8_gemm_kernel + fp8_gemm_pair_kernel "
                               "(tcgen05 kind::f8f6f4), all GEMM launches of the pass",
                     "achieved": gemm_achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": (gemm_achieved / fp8_peak) if gemm_achieved else None,
                     "peak_source": peak_source, "fp8_peak_measured": fp8,
                     "traffic": traffic,
                     "flops_per_launch_avg": flops / max(1, gemm_calls // K),
                     "avg_launch_ms": gemm_trace_ms / gemm_calls if gemm_calls else None,
                     "source": "CUDA events around each GEMM launch in K prefill passes run "
                               "right after the timed steps (%.3f ms per pass with the "
                               "events, %.3f ms without)" % (sum(traced_pre_ms) / K,
                                                             pre_s / K * 1e3)},
        "kernel_ms_per_prefill_pass": {k: v[1] for k, v in breakdown.items()},
        "gpu_launches": K * (Stack.decode_launches_per_pass() +
                             sum(c for c, _ in breakdown.values()) // 2),
        "clocks": clocks, "e2e": e2e, "setup_s": setup_s, "wall_s": wall_s,
        "act_cache": st.ctx.stats(),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        sample = OracleSample(args.cpu_rows)
        f, s1 = sample.run()
        try:
            fa, wall, cores = oracle_all_cores(args.cpu_rows // 2)
            all_cores = {"value": fa / wall / 1e12, "unit": "TFLOP/s", "cores": cores,
                         "seconds": wall,
                         "sample": "%d token rows of the same sample on each of %d "
                                   "processes, one per host core" % (args.cpu_rows // 2, cores)}
        except Exception as e:  # the GPU figures stand without it
            all_cores = {"error": repr(e)[:200]}
        line["cpu_baseline"] = {
            "value": f / s1 / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": "%d token rows of the M=2048 prefill through the 7 linears of "
                      "layer 0 (quant + exact FP8 dot products)" % args.cpu_rows,
            "seconds": s1,
            "all_cores": all_cores,
            "configs": oracle_config_numbers(sample)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def gemm_code_sha256(path):
    """SHA-256 of a CUDA source with its comments and blank space removed, so
    that the record of a kernel's DRAM traffic survives comment edits but
    not code changes."""
    import re
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()


def gemm_traffic_per_launch():
    """DRAM bytes per GEMM launch (stack average) from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "fp8_gemm_traffic.txt")
    src = os.path.join(ROOT, "quantized_linear_layers_gb300", "csrc", "rq_gemm.cu")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("kernel_code_sha256") != gemm_code_sha256(src):
        return None
    return int(rec["traffic_bytes_per_launch"])


def run_e2e(args, st, torch, rq, dev, stream, world):
    """Public-API end to end: each step copies the stack's input activation
    (layer 0's x) in from pinned host memory, runs both passes through
    rq_linear eagerly, and copies the last layer's down output back."""
    host_in = {M: torch.empty_like(st.acts[M][0]["x"], device="cpu").pin_memory()
               for M in (M_DECODE, M_PREFILL)}
    for M in host_in:
        host_in[M].copy_(st.acts[M][0]["x"])
    host_out = {M: torch.empty_like(st.out[M]["down"], device="cpu").pin_memory()
                for M in (M_DECODE, M_PREFILL)}
    steps = max(1, min(args.steps, 3))
    pre_ms = []
    for i in range(steps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for M in (M_DECODE, M_PREFILL):
            st.acts[M][0]["x"].copy_(host_in[M], non_blocking=True)
            st.ctx.rq_act_cache_invalidate()
            st.run_pass(M, stream)
            host_out[M].copy_(st.out[M]["down"], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i > 0:  # first iteration is warm-up
            pre_ms.append(e0.elapsed_time(e1))
    t = dist_max(sum(pre_ms) / 1e3, world)
    value = world * stack_flops(M_PREFILL) * steps / t / 1e12
    h2d = sum(host_in[M].numel() * 4 for M in host_in)
    d2h = sum(host_out[M].numel() * 4 for M in host_out)
    return {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "prefill FLOPs / (decode + prefill eager step with copies)"}


def graph_time_ms(torch, dev, calls, reps=2):
    """Device time per call of `calls` (a list of thunks), captured once in a
    CUDA graph and replayed `reps` times after one warm replay."""
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for c in calls[:3]:
            c()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for c in calls:
                c()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * len(calls))


def pass_graph_ms(torch, dev, st, M, reps=5):
    """One pass of the stack at M tokens captured in a CUDA graph (after an
    eager pass that fills the weight caches); mean replay time in ms."""
    stream = torch.cuda.current_stream(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        st.ctx.rq_act_cache_invalidate()
        st.run_pass(M, cap)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            st.ctx.rq_act_cache_invalidate()
            st.run_pass(M, cap)
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_sweep(args):
    """The configurations other than the headline line, one JSON line each:
    the decode GEMV over the decoder's shapes at M = 1, 4, 8 (graph replay,
    weights rotated through >= 512 MB so that every launch reads HBM); the
    FP8 GEMM at M = 512 on the four prefill shapes; the stack at 2 .. 16
    tokens through the GEMV route and through the FP8 route (graph replay),
    which locates the crossover of the two; the 28-layer prefill stack at
    M = 16 .. 4096 (eager, untraced; and one pass captured in a CUDA graph)."""
    import torch
    import quantized_linear_layers_gb300 as rq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    fp8 = measure_fp8_peak(torch, dev)
    fp8_peak = fp8["burst"] if fp8 and "burst" in fp8 else 2.0 * pk["bf16"]

    def out(d):
        print(json.dumps(d), flush=True)

    out({"sweep": "fp8_peak", "measured": fp8, "used_tflops": fp8_peak})
    parts = set(args.sweep_parts.split(","))
    # decode GEMV sweep
    for name, qt, N, K in [] if "gemv" not in parts else [("q,o", synthetic.Q4K, 3584, 3584), ("k", synthetic.Q4K, 512, 3584),
                           ("v", synthetic.Q6K, 512, 3584), ("gate,up", synthetic.Q4K, 18944, 3584),
                           ("down", synthetic.Q4K, 3584, 18944)]:
        W0 = torch.from_numpy(synthetic.weight_matrix(11, qt, N, K)).to(dev)
        Ws = [W0] + [W0.clone() for _ in range(-(-(512 << 20) // W0.numel()) - 1)]
        fn = rq.rq_q4k_gemv if qt == synthetic.Q4K else rq.rq_q6k_gemv
        for M in (1, 4, 8):
            x = torch.from_numpy(synthetic.activation(12 + M, M, K)).to(dev)
            y = torch.empty(M, N, device=dev)
            calls = [lambda W=W: fn(W, x, y, M, N, K) for W in Ws[:max(len(Ws), 20)]]
            rq.rq_gemv_exact_outputs()
            ms = graph_time_ms(torch, dev, calls)
            nbytes = packed_bytes(qt, N, K) + 4 * M * (K + N)
            out({"sweep": "gemv", "linear": name, "qtype": "Q4_K" if qt == synthetic.Q4K
                 else "Q6_K", "M": M, "N": N, "K": K, "us": ms * 1e3,
                 "GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / pk["hbm_gbs"],
                 "exact_outputs": rq.rq_gemv_exact_outputs()})
        del Ws, W0
    # FP8 GEMM at M = 512
    ctx = rq.Context()
    M = 512
    for N, K in [] if "gemm" not in parts else [(3584, 3584), (512, 3584), (18944, 3584),
                                                (3584, 18944)]:
        W = torch.from_numpy(synthetic.q4k_matrix(13, N, K)).to(dev)
        wq, wd = ctx.rq_fp8_weight_cache(synthetic.Q4K, W, N, K)
        x = torch.from_numpy(synthetic.activation(14, M, K, outlier_frac=1e-3)).to(dev)
        xq, xd = ctx.rq_fp8_act_cache(x, M, K)
        y = torch.empty(M, N, device=dev)
        calls = [lambda: rq.rq_fp8_gemm(xq, xd, wq, wd, y, M, N, K)] * 20
        ms = graph_time_ms(torch, dev, calls)
        tf = 2.0 * M * N * K / ms / 1e9
        out({"sweep": "fp8_gemm", "M": M, "N": N, "K": K, "us": ms * 1e3, "TFLOP/s": tf,
             "frac_fp8_peak": tf / fp8_peak})
    ctx.close()
    # route crossover: the stack at a few tokens through the GEMV route
    # (threshold above M; chunks of 8 tokens) and through the FP8 route
    # (threshold 1), each pass graph-replayed
    if "route" in parts:
        Ms = (2, 3, 4, 5, 6, 8, 12, 16)
        st = Stack(rq, torch, dev, Ms=Ms)
        for M in Ms:
            row = {}
            for route, th in (("gemv", M + 1), ("fp8", 1)):
                st.ctx.set_gemm_threshold(th)
                row[route] = pass_graph_ms(torch, dev, st, M)
            out({"sweep": "route", "M": M, "gemv_ms": row["gemv"], "fp8_ms": row["fp8"],
                 "faster": min(row, key=row.get)})
        st.ctx.close()
        del st
        torch.cuda.empty_cache()
    if "stack" not in parts:
        if rq.rq_get_device_status() != 0:
            raise SystemExit(1)
        return
    # prefill stack at several M
    Ms = (16, 128, 512, 2048, 4096)
    st = Stack(rq, torch, dev, Ms=Ms)
    for M in Ms:
        st.run_pass(M)  # weight cache on the first pass
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        e0.record()
        for _ in range(reps):
            st.ctx.rq_act_cache_invalidate()
            st.run_pass(M)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        stats = st.ctx.stats()
        gms = pass_graph_ms(torch, dev, st, M)
        out({"sweep": "prefill_stack", "M": M, "ms_per_pass": ms,
             "TFLOP/s": stack_flops(M) / ms / 1e9,
             "graph_ms_per_pass": gms, "graph_TFLOP/s": stack_flops(M) / gms / 1e9,
             "act_cache": stats})
    if rq.rq_get_device_status() != 0:
        raise SystemExit(1)


def run_case(args):
    """One kernel on one shape, `--launches` times after 3 warm-up launches:
    the small, self-contained command the ncu captures use."""
    import torch
    import quantized_linear_layers_gb300 as rq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M, N, K = args.M, args.N, args.K
    if args.case in ("gemv_q4k", "gemv_q6k"):
        qt = synthetic.Q4K if args.case == "gemv_q4k" else synthetic.Q6K
        W0 = torch.from_numpy(synthetic.weight_matrix(1, qt, N, K)).to(dev)
        # copies of the weight so that successive launches read HBM, not L2
        Ws = [W0] + [W0.clone() for _ in range(-(-(512 << 20) // W0.numel()) - 1)]
        x = torch.from_numpy(synthetic.activation(2, M, K)).to(dev)
        y = torch.empty(M, N, device=dev)
        fn = rq.rq_q4k_gemv if qt == synthetic.Q4K else rq.rq_q6k_gemv
        wit = iter(range(1 << 62))
        call = lambda: fn(Ws[next(wit) % len(Ws)], x, y, M, N, K)  # noqa: E731
    elif args.case in ("absmax", "quant", "act_cache"):
        # enough copies of the activation that successive launches read
        # HBM, not L2 (at least 512 MB in all)
        x0 = torch.from_numpy(synthetic.activation(3, M, K, outlier_frac=1e-3)).to(dev)
        xs = [x0] + [x0.clone() for _ in range(max(0, -(-(512 << 20) // (4 * M * K)) - 1))]
        it = iter(range(1 << 62))
        bits = torch.zeros(1, dtype=torch.int32, device=dev)
        out = torch.empty(M * K, dtype=torch.uint8, device=dev)
        deq = torch.empty(1, device=dev)
        rq.rq_absmax(x0, M * K, bits)
        ctx = rq.Context()

        def call():
            x = xs[next(it) % len(xs)]
            if args.case == "absmax":
                rq.rq_absmax(x, M * K, bits)
            elif args.case == "quant":
                rq.rq_quant_e4m3(x, M * K, bits, out, deq)
            else:
                ctx.rq_act_cache_invalidate()
                ctx.rq_fp8_act_cache(x, M, K)
    elif args.case == "gemm":
        ctx = rq.Context()
        W = torch.from_numpy(synthetic.q4k_matrix(4, N, K)).to(dev)
        # FP8 caches of copies of the weight (at least 512 MB in all), so
        # that successive launches read their weight from HBM, not L2
        Wsrc = [W] + [W.clone() for _ in range(-(-(512 << 20) // (N * K)) - 1)]
        caches = [ctx.rq_fp8_weight_cache(synthetic.Q4K, Wc, N, K) for Wc in Wsrc]
        wit = iter(range(1 << 62))
        x = torch.from_numpy(synthetic.activation(5, M, K, outlier_frac=1e-3)).to(dev)
        m_pad = (M + 15) // 16 * 16
        bits = torch.zeros(1, dtype=torch.int32, device=dev)
        xq = torch.zeros(m_pad * K, dtype=torch.uint8, device=dev)
        xd = torch.empty(1, device=dev)
        rq.rq_absmax(x, M * K, bits)
        rq.rq_quant_e4m3(x, M * K, bits, xq, xd)
        y = torch.empty(M, N, device=dev)
        def call():
            wq, wd = caches[next(wit) % len(caches)]
            rq.rq_fp8_gemm(xq, xd, wq, wd, y, M, N, K)
    else:
        raise SystemExit("unknown case " + args.case)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.graph:
        # the launches replayed from a CUDA graph: device time without the
        # host's per-call cost
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(dev)
        cs.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cs):
            for _ in range(3):  # warm the capture stream too
                call()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cs):
                for _ in range(args.launches):
                    call()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        s.record()
        g.replay()
        e.record()
    else:
        s.record()
        for _ in range(args.launches):
            call()
        e.record()
    torch.cuda.synchronize()
    status = rq.rq_get_device_status()
    ms = s.elapsed_time(e) / args.launches
    m_pad = (M + 15) // 16 * 16
    moved = {"absmax": 4 * M * K, "quant": 5 * M * K,
             "act_cache": 4 * M * K + m_pad * K,
             "gemv_q4k": N * (K // 256) * 144 + 4 * M * (K + N),
             "gemv_q6k": N * (K // 256) * 210 + 4 * M * (K + N)}.get(args.case)
    print(json.dumps({"case": args.case, "M": M, "N": N, "K": K, "ms_per_launch": ms,
                      "gbs": moved / ms / 1e6 if moved else None,
                      "status": status}), flush=True)
    if status != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-rows", type=int, default=16,
                    help="token rows per step of the reference arm's oracle sample")
    ap.add_argument("--cpu-rows", type=int, default=64,
                    help="token rows of the cpu_baseline oracle sample (about 10 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (profiling runs only)")
    ap.add_argument("--case", default=None,
                    help="single-kernel mode: gemv_q4k, gemv_q6k, absmax, quant, "
                         "act_cache, gemm")
    ap.add_argument("--M", type=int, default=2048)
    ap.add_argument("--N", type=int, default=3584)
    ap.add_argument("--K", type=int, default=3584)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--sweep-parts", default="gemv,gemm,route,stack",
                    help="comma-separated parts of --sweep: gemv, gemm, route, stack")
    ap.add_argument("--sweep", action="store_true",
                    help="print the GEMV, FP8 GEMM and prefill-stack sweeps instead")
    ap.add_argument("--graph", action="store_true",
                    help="single-kernel mode: time the launches as one CUDA graph replay")
    args = ap.parse_args()
    if args.case:
        return run_case(args)
    if args.sweep:
        return run_sweep(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
