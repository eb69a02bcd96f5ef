"""Benchmark of the FP8 weight-only linear layer on one GB300 (or N replicas).

One step = one pass of the decode-layer stack of an 8B-style block (hidden
4096, 32 q / 8 kv heads of 128, intermediate 14336): the q, k, v, o, gate, up
and down linears run back to back at M = 1, then M = 8, then M = 32 tokens
(21 fp8w_linear calls), weights quantised once beforehand with fp8w_quantize.
Inputs are seeded synthetic data of those shapes (W ~ N(0, 0.02), bias ~
N(0, 0.01), x bf16 ~ N(0, 1)); nothing is cached between steps.

value = algorithmic bytes of the step (codes N*K + scale 4N + bias 4N + x
2MK + y 2MN per call) / device time of the step, in GB/s, timed over
replays of the step captured in a CUDA graph.  Each step streams 654 MB of
codes; two weight replicas alternate between the M passes so every weight
read comes from HBM (inputs larger than L2, no reuse within 436 MB).  The
weights are quantised and synchronised before the timed region, so the
calls pass FP8W_FLAG_WEIGHTS_READY (the code stream starts while the
previous kernel drains); the same step without the flag is reported too.

Also printed: every call of the step and every configuration of the
workload timed directly (graph-replayed back-to-back launches of that call
alone over weight replicas larger than L2), the roofline fraction of the
dominant kernel from those direct timings, the t(M)/t(1) ratios of the
skinny sweep, the W8A8 path, the quantiser, the dequantiser, an end-to-end
figure through the Python API with pinned host buffers, the CPU oracle on a
bounded sample (linear and quantise) with the weight error report and the
outputs' error against it, and SM clocks sampled during the timed loop.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "FP8-weight linear effective GB/s and % of GB300 HBM peak at M=1..32"
WORKLOAD = ("decode_stack: 8B-style block linears q[4096x4096], k[1024x4096], v[1024x4096], "
            "o[4096x4096], gate[14336x4096], up[14336x4096], down[4096x14336] ([N x K]) back to back "
            "at M=1, 8, 32; bf16 activations, e4m3 per-channel weights, fp32 bias")


def step_calls():
    """(M, matrix name, N, K) of every linear call of one step, in order."""
    return [(m, name, n, k) for m in synthetic.DECODE_STACK_M for (name, n, k) in synthetic.DECODE_STACK]


def call_bytes(m, n, k, with_bias=True):
    return n * k + 4 * n + (4 * n if with_bias else 0) + 2 * m * k + 2 * m * n


def step_bytes():
    return sum(call_bytes(m, n, k) for (m, _, n, k) in step_calls())


def step_flops():
    return sum(2 * m * n * k for (m, _, n, k) in step_calls())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    return 6800.0, "fallback (6.8 TB/s, one earlier GB300 measurement)"


# ------------------------------------------------------------ dist helpers --

def job_time_ms(ms_local, dist, device):
    """The job's timed-region length: the maximum over ranks of each rank's
    own (every rank timed the same K steps between barriers)."""
    if dist is None:
        return ms_local
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step, n_ranks, steps, ms_total):
    """Whole-job throughput in GB/s: the bytes all ranks processed over the
    job's time (weak scaling: every rank runs the full step)."""
    return bytes_per_step * n_ranks * steps / (ms_total / 1e3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------ clock sampler --

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- CPU baseline --

CPU_STRIDE = 2  # the CPU sample takes every 2nd output channel of every call
CPU_STRIDE_1T = 32  # the single-thread figure: every 32nd channel
REF_BUDGET_S = 90.0  # host time the reference arm's timed steps may take


def cpu_sample(m_list=synthetic.DECODE_STACK_M, stride=CPU_STRIDE):
    """Inputs of the CPU sample: every call of the step, every stride-th channel."""
    import oracle
    out = []
    for m in m_list:
        for (name, n, k) in synthetic.DECODE_STACK:
            c = synthetic.case("decode_stack", m, name)
            cols = np.arange(0, n, stride)
            codes, scales = oracle.quantize(c["w"][cols])
            out.append((c["x"], codes, scales, c["bias"][cols], m, len(cols), k))
    return out


def run_cpu(sample, threads):
    import oracle
    t0 = time.perf_counter()
    for (x, codes, scales, bias, m, n, k) in sample:
        oracle.linear(x, oracle.ACT_BF16, codes, scales, bias, threads=threads)
    dt = time.perf_counter() - t0
    nbytes = sum(call_bytes(m, n, k) for (_, _, _, _, m, n, k) in sample)
    return nbytes / dt / 1e9, dt


def ordinal(i):
    return "%d%s" % (i, "th" if 10 <= i % 100 <= 20 else {1: "st", 2: "nd", 3: "rd"}.get(i % 10, "th"))


def oracle_quantize_rows(w, threads):
    """The oracle quantiser over row blocks on `threads` host threads (each
    block one oracle call; ctypes releases the interpreter lock): the same
    codes and scales as one call."""
    import concurrent.futures as cf
    import oracle
    n = w.shape[0]
    if threads <= 1 or n < 2 * threads:
        return oracle.quantize(w)
    edges = [n * i // threads for i in range(threads + 1)]
    with cf.ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda i: oracle.quantize(w[edges[i]:edges[i + 1]]), range(threads)))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def cpu_quantize_timing(cores):
    """The oracle quantiser timed on the host: the gate weight's first 2048
    rows on one thread, and the whole gate weight on all cores."""
    c = synthetic.case("decode_stack", 1, "gate")
    w = c["w"]
    sub = np.ascontiguousarray(w[:2048])
    t0 = time.perf_counter()
    oracle_quantize_rows(sub, 1)
    dt1 = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle_quantize_rows(w, cores)
    dtn = time.perf_counter() - t0
    b1 = 5 * sub.size + 4 * sub.shape[0]
    bn = 5 * w.size + 4 * w.shape[0]
    return {"single_thread": {"gbs": round(b1 / dt1 / 1e9, 4), "seconds": round(dt1, 3), "cores": 1,
                              "sample": "gate [14336 x 4096], its first 2048 rows"},
            "all_cores": {"gbs": round(bn / dtn / 1e9, 4), "seconds": round(dtn, 3), "cores": cores,
                          "sample": "gate [14336 x 4096], all rows, split over the threads"},
            "unit": "GB/s", "bytes": "5 B per weight + 4 B per row", "kind": "oracle"}


def _rel_cos(y_bits, ref_bits, act):
    """rel_l2 over all outputs and the least per-row (per-token) cosine, fp64."""
    def vals(b):
        b = np.asarray(b, dtype=np.uint16)
        if act == synthetic.ACT_F16:
            return b.view(np.float16).astype(np.float64)
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y, r = vals(y_bits), vals(ref_bits)
    rel = float(np.linalg.norm(y - r) / max(np.linalg.norm(r), 1e-300))
    num = np.sum(y * r, axis=1)
    den = np.linalg.norm(y, axis=1) * np.linalg.norm(r, axis=1)
    cos = float(np.min(np.where(den > 0, num / np.where(den > 0, den, 1.0), 1.0)))
    return rel, cos, float(np.mean(np.asarray(y_bits) == np.asarray(ref_bits)))


def accuracy_report(gpu_ys, cores):
    """The contract's report on every configuration: the weight error report
    fp8_error(weight, q, scale) of each weight (rel_l2, worst channel,
    underflow, crest), and the outputs the bench's GPU run produced against
    the oracle (rel_l2, least per-token cosine, share bit-equal; every
    channel of the small cases, every 4th of the 58.7 MB and decode-stack
    weights)."""
    import oracle
    weights = {}
    cases = {}
    worst_rel, worst_cos = 0.0, 1.0
    for key, ybits in gpu_ys.items():
        name, m, matrix = key
        c = synthetic.case(name, m, matrix) if name == "decode_stack" else \
            synthetic.case(name, m) if name == "skinny_sweep" else synthetic.case(name)
        wkey = (name, matrix)
        if wkey not in weights:
            codes, scales = oracle_quantize_rows(c["w"], cores)
            rep = oracle.fp8_error(c["w"], codes, scales)
            weights[wkey] = (codes, scales, {kk: round(float(v), 6) for kk, v in rep.items()})
        codes, scales, _ = weights[wkey]
        n = c["n"]
        stride = 1 if n * c["k"] <= 2 ** 24 else 4
        cols = np.arange(0, n, stride)
        bias = None if c["bias"] is None else c["bias"][cols]
        ref = oracle.linear(c["x"], c["act"], codes[cols], scales[cols], bias, threads=cores)
        rel, cos, eq = _rel_cos(ybits[:, cols], ref, c["act"])
        label = name if name in ("tiny_gemv", "outlier_gemv", "fp16_template") else \
            "%s@M%d" % (name, m) if name == "skinny_sweep" else "%s@M%d" % (matrix, m)
        cases[label] = {"rel_l2": float("%.3g" % rel), "min_cosine": round(cos, 7), "bit_equal": round(eq, 4),
                        "channels": "all" if stride == 1 else "every %s" % ordinal(stride)}
        worst_rel, worst_cos = max(worst_rel, rel), min(worst_cos, cos)
    return {"max_rel_l2": float("%.3g" % worst_rel), "min_cosine": round(worst_cos, 7),
            "gates": {"rel_l2": 2e-3, "min_cosine": 0.9999},
            "fp8_error": {("%s:%s" % wk if wk[1] else wk[0]): rep for wk, (_, _, rep) in weights.items()},
            "cases": cases,
            "note": "weight report of fp8_error(weight, q, scale): rel_l2 = ||W - Wq||_F / ||W||_F, worst "
                    "channel's, share of nonzero weights whose code is +-0, largest amax / rms of a row; outputs "
                    "of the bench's own GPU run against the oracle's fp64 result rounded once"}


def cpu_baseline_obj(gbs, dt, cores, stride=None):
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "the full step (21 calls, M=1,8,32) restricted to every %s output channel; "
                      "plain C fp64 oracle, %d threads; %.2f s" % (ordinal(stride or CPU_STRIDE), cores, dt)}


# ------------------------------------------------------------------- ours --

def build_state(torch, fw, dev, replicas=2):
    """Quantise the seven matrices on the GPU; keep codes, scales, bias resident."""
    mats = {}
    wdev = {}
    for (name, n, k) in synthetic.DECODE_STACK:
        c = synthetic.case("decode_stack", 1, name)
        w = torch.from_numpy(c["w"]).to(dev)
        codes, scales = fw.quantize(w)
        bias = torch.from_numpy(c["bias"]).to(dev)
        reps = [codes] + [codes.clone() for _ in range(replicas - 1)]
        mats[name] = {"codes": reps, "scales": scales, "bias": bias, "n": n, "k": k}
        wdev[name] = w
    xs, ys = {}, {}
    for (m, name, n, k) in step_calls():
        c = synthetic.case("decode_stack", m, name)
        xs[(m, name)] = torch.from_numpy(c["x"].view(np.int16)).to(dev).view(torch.bfloat16)
        ys[(m, name)] = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    return mats, wdev, xs, ys


def enqueue_step(fw, mats, xs, ys, weights_ready=True):
    launches = 0
    for (m, name, n, k) in step_calls():
        mt = mats[name]
        rep = synthetic.DECODE_STACK_M.index(m) % len(mt["codes"])
        fw.linear(xs[(m, name)], mt["codes"][rep], mt["scales"], mt["bias"], out=ys[(m, name)],
                  weights_ready=weights_ready)
        launches += 1
    return launches


def replay_us(torch, s, launch, launches, reps=5):
    """Median device time per launch (us) of `launches` calls launch(i)
    captured in one CUDA graph and replayed back to back (CUDA events on the
    launching stream, after a warm-up replay)."""
    with torch.cuda.stream(s):
        launch(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(launches):
            launch(i)
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / launches)
    del g
    return float(np.median(times))


REPLICA_BYTES = 400 * 2 ** 20   # weight replicas of a directly timed call: > 3x the 129 MB L2


def replicas(torch, codes, scales):
    nrep = max(3, -(-REPLICA_BYTES // (codes.numel() * codes.element_size())))
    return [(codes, scales)] + [(codes.clone(), scales.clone()) for _ in range(nrep - 1)]


def kernel_name(m, k):
    """The kernel (template instance, as ncu names it) that runs a call."""
    if m == 1:
        # row pairs, bf16, fp32 x up to 8192 codes a row (16-bit x beyond), one scale a row
        return "fp8w::gemv_kernel<2, 1, 1, 0>" if k <= 8192 else "fp8w::gemv_kernel<2, 1, 0, 0>"
    # tokens a launch, bf16, per-row scales
    return "fp8w::skinny_kernel<%d, 1, 0, 1>" % (16 if m <= 16 else 32)


KERNEL_SOURCES = {"skinny_kernel": ["skinny.cu", "fp8w_device.cuh"], "gemv_kernel": ["gemv.cu", "fp8w_device.cuh"]}


def kernel_source_hash(kernel):
    """sha256 over the sources a kernel is built from (to tell whether a stored
    ncu figure still describes the kernel as it is now)."""
    base = kernel.split("::")[-1].split("<")[0]
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[base]:
        with open(os.path.join(ROOT, "fp8_weight_only_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


TRAFFIC_COMMAND = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none "
                   "-k regex:'gemv_kernel|skinny_kernel' -c 21 --csv --log-file traffic.csv "
                   "python bench.py --steps 2 --warmup 1 --no-cpu")


def record_traffic(csv_path):
    """Write profiles/dram_traffic_decode_stack.json from the CSV of
    TRAFFIC_COMMAND: the first 21 linear launches (one eager step, every
    call once, L2 flushed by ncu before each launch), DRAM bytes per launch
    by kernel, with the source hash they were taken on."""
    import csv
    per = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if len(r) > 10]
    hdr = rows[0]
    ik, im, iv, iid = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value"), hdr.index("ID")
    vals = {}
    for r in rows[1:]:
        name = r[ik].replace("void ", "", 1).split("(")[0].strip()
        if "::" not in name:
            name = "fp8w::" + name
        vals.setdefault((r[iid], name), {})[r[im]] = float(r[iv].replace(",", ""))
    for (_, name), m in vals.items():
        d = per.setdefault(name, {"launches": 0, "bytes": 0.0})
        d["launches"] += 1
        d["bytes"] += m["dram__bytes_read.sum"] + m["dram__bytes_write.sum"]
    out = {"command": TRAFFIC_COMMAND, "kernels": {}}
    for name, d in per.items():
        out["kernels"][name] = {"launches": d["launches"], "dram_bytes_per_launch": round(d["bytes"] / d["launches"]),
                                "source_sha256": kernel_source_hash(name)}
    with open(os.path.join(ROOT, "profiles", "dram_traffic_decode_stack.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(json.dumps(out, indent=1))


def stored_traffic(kernel):
    """DRAM bytes per launch of `kernel` over the step's launches, from the
    committed ncu summary, or (None, why) when absent or taken on other source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic_decode_stack.json")
    if not os.path.exists(p):
        return None, "no stored ncu traffic"
    with open(p) as f:
        d = json.load(f)
    short = kernel.split("::")[-1]
    rec = next((v for kk, v in d.get("kernels", {}).items() if kk.split("::")[-1] == short), None)
    if rec is None:
        return None, "no stored ncu traffic for this kernel"
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None, "kernel source changed since the stored ncu capture"
    return rec["dram_bytes_per_launch"], "ncu dram__bytes_read.sum + dram__bytes_write.sum, " + d.get("command", "")


FUSED_GROUPS = (("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",)))


def run_fused(torch, fw, mats, xs, dev, s, steps, warmup, peak):
    """The decode stack with q/k/v and gate/up fused: one call over the
    concatenated rows of each group, on one shared x (the first member's), as
    a decode layer runs them; 4 calls per M instead of 7.  Same weights, same
    two replicas alternating between the M passes, same graph replay."""
    fmats = {}
    for gname, members in FUSED_GROUPS:
        reps = [torch.cat([mats[nm]["codes"][r] for nm in members]) for r in range(len(mats["q"]["codes"]))]
        fmats[gname] = {"codes": reps, "scales": torch.cat([mats[nm]["scales"] for nm in members]),
                        "bias": torch.cat([mats[nm]["bias"] for nm in members]),
                        "n": sum(mats[nm]["n"] for nm in members), "k": mats[members[0]]["k"], "x_of": members[0]}
    calls = [(m, g) for m in synthetic.DECODE_STACK_M for (g, _) in FUSED_GROUPS]
    ys = {(m, g): torch.empty((m, fmats[g]["n"]), dtype=torch.bfloat16, device=dev) for (m, g) in calls}

    def step():
        for (m, g) in calls:
            f = fmats[g]
            rep = synthetic.DECODE_STACK_M.index(m) % len(f["codes"])
            fw.linear(xs[(m, f["x_of"])], f["codes"][rep], f["scales"], f["bias"], out=ys[(m, g)])
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        step()
    for _ in range(warmup):
        gr.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(steps):
            gr.replay()
        e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = sum(call_bytes(m, fmats[g]["n"], fmats[g]["k"]) for (m, g) in calls)
    gbs = nbytes / (ms / 1e3) / 1e9
    # the fused calls give the parts' outputs (the GEMV bit for bit)
    x = xs[(1, "q")]
    yq = torch.empty((1, mats["q"]["n"]), dtype=torch.bfloat16, device=dev)
    fw.linear(x, mats["q"]["codes"][0], mats["q"]["scales"], mats["q"]["bias"], out=yq)
    yf = torch.empty((1, fmats["qkv"]["n"]), dtype=torch.bfloat16, device=dev)
    fw.linear(x, fmats["qkv"]["codes"][0], fmats["qkv"]["scales"], fmats["qkv"]["bias"], out=yf)
    torch.cuda.synchronize()
    assert torch.equal(yf[:, :mats["q"]["n"]], yq)
    del gr
    return {"value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 5), "frac_of_hbm_peak": round(gbs / peak, 4),
            "calls_per_step": len(calls), "bytes_per_step": nbytes, "steps": steps,
            "note": "q/k/v and gate/up fused into one call each (concatenated weight rows, one shared x), "
                    "o and down alone; M = 1, 8, 32; same weights, replicas and graph replay as the main step"}


def run_grouped(torch, fw, dev, s, peak, launches=100):
    """The per-group forms on the gate weight [14336 x 4096] (fp32 scales per
    128 and per 32, and the MX-style E8M0 byte per 32): the GEMV at M = 1,
    the tensor-core kernel's per-group form at M = 8 and 32 (and fp16
    activations with E8M0 bytes), and the prefill GEMM's per-group form at
    M = 2048; per-launch time over graph-replayed back-to-back launches,
    weight replicas (codes and scales) rotating so every read comes from HBM.
    The M = 1 entries keep the keys g128, g32 and mx."""
    c = synthetic.case("decode_stack", 1, "gate")
    w = torch.from_numpy(c["w"]).to(dev)
    bias = torch.from_numpy(c["bias"]).to(dev)
    n, k = w.shape
    rng = np.random.default_rng(7)
    out = {}

    def timed(x, reps, y, nl):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            fw.linear(x, reps[0][0], reps[0][1], bias, out=y)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                for i in range(nl):
                    cd, sd = reps[i % len(reps)]
                    fw.linear(x, cd, sd, bias, out=y)
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) * 1e3 / nl

    for group in (128, 32, "mx"):
        codes, scales = fw.quantize_mx(w) if group == "mx" else fw.quantize(w, group=group)
        nrep = max(3, -(-3 * 129 * 2 ** 20 // codes.numel()))
        reps = [(codes, scales)] + [(codes.clone(), scales.clone()) for _ in range(nrep - 1)]
        name = group if group == "mx" else "g%d" % group
        cases = [(1, torch.bfloat16), (8, torch.bfloat16), (32, torch.bfloat16)]
        if group == "mx":
            cases += [(8, torch.float16), (32, torch.float16)]
        for m, dt in cases:
            xf = rng.standard_normal((m, k)).astype(np.float32)
            x = torch.from_numpy(xf).to(dev).to(dt)
            y = torch.empty((m, n), dtype=dt, device=dev)
            us = timed(x, reps, y, launches if m == 1 else 40)
            nbytes = n * k + scales.numel() * scales.element_size() + 4 * n + 2 * m * k + 2 * m * n
            key = name if m == 1 else "%s@M%d%s" % (name, m, "" if dt == torch.bfloat16 else "_fp16")
            out[key] = {"us_per_launch": round(us, 3), "gbs": round(nbytes / us / 1e3, 1),
                        "frac": round(nbytes / us / 1e3 / peak, 4), "bytes": nbytes}
        del reps
        if group != "mx":
            # the prefill GEMM's per-group form, compute-bound: TFLOP/s
            m = 2048
            x = torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).to(dev).to(torch.bfloat16)
            y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            us = timed(x, [(codes, scales)], y, 10)
            tf = 2.0 * m * n * k / us / 1e6
            bpeak, src = bf16_peak()
            out["%s@M%d" % (name, m)] = {"us_per_launch": round(us, 2), "tflops": round(tf, 1),
                                         "frac_of_bf16_peak": round(tf / bpeak, 4)}
        del codes, scales
    out["note"] = ("gate [14336 x 4096], bf16 unless marked fp16; M = 1: the GEMV, M = 8 and 32: the tensor-core "
                   "kernel's per-group form (each group's products in their own TMEM accumulator, scaled in the "
                   "epilogue), M = 2048: the prefill GEMM's per-group form (TFLOP/s against the measured bf16 "
                   "peak); bytes = codes + group scales (4 B, or 1 B for the E8M0 byte of mx) + bias + x + y; "
                   "graph-replayed back-to-back launches over weight replicas larger than L2")
    return out


def run_warm_l2(torch, fw, dev, s, launches=200):
    """[22, 1024] x [1024, 4096] with fp16 activations (the pages' Triton
    figure, 5.6 us with a warm L2 on an sm_120 GPU): the same buffers
    replayed back to back, so the 4.2 MB weight stays in L2."""
    c = synthetic.case("fp16_template")
    w = torch.from_numpy(c["w"]).to(dev)
    x = torch.from_numpy(c["x"].view(np.int16)).to(dev).view(torch.float16)
    bias = torch.from_numpy(c["bias"]).to(dev)
    codes, scales = fw.quantize(w)
    y = torch.empty((c["m"], c["n"]), dtype=torch.float16, device=dev)
    def timed(ready):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            fw.linear(x, codes, scales, bias, out=y, weights_ready=ready)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                for _ in range(launches):
                    fw.linear(x, codes, scales, bias, out=y, weights_ready=ready)
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / launches
        del g
        return round(us, 3)
    return {"us_per_launch": timed(False), "us_per_launch_weights_ready": timed(True),
            "shape": "[22, 1024] x [1024, 4096], fp16",
            "note": "same buffers, graph-replayed back-to-back launches (warm L2), without and with the "
                    "weights-ready flag (weights quantised before the stream's previous kernel, as in a "
                    "serving loop); context: the pages report 5.6 us for this shape with a warm L2 on another GPU"}


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    return 1900.0, "fallback"


def run_prefill(torch, fw, dev, s, m=2048, launches=10):
    """The prefill GEMM on the gate weight [14336 x 4096] at m tokens (bf16):
    graph-replayed back-to-back launches; a compute-bound shape, so TFLOP/s
    against the measured bf16 tensor peak."""
    c = synthetic.case("decode_stack", 1, "gate")
    w = torch.from_numpy(c["w"]).to(dev)
    bias = torch.from_numpy(c["bias"]).to(dev)
    n, k = w.shape
    codes, scales = fw.quantize(w)
    del w
    x = torch.from_numpy(synthetic.to_bf16_bits(np.random.default_rng(m).standard_normal((m, k)).astype(np.float32))
                         .view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fw.linear(x, codes, scales, bias, out=y)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(launches):
                fw.linear(x, codes, scales, bias, out=y)
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / launches
    del g
    tf = 2.0 * m * n * k / us / 1e6
    peak, src = bf16_peak()
    return {"shape": "[%d, 4096] x gate [14336 x 4096], bf16" % m, "us_per_launch": round(us, 2),
            "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peak, 4), "peak_source": src,
            "kernel": "fp8w::prefill_kernel<256, 1, 0>"}


def direct_calls(torch, fw, mats, xs, dev, s, launches=40):
    """Every call of the step timed alone: its launches graph-replayed back
    to back over weight replicas larger than L2 (weights ready, as in the
    step).  Returns {(m, name): us per launch}."""
    out = {}
    for (name, n, k) in synthetic.DECODE_STACK:
        mt = mats[name]
        reps = replicas(torch, mt["codes"][0], mt["scales"])
        for m in synthetic.DECODE_STACK_M:
            x = xs[(m, name)]
            y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

            def launch(i, x=x, y=y):
                cd, sd = reps[i % len(reps)]
                fw.linear(x, cd, sd, mt["bias"], out=y, weights_ready=True)
            out[(m, name)] = replay_us(torch, s, launch, launches)
        del reps
    return out


def time_case(torch, fw, dev, s, c, weights_ready=True, launches=40):
    """One configuration (synthetic.case dict) timed directly: device us per
    launch over weight replicas larger than L2, and its algorithmic bytes."""
    w = torch.from_numpy(c["w"]).to(dev)
    codes, scales = fw.quantize(w)
    del w
    torch.cuda.synchronize()
    dt = torch.bfloat16 if c["act"] == synthetic.ACT_BF16 else torch.float16
    x = torch.from_numpy(np.ascontiguousarray(c["x"]).view(np.int16)).to(dev).view(dt)
    bias = None if c["bias"] is None else torch.from_numpy(c["bias"]).to(dev)
    y = torch.empty((c["m"], c["n"]), dtype=dt, device=dev)
    reps = replicas(torch, codes, scales)

    def launch(i):
        cd, sd = reps[i % len(reps)]
        fw.linear(x, cd, sd, bias, out=y, weights_ready=weights_ready)
    us = replay_us(torch, s, launch, launches)
    del reps
    return us, call_bytes(c["m"], c["n"], c["k"], with_bias=c["bias"] is not None)


def run_configs(torch, fw, dev, s, peak):
    """The workload's configurations, each timed directly: tiny GEMV,
    outlier GEMV, the skinny sweep at M = 1..32 on K = 4096, N = 14336 with
    t(M) / t(1), the 58.7 MB weight at M = 1 in both orientations, and the
    fp16 template (cold L2)."""
    def entry(us, nbytes, m, n, k):
        gbs = nbytes / us / 1e3
        return {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                "tflops": round(2 * m * n * k / us / 1e6, 3), "bytes": nbytes}
    out = {}
    for name in ("tiny_gemv", "outlier_gemv", "fp16_template"):
        c = synthetic.case(name)
        us, nb = time_case(torch, fw, dev, s, c)
        out[name] = entry(us, nb, c["m"], c["n"], c["k"])
    sweep = {}
    for m in (1,) + synthetic.SKINNY_M:
        c = synthetic.case("skinny_sweep", m)
        us, nb = time_case(torch, fw, dev, s, c)
        sweep[str(m)] = entry(us, nb, m, c["n"], c["k"])
    t1 = sweep["1"]["us"]
    for m in synthetic.SKINNY_M:
        sweep[str(m)]["t_over_t1"] = round(sweep[str(m)]["us"] / t1, 3)
    out["skinny_sweep"] = sweep
    # the targets: M = 1 at >= 80% of the HBM peak on the 58.7 MB
    # weight (both orientations), and t(M) <= 1.3 t(1) up to M = 32
    c3 = synthetic.case("decode_stack", 1, "down")
    us3, nb3 = time_case(torch, fw, dev, s, c3)
    out["m1_targets"] = {
        "gate_14336x4096": dict(sweep["1"], target_frac=0.8, met=sweep["1"]["frac"] >= 0.8),
        "down_4096x14336": dict(entry(us3, nb3, 1, c3["n"], c3["k"]), target_frac=0.8),
        "max_t_over_t1": max(sweep[str(m)]["t_over_t1"] for m in synthetic.SKINNY_M), "target_t_over_t1": 1.3}
    out["m1_targets"]["down_4096x14336"]["met"] = out["m1_targets"]["down_4096x14336"]["frac"] >= 0.8
    out["note"] = ("each case timed alone: graph-replayed back-to-back launches over weight replicas larger than "
                   "L2 (cold L2), weights ready; frac of the measured HBM peak")
    return out


def run_w8a8(torch, fw, dev, s, peak):
    """The W8A8 path: per-token activation quantisation, then the e4m3 x e4m3
    tensor-core GEMM, on the gate and down weights at M = 1, 8, 32, and the
    prefill shape against the fp8 tensor peak."""
    out = {}
    for name in ("gate", "down"):
        c = synthetic.case("decode_stack", 32, name)
        n, k = c["n"], c["k"]
        w = torch.from_numpy(c["w"]).to(dev)
        codes, scales = fw.quantize(w)
        del w
        bias = torch.from_numpy(c["bias"]).to(dev)
        reps = replicas(torch, codes, scales)
        for m in synthetic.DECODE_STACK_M:
            x = torch.from_numpy(np.ascontiguousarray(c["x"][:m]).view(np.int16)).to(dev).view(torch.bfloat16)
            qx, sx = fw.quantize_act(x)
            y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

            def gemm(i):
                cd, sd = reps[i % len(reps)]
                fw.linear_w8a8(qx, sx, cd, sd, bias, out=y, weights_ready=True)

            def both(i):
                fw.quantize_act(x, qx, sx)
                gemm(i)
            us_g = replay_us(torch, s, gemm, 40)
            us_b = replay_us(torch, s, both, 40)
            nb = n * k + 8 * n + m * k + 4 * m + 2 * m * n
            out["%s@M%d" % (name, m)] = {"gemm_us": round(us_g, 3), "gemm_gbs": round(nb / us_g / 1e3, 1),
                                         "gemm_frac": round(nb / us_g / 1e3 / peak, 4),
                                         "with_activation_quantise_us": round(us_b, 3)}
        del reps
    # prefill: compute-bound; the fp8 peak is the measured bf16 peak times
    # the nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
    c = synthetic.case("decode_stack", 1, "gate")
    n, k = c["n"], c["k"]
    w = torch.from_numpy(c["w"]).to(dev)
    codes, scales = fw.quantize(w)
    del w
    m = 2048
    x = torch.from_numpy(synthetic.to_bf16_bits(np.random.default_rng(m).standard_normal((m, k)).astype(np.float32))
                         .view(np.int16)).to(dev).view(torch.bfloat16)
    qx, sx = fw.quantize_act(x)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    us = replay_us(torch, s, lambda i: fw.linear_w8a8(qx, sx, codes, scales, None, out=y), 10)
    bf, src = bf16_peak()
    tf = 2.0 * m * n * k / us / 1e6
    out["prefill_gate_m2048"] = {"us": round(us, 2), "tflops": round(tf, 1), "peak_tflops": 2 * bf,
                                 "frac_of_fp8_peak": round(tf / (2 * bf), 4),
                                 "peak_source": src + " x 2 (nominal fp8 / bf16 dense ratio)"}
    out["note"] = ("gemm: fp8w_linear_w8a8 alone, weights ready, graph-replayed over weight replicas larger than L2; "
                   "bytes = codes + scales + bias + activation codes and scales + y; with_activation_quantise adds "
                   "fp8w_quantize_act of the bf16 activations in front of every call")
    return out


def gpu_outputs(torch, fw, dev, ys):
    """Outputs of the GPU path on every configuration, for the accuracy
    report: the decode stack's from the last timed step, the others from one
    call each (weights quantised on the GPU)."""
    out = {}
    torch.cuda.synchronize()
    for (m, name, n, k) in step_calls():
        out[("decode_stack", m, name)] = ys[(m, name)].view(torch.int16).cpu().numpy().view(np.uint16)
    cases = [("tiny_gemv", None), ("outlier_gemv", None), ("fp16_template", None)] + \
        [("skinny_sweep", m) for m in (1,) + synthetic.SKINNY_M]
    codes = scales = None
    for name, m in cases:
        c = synthetic.case(name, m) if m is not None else synthetic.case(name)
        if name != "skinny_sweep" or codes is None:
            w = torch.from_numpy(c["w"]).to(dev)
            codes, scales = fw.quantize(w)
            del w
        dt = torch.bfloat16 if c["act"] == synthetic.ACT_BF16 else torch.float16
        x = torch.from_numpy(np.ascontiguousarray(c["x"]).view(np.int16)).to(dev).view(dt)
        bias = None if c["bias"] is None else torch.from_numpy(c["bias"]).to(dev)
        y = fw.linear(x, codes, scales, bias)
        out[(name, m, None)] = y.view(torch.int16).cpu().numpy().view(np.uint16)
        if name != "skinny_sweep":
            codes = None
    return out


def run_ours(args, torch, dist):
    import fp8_weight_only_gb300 as fw
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mats, wdev, xs, ys = build_state(torch, fw, dev)
    s = torch.cuda.Stream(device=dev)

    # warm-up eagerly (module load, attribute setup), then capture the step
    with torch.cuda.stream(s):
        for _ in range(max(1, args.warmup)):
            enqueue_step(fw, mats, xs, ys)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        launches_per_step = enqueue_step(fw, mats, xs, ys)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # events at chunk boundaries inside the timed region give the spread of
    # the per-step time across the run (recording an event costs nothing)
    n_chunks = 5 if args.steps >= 5 else 1
    bounds = [args.steps * i // n_chunks for i in range(n_chunks + 1)]
    ce = [torch.cuda.Event(enable_timing=True) for _ in range(n_chunks - 1)]
    with torch.cuda.stream(s):
        e0.record(s)
        for i in range(args.steps):
            if 0 < i and i in bounds[1:-1]:
                ce[bounds.index(i) - 1].record(s)
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = job_time_ms(e0.elapsed_time(e1), dist, dev)
    ms_step = ms_total / args.steps
    marks = [e0] + ce + [e1]
    chunk_ms = [marks[i].elapsed_time(marks[i + 1]) / (bounds[i + 1] - bounds[i]) for i in range(n_chunks)]
    n_ranks = ws
    value = job_value(step_bytes(), n_ranks, args.steps, ms_total)

    # the same step without FP8W_FLAG_WEIGHTS_READY (every kernel waits for
    # the previous one before its first code copy)
    gnf = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gnf, stream=s):
        enqueue_step(fw, mats, xs, ys, weights_ready=False)
    nf_steps = max(3, min(args.steps, 500))
    for _ in range(args.warmup):
        gnf.replay()
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        f0.record(s)
        for _ in range(nf_steps):
            gnf.replay()
        f1.record(s)
    torch.cuda.synchronize()
    ms_nf = f0.elapsed_time(f1) / nf_steps
    del gnf

    # every call of the step timed alone (direct device times, not shares of
    # the step): the per-kernel and per-M figures and the roofline use these
    per_call = direct_calls(torch, fw, mats, xs, dev, s)
    peak, peak_src = peaks()

    result = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
              "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
              "dtype_detail": "e4m3 weights x bf16 activations, fp32 accumulate, bf16 out",
              "data": "synthetic",
              "config": {"workload": WORKLOAD, "M": list(synthetic.DECODE_STACK_M), "calls_per_step": 21,
                         "bytes_per_step": step_bytes(), "flops_per_step": step_flops(),
                         "l2": "inputs larger than L2: 654 MB of codes per step, two weight replicas "
                               "alternate between the M passes",
                         "graph": "step captured in one CUDA graph", "parallelism": "replicas (dp%d)" % ws,
                         "weights_ready": "FP8W_FLAG_WEIGHTS_READY on every call: the weights are quantised and "
                                          "synchronised before the timed region, as a serving loop loads them"},
              "clocks": clocks, "gpu_launches": launches_per_step * args.steps,
              "frac_of_hbm_peak": round(value / n_ranks / peak, 4), "peak_source": peak_src,
              "tflops": round(step_flops() * n_ranks / (ms_step / 1e3) / 1e12, 2),
              "spread": {"chunks": n_chunks,
                         "ms_per_step_p10": round(float(np.percentile(chunk_ms, 10)), 5),
                         "ms_per_step_median": round(float(np.median(chunk_ms)), 5),
                         "ms_per_step_p90": round(float(np.percentile(chunk_ms, 90)), 5),
                         "note": "per-step time of each of the chunks the timed steps fall into (rank 0)"},
              "without_weights_ready": {"value": round(job_value(step_bytes(), n_ranks, 1, ms_nf), 2), "unit": "GB/s",
                                        "ms_per_step": round(ms_nf, 5), "steps": nf_steps,
                                        "note": "the same step, every call waiting for the previous kernel before "
                                                "its first code copy"}}

    calls = step_calls()
    by_kernel = {}
    by_m = {}
    for (m, name, n, k) in calls:
        us = per_call[(m, name)]
        kn = kernel_name(m, k)
        d = by_kernel.setdefault(kn, {"us": 0.0, "bytes": 0, "launches": 0})
        d["us"] += us
        d["bytes"] += call_bytes(m, n, k)
        d["launches"] += 1
        e = by_m.setdefault(m, {"us": 0.0, "bytes": 0})
        e["us"] += us
        e["bytes"] += call_bytes(m, n, k)
    total = sum(d["us"] for d in by_kernel.values())
    top = max(by_kernel, key=lambda kk: by_kernel[kk]["us"])
    d = by_kernel[top]
    achieved = d["bytes"] / d["us"] / 1e3   # bytes per launch / mean launch time, GB/s
    traffic, traffic_src = stored_traffic(top)
    result["roofline"] = {"bound": "hbm", "kernel": top, "achieved": round(achieved, 1),
                          "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                          "traffic": traffic, "traffic_source": traffic_src,
                          "algorithmic_bytes_per_launch": round(d["bytes"] / d["launches"]),
                          "mean_launch_us": round(d["us"] / d["launches"], 3),
                          "share": round(d["us"] / total, 4),
                          "note": "achieved = algorithmic bytes per launch / mean device time per launch, each of "
                                  "the kernel's calls of the step timed directly (CUDA events around "
                                  "graph-replayed back-to-back launches of that call over weight replicas larger "
                                  "than L2, on the launching stream); share = its part of the summed call times; "
                                  "peak is " + peak_src}
    result["kernels"] = {kk: {"share": round(v["us"] / total, 4), "launches_per_step": v["launches"],
                              "us_per_step": round(v["us"], 3),
                              "gbs": round(v["bytes"] / v["us"] / 1e3, 1),
                              "frac": round(v["bytes"] / v["us"] / 1e3 / peak, 4)}
                         for kk, v in by_kernel.items()}
    result["per_m"] = {str(m): {"us": round(v["us"], 3), "gbs": round(v["bytes"] / v["us"] / 1e3, 1),
                                "frac": round(v["bytes"] / v["us"] / 1e3 / peak, 4)}
                       for m, v in by_m.items()}
    result["per_call_us"] = {"%s@M%d" % (name, m): round(per_call[(m, name)], 2) for (m, name, n, k) in calls}
    result["per_call_note"] = ("each call timed alone (direct device time per launch); their sum, %.1f us, exceeds "
                               "the step's %.1f us because the step's launches overlap (programmatic dependent "
                               "launch)" % (total, ms_step * 1e3))
    result["configs"] = run_configs(torch, fw, dev, s, peak)
    result["w8a8"] = run_w8a8(torch, fw, dev, s, peak)

    result["fused_stack"] = run_fused(torch, fw, mats, xs, dev, s, min(args.steps, 500), args.warmup, peak)

    result["grouped"] = run_grouped(torch, fw, dev, s, peak)
    result["warm_l2"] = run_warm_l2(torch, fw, dev, s)
    result["prefill"] = run_prefill(torch, fw, dev, s)

    # quantiser throughput on the seven matrices (load-time step)
    qcodes = {name: torch.empty_like(mats[name]["codes"][0]) for name in wdev}
    qscales = {name: torch.empty_like(mats[name]["scales"]) for name in wdev}
    with torch.cuda.stream(s):
        for _ in range(2):
            for name in wdev:
                fw.quantize(wdev[name], qcodes[name], qscales[name])
    torch.cuda.synchronize()
    q0 = torch.cuda.Event(enable_timing=True)
    q1 = torch.cuda.Event(enable_timing=True)
    qreps = 5
    gq = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gq, stream=s):
        for _ in range(qreps):
            for name in wdev:
                fw.quantize(wdev[name], qcodes[name], qscales[name])
    gq.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        q0.record(s)
        gq.replay()
        q1.record(s)
    torch.cuda.synchronize()
    del gq
    qbytes = sum(5 * n * k + 4 * n for (_, n, k) in synthetic.DECODE_STACK)
    qms = q0.elapsed_time(q1) / qreps
    result["quantize"] = {"gbs": round(qbytes / (qms / 1e3) / 1e9, 1), "ms_per_pass": round(qms, 4),
                          "frac": round(qbytes / (qms / 1e3) / 1e9 / peak, 4),
                          "bytes_per_pass": qbytes, "note": "7 matrices, 5 B/element + 4 B/row, graph-replayed launches"}
    for name in wdev:
        assert torch.equal(qcodes[name], mats[name]["codes"][0])

    # dequantiser throughput on the seven matrices (bf16 out, the pages' fallback weight)
    dq = {name: torch.empty((mats[name]["n"], mats[name]["k"]), dtype=torch.bfloat16, device=dev) for name in wdev}
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=s):
        for r in range(qreps):
            for name in wdev:
                fw.dequantize(mats[name]["codes"][r % len(mats[name]["codes"])], mats[name]["scales"], out=dq[name])
    gd.replay()
    torch.cuda.synchronize()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        d0.record(s)
        gd.replay()
        d1.record(s)
    torch.cuda.synchronize()
    del gd
    dbytes = sum(3 * n * k + 4 * n for (_, n, k) in synthetic.DECODE_STACK)
    dms = d0.elapsed_time(d1) / qreps
    result["dequantize"] = {"gbs": round(dbytes / (dms / 1e3) / 1e9, 1), "ms_per_pass": round(dms, 4),
                            "frac": round(dbytes / (dms / 1e3) / 1e9 / peak, 4), "bytes_per_pass": dbytes,
                            "note": "7 matrices to bf16, 1 B read + 2 B written per element + 4 B/row, graph-replayed launches"}
    del dq

    # end to end through the Python API: every step copies all its inputs in
    # from pinned host memory (one packed copy) and all its outputs back (one
    # packed copy); timed by the host's wall clock, the step captured in a
    # CUDA graph and replayed (as a serving loop runs it), and eagerly
    keys_x, keys_y = list(xs), list(ys)
    xoff, yoff = {}, {}
    o = 0
    for key in keys_x:
        xoff[key] = o
        o += xs[key].numel()
    xpack = torch.empty(o, dtype=torch.bfloat16, device=dev)
    o = 0
    for key in keys_y:
        yoff[key] = o
        o += ys[key].numel()
    ypack = torch.empty(o, dtype=torch.bfloat16, device=dev)
    xv = {key: xpack[xoff[key]:xoff[key] + xs[key].numel()].view(xs[key].shape) for key in keys_x}
    yv = {key: ypack[yoff[key]:yoff[key] + ys[key].numel()].view(ys[key].shape) for key in keys_y}
    hxpack = torch.cat([xs[key].reshape(-1) for key in keys_x]).cpu().pin_memory()
    hypack = torch.empty(ypack.numel(), dtype=torch.bfloat16).pin_memory()
    h2d, d2h = hxpack.numel() * 2, hypack.numel() * 2

    def e2e_step():
        xpack.copy_(hxpack, non_blocking=True)
        enqueue_step(fw, mats, xv, yv)
        hypack.copy_(ypack, non_blocking=True)

    def wall(run):
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(s):
            for _ in range(args.steps):
                run()
            s.synchronize()
        dt = time.perf_counter() - t0
        if dist is not None:
            t = torch.tensor([dt], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            dt = float(t.item())
        return dt

    with torch.cuda.stream(s):
        for _ in range(max(1, args.warmup)):
            e2e_step()
    torch.cuda.synchronize()
    eager_s = wall(e2e_step)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=s):
        e2e_step()
    for _ in range(args.warmup):
        ge.replay()
    torch.cuda.synchronize()
    e2e_s = wall(ge.replay)
    # the host outputs are the device path's outputs
    ycheck = torch.cat([ys[key].reshape(-1) for key in keys_y]).cpu()
    assert torch.equal(hypack, ycheck)
    del ge

    # the same steps as a serving loop pipelines them: two sets of device
    # buffers; step i+1's inputs are copied in and step i's outputs copied out
    # on their own streams while step i computes, ordered by events
    xpk = [xpack, torch.empty_like(xpack)]
    ypk = [ypack, torch.empty_like(ypack)]
    hyk = [hypack, torch.empty_like(hypack).pin_memory()]
    gsteps = []
    for b in range(2):
        xvb = {key: xpk[b][xoff[key]:xoff[key] + xs[key].numel()].view(xs[key].shape) for key in keys_x}
        yvb = {key: ypk[b][yoff[key]:yoff[key] + ys[key].numel()].view(ys[key].shape) for key in keys_y}
        gb = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gb, stream=s):
            enqueue_step(fw, mats, xvb, yvb)
        gsteps.append(gb)
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    step_i = [0]

    def pipelined_step():
        b = step_i[0] % 2
        step_i[0] += 1
        with torch.cuda.stream(cin):
            cin.wait_event(comp_done[b])          # the step two back has read these inputs
            xpk[b].copy_(hxpack, non_blocking=True)
            in_done[b].record(cin)
        s.wait_event(in_done[b])
        s.wait_event(out_done[b])                 # the step two back's outputs are out
        gsteps[b].replay()
        comp_done[b].record(s)
        with torch.cuda.stream(cout):
            cout.wait_event(comp_done[b])
            hyk[b].copy_(ypk[b], non_blocking=True)
            out_done[b].record(cout)

    def wall_pipelined(nsteps):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(s):
            for _ in range(nsteps):
                pipelined_step()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if dist is not None:
            t = torch.tensor([dt], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            dt = float(t.item())
        return dt

    with torch.cuda.stream(s):
        for _ in range(max(2, args.warmup)):
            pipelined_step()
    torch.cuda.synchronize()
    pipe_s = wall_pipelined(args.steps)
    assert torch.equal(hyk[(step_i[0] - 1) % 2], ycheck)
    del gsteps
    result["e2e"] = {"value": round(step_bytes() * n_ranks * args.steps / pipe_s / 1e9, 2), "unit": "GB/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "ms_per_step": round(pipe_s / args.steps * 1e3, 4),
                     "note": "fp8w.linear calls of each step plus one pinned-host copy of all its inputs in and one "
                             "of all its outputs back, every step; the step captured in a CUDA graph, its copies on "
                             "their own streams so that they overlap the neighbouring steps' compute (two buffer "
                             "sets, event-ordered); host wall clock"}
    result["e2e_serial"] = {"value": round(step_bytes() * n_ranks * args.steps / e2e_s / 1e9, 2), "unit": "GB/s",
                            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                            "ms_per_step": round(e2e_s / args.steps * 1e3, 4),
                            "note": "the same, with the copies and the step in one graph on one stream, one after "
                                    "another; host wall clock"}
    result["e2e_eager"] = {"value": round(step_bytes() * n_ranks * args.steps / eager_s / 1e9, 2), "unit": "GB/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "ms_per_step": round(eager_s / args.steps * 1e3, 4),
                           "note": "the same step issued eagerly from Python (21 fp8w.linear calls, two packed "
                                   "copies); host wall clock"}
    if rank == 0 and not args.no_cpu:
        result["_gpu_ys"] = gpu_outputs(torch, fw, dev, ys)
    err = fw.device_error()
    if err != 0:
        result["device_error"] = err
    return result


def run_profile_case(args):
    """One decode-stack linear, for ncu captures and launch-shape sweeps: eager
    launches first (what ncu captures), then --reps launches captured in a
    CUDA graph and replayed, timed with events (device time per launch)."""
    import torch
    import fp8_weight_only_gb300 as fw
    name, m = args.profile.split(":")
    m = int(m)
    dev = torch.device("cuda:0")
    c = synthetic.case("decode_stack", m, name)
    w = torch.from_numpy(c["w"]).to(dev)
    # per-group scales (--group 32, 64, 128 or mx): the automatic kernel choice
    if args.group == "mx":
        codes, scales = fw.quantize_mx(w)
    elif args.group:
        codes, scales = fw.quantize(w, group=int(args.group))
    else:
        codes, scales = fw.quantize(w)
    del w
    kw = {} if args.group else {"kernel": args.kernel, "cluster": args.cluster, "tiles": args.tiles}
    nrep = max(3, -(-3 * 129 * 2 ** 20 // codes.numel()))   # replicas covering > 3x L2
    reps = [codes] + [codes.clone() for _ in range(nrep - 1)]
    bias = torch.from_numpy(c["bias"]).to(dev)
    x = torch.from_numpy(c["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((m, c["n"]), dtype=torch.bfloat16, device=dev)
    if args.w8a8:
        # the W8A8 GEMM on the same weight: activation codes made once
        qx, sx = fw.quantize_act(x)
        torch.cuda.synchronize()

        def call(cd):
            fw.linear_w8a8(qx, sx, cd, scales, bias, out=y)
    else:
        def call(cd):
            fw.linear(x, cd, scales, bias, out=y, **kw)
    for i in range(3):
        call(reps[i % nrep])
    torch.cuda.synchronize()
    out = {"case": args.profile, "group": args.group, "kernel": args.kernel, "cluster": args.cluster, "tiles": args.tiles,
           "bytes": call_bytes(m, c["n"], c["k"]) - 4 * c["n"] + scales.numel() * scales.element_size()
           - (m * c["k"] - 4 * m if args.w8a8 else 0), "w8a8": bool(args.w8a8)}
    if args.reps > 3:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(args.reps):
                call(reps[i % nrep])
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (3 * args.reps)
        out.update({"us_per_launch": round(us, 3), "gbs": round(out["bytes"] / (us / 1e6) / 1e9, 1)})
    print(json.dumps(out))
    assert fw.device_error() == 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--profile", default=None, metavar="MATRIX:M",
                    help="profiling case: quantise one decode-stack matrix and run fp8w_linear --reps times "
                         "(three weight replicas, so every read comes from HBM); prints per-launch times")
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--kernel", type=int, default=0, help="with --profile: 0 auto, 1 gemv, 2 tensor-core (few tokens), 3 prefill GEMM")
    ap.add_argument("--cluster", type=int, default=0, help="with --profile: tensor-core CTAs per cluster (0 = from the shape)")
    ap.add_argument("--tiles", type=int, default=0, help="with --profile and --cluster: 128-channel tiles a cluster shares")
    ap.add_argument("--w8a8", action="store_true", help="with --profile: the W8A8 GEMM on the same weight")
    ap.add_argument("--group", default=None, choices=["32", "64", "128", "mx"],
                    help="with --profile: per-group fp32 scales (or mx: E8M0 bytes), the automatic kernel choice")
    ap.add_argument("--record-traffic", default=None, metavar="CSV",
                    help="write profiles/dram_traffic_decode_stack.json from an ncu CSV (see TRAFFIC_COMMAND)")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic)
        return
    if args.profile:
        run_profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()

    if args.impl == "reference":
        # the reference arm is the CPU oracle, timed on the host cores
        if rank != 0:
            return
        import oracle
        cores = oracle.host_cores()
        # each step samples every stride-th channel of every call, the stride
        # chosen so that the whole run fits REF_BUDGET_S of host time: a
        # pass over every 64th channel prices a full step first
        _, dt_probe = run_cpu(cpu_sample(stride=64), cores)
        stride = max(CPU_STRIDE, int(math.ceil(dt_probe * 64 * args.steps / REF_BUDGET_S)))
        sample = cpu_sample(stride=stride)
        for _ in range(args.warmup):
            run_cpu(sample[:1], cores)
        tot_bytes, tot_s = 0, 0.0
        for _ in range(args.steps):
            gbs, dt = run_cpu(sample, cores)
            tot_s += dt
            tot_bytes += gbs * dt * 1e9
        value = tot_bytes / tot_s / 1e9
        out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic",
               "config": {"workload": WORKLOAD, "M": list(synthetic.DECODE_STACK_M),
                          "sample": "every %s output channel of every call" % ordinal(stride)},
               "cpu_baseline": cpu_baseline_obj(value, tot_s / args.steps, cores, stride),
               "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return

    import torch
    dist = None
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    result = run_ours(args, torch, dist)
    gpu_ys = result.pop("_gpu_ys", None)
    if rank == 0 and not args.no_cpu:
        import oracle
        cores = oracle.host_cores()
        gbs, dt = run_cpu(cpu_sample(), cores)
        result["cpu_baseline"] = cpu_baseline_obj(gbs, dt, cores)
        gbs1, dt1 = run_cpu(cpu_sample(stride=CPU_STRIDE_1T), 1)
        result["cpu_baseline"]["single_thread"] = {
            "value": round(gbs1, 4), "unit": "GB/s", "cores": 1, "seconds": round(dt1, 2),
            "sample": "every %s output channel of every call, one thread" % ordinal(CPU_STRIDE_1T)}
        result["cpu_baseline"]["quantize"] = cpu_quantize_timing(cores)
        # the oracle leg also checks this run's outputs and reports the weights' error
        result["accuracy"] = accuracy_report(gpu_ys, cores)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


if __name__ == "__main__":
    main()
