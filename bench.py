"""Throughput of the W4A16 NVFP4 weight-only GEMM on one GB300 (or N replicas).

Default workload: the decode dense linears -- M in {1,2,4,8,16} x (K,N) in
{(4096,4096),(4096,14336),(14336,4096),(5120,25600)}, weights quantized from
N(0,0.02), activations ~N(0,1) BF16.  One step = the 20 GEMMs once, captured
in a CUDA graph and replayed; every GEMM of a step reads its own weight copy
(745 MB of distinct weights per step, larger than L2).  The metric is the
algorithmic bytes moved per second (weights at 0.5625 B/element plus BF16
activations in and out), with TFLOP/s beside it.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]
                    [--workload decode|prefill|lmhead|moe|mlp|tails] [--dtype bf16|f16]

--dtype f16 runs the same workload with FP16 activations (FP16 weights operand
and output) through the *_f16 entry points.

Under torchrun each rank runs its own replica (the path has no data exchange);
rank 0 prints one JSON line with the max-over-ranks time.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# The CPU baseline is the numpy oracle run single-threaded; pin BLAS before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

DECODE_SHAPES = [(4096, 4096), (4096, 14336), (14336, 4096), (5120, 25600)]
DECODE_M = [1, 2, 4, 8, 16]


def weight_bytes(N, K):
    return N * K // 2 + N * K // 16 + 4


def algo_bytes(M, N, K):
    return weight_bytes(N, K) + 2 * M * K + 2 * M * N


def flops(M, N, K):
    return 2 * M * N * K


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                        bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                        source="measured")
        except Exception:
            pass
    return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0,
                source="fallback")


def in_run_peaks(device):
    """Copy bandwidth and cuBLAS BF16 GEMM throughput measured in this run
    (context beside the peaks the roofline divides by): a 1 GiB
    device-to-device copy (read + write bytes) and an 8192^3 BF16 matmul,
    each timed with CUDA events over 10 repetitions after 3 warm-ups."""
    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / 10
    n = 1 << 29                                         # elements: 1 GiB of BF16
    a = torch.empty(n, dtype=torch.bfloat16, device=device)
    b = torch.empty_like(a)
    t_copy = timed(lambda: b.copy_(a))
    del a, b
    m = 8192
    A = torch.randn(m, m, dtype=torch.bfloat16, device=device)
    B = torch.randn(m, m, dtype=torch.bfloat16, device=device)
    t_mm = timed(lambda: torch.matmul(A, B))
    del A, B
    torch.cuda.empty_cache()
    return {"hbm_copy_gbs": round(2 * 2 * n / t_copy / 1e9, 1),
            "bf16_gemm_tflops": round(2 * m ** 3 / t_mm / 1e12, 1),
            "note": "measured in this run (1 GiB D2D copy; cuBLAS 8192^3 BF16 matmul); context only"}


def gpu_index():
    """nvidia-smi index of the current CUDA device."""
    if "CUDA_VISIBLE_DEVICES" not in os.environ:
        return torch.cuda.current_device()
    return int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[torch.cuda.current_device()])


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"], samples=0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None,
                    reasons=sorted(reasons), samples=len(sm))


# DRAM traffic per launch of the dominant kernel, from a committed ncu capture:
# dram bytes read + written / algorithmic bytes of the captured launch, kept in
# a small JSON beside the capture's summary under profiles/, valid only while
# the kernel's sources hash to the value recorded there.
PROFILE_FOR = {
    "decode": ("profiles/decode_kernel_lmhead_m8.traffic.json",
               ["gemm_decode.cu", "stream_mma.cuh", "common.cuh", "ptx.cuh"]),
    "tensor": ("profiles/tc_gemm_kernel_prefill_2048x5120x13824.traffic.json",
               ["gemm_tc.cu", "tc_ptx.cuh", "common.cuh", "ptx.cuh"]),
}


def kernel_sources_sha(srcs):
    """Hash of the kernel's sources with comments and blank lines removed, so
    that editing a comment does not invalidate a capture."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in srcs:
        text = open(os.path.join(ROOT, "w4a16_nvfp4_weight_gb300", "csrc", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def traffic_ratio(kind):
    """(ratio, capture file) when the capture matches the current sources, else (None, reason)."""
    path, srcs = PROFILE_FOR[kind]
    try:
        rec = json.load(open(os.path.join(ROOT, path)))
    except (OSError, ValueError):
        return None, f"no capture record ({path})"
    if rec.get("kernel_sources_sha") != kernel_sources_sha(srcs):
        return None, f"{path}: kernel sources changed since the capture"
    return float(rec["traffic_ratio"]), path


# ------------------------------------------------------------------ inputs --
# Activation type of the run (--dtype): "bf16" (default) or "f16".
ACT = "bf16"


def act_torch():
    return torch.bfloat16 if ACT == "bf16" else torch.float16


def bits_tensor(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(act_torch()).to(device)


def build_decode_workload(nv, synth, device, awq=False):
    """Weights (distinct copy per GEMM of a step) and activations (with a
    per-channel AWQ pre-quant scale per GEMM when awq)."""
    launches = []
    base = {}
    for si, (K, N) in enumerate(DECODE_SHAPES):
        packed, scales, d = synth.weight_only(K, N, synth.seed_for(1, si))
        w = nv.repack(torch.from_numpy(packed).to(device), torch.from_numpy(scales).to(device),
                      float(d), N, K)
        base[(K, N)] = (w, packed, scales, d)
    r = synth.rng(synth.seed_for(1, 99))
    for M in DECODE_M:
        for (K, N) in DECODE_SHAPES:
            w0 = base[(K, N)][0]
            w = nv.NVFP4Weight(w0.buf.clone(), N, K)       # a copy per GEMM: no L2 reuse in a step
            x_bits = synth.normal_act(r, (M, K), ACT)
            pqs_bits = synth.awq_scale_bits(r, K, ACT) if awq else None
            launches.append(dict(M=M, K=K, N=N, w=w, x=bits_tensor(x_bits, device), x_bits=x_bits,
                                 pqs_bits=pqs_bits, pqs=bits_tensor(pqs_bits, device) if awq else None,
                                 y=torch.empty((M, N), dtype=act_torch(), device=device)))
    return launches, base


def build_toy_workload(nv, synth, device):
    """The small single linear: M=4, K=N=256, uniform codes, divisor 448."""
    c = synth.uniform_codes_case()
    w = nv.repack(torch.from_numpy(c.packed).to(device), torch.from_numpy(c.scales).to(device),
                  float(c.divisor), c.N, c.K)
    x_bits = c.x_bits if ACT == "bf16" else synth.normal_act(synth.rng(5), (c.M, c.K), ACT)
    launch = dict(M=c.M, K=c.K, N=c.N, w=w, x=bits_tensor(x_bits, device), x_bits=x_bits, pqs=None,
                  pqs_bits=None, y=torch.empty((c.M, c.N), dtype=act_torch(), device=device))
    return [launch], {(c.K, c.N): (w, c.packed, c.scales, c.divisor)}


def build_dense_workload(nv, synth, device, shapes, wl_index, awq=False):
    launches, base = [], {}
    r = synth.rng(synth.seed_for(wl_index, 99))
    for si, (M, K, N) in enumerate(shapes):
        if (K, N) not in base:
            packed, scales, d = synth.weight_only(K, N, synth.seed_for(wl_index, si))
            w = nv.repack(torch.from_numpy(packed).to(device), torch.from_numpy(scales).to(device),
                          float(d), N, K)
            base[(K, N)] = (w, packed, scales, d)
        w = base[(K, N)][0]
        x_bits = synth.normal_act(r, (M, K), ACT)
        pqs_bits = synth.awq_scale_bits(r, K, ACT) if awq else None
        launches.append(dict(M=M, K=K, N=N, w=w, x=bits_tensor(x_bits, device), x_bits=x_bits,
                             pqs_bits=pqs_bits,
                             pqs=bits_tensor(pqs_bits, device) if awq else None,
                             y=torch.empty((M, N), dtype=act_torch(), device=device)))
    return launches, base


# --------------------------------------------------------------- GPU arm --
def run_ours(args, rank, world, device):
    import w4a16_nvfp4_weight_gb300 as nv
    from w4a16_nvfp4_weight_gb300 import synth

    nv._lib.load()
    torch.cuda.set_device(device)
    wl = args.workload
    if wl == "decode":
        launches, base = build_decode_workload(nv, synth, device, awq=args.awq)
        config = {"workload": "decode dense linears M{1,2,4,8,16} x (K,N){(4096,4096),(4096,14336),"
                              "(14336,4096),(5120,25600)}" + (" with AWQ" if args.awq else ""),
                  "gemms_per_step": len(launches)}
    elif wl == "prefill":
        shapes = [(M, K, N) for M in (512, 2048, 8192) for (K, N) in ((5120, 13824), (13824, 5120), (8192, 28672))]
        launches, base = build_dense_workload(nv, synth, device, shapes, 2, awq=args.awq)
        config = {"workload": "prefill dense linears M{512,2048,8192} x (K,N){(5120,13824),(13824,5120),"
                              "(8192,28672)}" + (" with AWQ" if args.awq else ""), "gemms_per_step": len(launches)}
    elif wl == "lmhead":
        shapes = [(M, 4096, 151936) for M in (1, 8, 256)]
        launches, base = build_dense_workload(nv, synth, device, shapes, 4)
        config = {"workload": "LM head M{1,8,256} x K=4096 x N=151936", "gemms_per_step": len(launches)}
    elif wl == "tails":
        shapes = [(M, K, N) for M in (1, 8, 256) for (K, N) in ((2064, 1000), (720, 3000))]
        launches, base = build_dense_workload(nv, synth, device, shapes, 4)
        config = {"workload": "odd shapes M{1,8,256} x (K,N){(2064,1000),(720,3000)}", "gemms_per_step": len(launches)}
    elif wl == "toy":
        launches, base = build_toy_workload(nv, synth, device)
        config = {"workload": "single linear M=4 K=256 N=256 (uniform random E2M1 codes, uniform E4M3 scales, "
                              "global divisor 448; latency-bound)", "gemms_per_step": len(launches)}
    elif wl == "moe":
        return run_moe(args, rank, world, device, nv, synth)
    elif wl == "mlp":
        return run_mlp(args, rank, world, device, nv, synth)
    else:
        raise SystemExit(f"unknown workload {wl}")

    for L in launches:
        L["ws"] = None
        need = nv.gemm_workspace_size(L["M"], L["N"], L["K"], L["pqs"] is not None)
        if need:
            L["ws"] = torch.empty(need, dtype=torch.uint8, device=device)

    def step():
        for L in launches:
            nv.gemm(L["x"], L["w"], pre_quant_scale=L["pqs"], out=L["y"], workspace=L["ws"])

    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        assert nv.device_status() == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
    torch.cuda.synchronize()

    bytes_step = sum(algo_bytes(L["M"], L["N"], L["K"]) for L in launches)
    flops_step = sum(flops(L["M"], L["N"], L["K"]) for L in launches)
    launches_per_step = sum(launch_count(nv, L) for L in launches)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_index())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    ms_step = ms / args.steps
    assert nv.device_status() == 0

    # per-launch kernel durations (CUDA events around graphs of back-to-back launches)
    kern = kernel_timing(nv, launches, base, stream, device)

    bw_unit = wl in ("decode", "lmhead", "tails", "toy")
    ratio, traffic_src = traffic_ratio("decode" if bw_unit else "tensor")
    traffic = None if ratio is None else round(ratio * kern["bytes"] / len(launches))
    e2e_graph = run_e2e(nv, launches, stream, args, bw_unit)
    e2e = run_e2e_per_call(nv, launches, stream, args, bw_unit)
    pk = peaks()
    if bw_unit:
        unit, value = "GB/s", world * bytes_step / (ms_step * 1e-3) / 1e9
        bound, ach_unit = "hbm", "GB/s"
        achieved = kern["bytes"] / kern["seconds"] / 1e9
        peak, peak_name = pk["hbm"], "HBM copy"
    else:
        # the per-shape kernel times are short graphs of one shape (the kernel
        # timed on its own): the burst BF16 peak is the matching denominator
        unit, value = "TFLOP/s", world * flops_step / (ms_step * 1e-3) / 1e12
        bound, ach_unit = "tensor", "TFLOP/s"
        achieved = kern["flops"] / kern["seconds"] / 1e12
        peak, peak_name = pk["bf16"], "bf16 burst (kernels timed in isolation)"
    res = {
        "metric": "W4A16 NVFP4 GEMM TFLOPS & weight GB/s (1 GB300) and % of roofline",
        "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": ACT,
        "data": "synthetic (seeded; NVFP4 weights quantized from N(0,0.02), X~N(0,1))",
        "config": dict(config, parallelism=f"replicas{world}" if world > 1 else "single GPU",
                       l2="inputs larger than L2: each GEMM of a step reads its own weight copy "
                          f"({sum(weight_bytes(L['N'], L['K']) for L in launches) / 1e6:.0f} MB per step)"),
        "tflops": round(world * flops_step / (ms_step * 1e-3) / 1e12, 3),
        "weight_gbs": round(world * sum(weight_bytes(L["N"], L["K"]) for L in launches) / (ms_step * 1e-3) / 1e9, 2),
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": ach_unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_note": "bytes per launch: DRAM/algorithmic ratio of a committed ncu capture "
                                     f"({traffic_src}) times this workload's mean algorithmic bytes per launch",
                     "peak_source": f"{pk['source']} ({peak_name})",
                     "kernel": "nvfp4::decode_kernel" if bound == "hbm" else "nvfp4::tc_gemm_kernel",
                     "per_shape_us": kern["per_shape_us"]},
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"]},
        "e2e": e2e,
        "e2e_graph": e2e_graph,
        "gpu_launches": launches_per_step * args.steps,
    }
    if world == 1:
        res["roofline"]["peaks_in_run"] = in_run_peaks(device)
    res["_base"] = base
    res["_cases"] = host_cases(launches)
    return res


def host_cases(launches):
    """Host copies of each launch's inputs for the oracle baselines:
    (M, K, N, activation bits, AWQ scale bits or None)."""
    return [(L["M"], L["K"], L["N"], L["x_bits"], L.get("pqs_bits")) for L in launches]


MOE_E, MOE_TOPK, MOE_H, MOE_I = 128, 8, 2048, 768
MOE_T = (1, 16, 256, 4096)


def run_moe(args, rank, world, device, nv, synth):
    """The MoE layer (128 experts, top-8, hidden 2048, intermediate 768) at
    T = 1, 16, 256, 4096 tokens, one call each per step."""
    fc1, fc2 = synth.moe_weights(MOE_E, MOE_H, MOE_I, synth.seed_for(3, 500))

    def experts(ws, N, K):
        size = nv.repack_size(N, K)
        buf = torch.empty(len(ws) * size, dtype=torch.uint8, device=device)
        for e, (p, sc, d) in enumerate(ws):
            nv.repack(torch.from_numpy(p).to(device), torch.from_numpy(sc).to(device), float(d), N, K,
                      out=buf[e * size:(e + 1) * size])
        return buf, size

    d1, sz1 = experts(fc1, 2 * MOE_I, MOE_H)
    d2, sz2 = experts(fc2, MOE_H, MOE_I)
    # four copies of the expert weights (4 x 340 MB), rotated between steps and
    # between repeated calls, so that no call finds its experts in L2
    wcopies = [(d1, d2)] + [(d1.clone(), d2.clone()) for _ in range(3)]
    calls = []
    for T in MOE_T:
        c = synth.moe_case(T, synth.seed_for(3, T), E=MOE_E, topk=MOE_TOPK, H=MOE_H, I=MOE_I, weights=(fc1, fc2))
        x = bits_tensor(c.x_bits, device)
        lg = torch.from_numpy(np.ascontiguousarray(c.logits)).to(device)
        ws = torch.empty(nv.moe_workspace_size(T, MOE_E, MOE_TOPK, MOE_H, MOE_I), dtype=torch.uint8, device=device)
        out = torch.empty((T, MOE_H), dtype=act_torch(), device=device)
        offs = torch.empty(MOE_E + 1, dtype=torch.int32, device=device)
        calls.append(dict(T=T, x=x, lg=lg, ws=ws, out=out, offs=offs, case=c))

    def call(C, w=0):
        # routing tables come back through offsets_out so the bench can count active experts
        h = nv._lib.load()
        w1, w2 = wcopies[w % len(wcopies)]
        fn = h.nvfp4_w4a16_moe_grouped_f16 if ACT == "f16" else h.nvfp4_w4a16_moe_grouped
        nv._lib.check(fn(
            nv._ptr(C["x"]), nv._ptr(C["lg"]), nv._ptr(w1), nv._ptr(w2), None, C["T"], MOE_E, MOE_TOPK,
            MOE_H, MOE_I, nv._ptr(C["out"]), None, None, None, nv._ptr(C["offs"]), nv._ptr(C["ws"]),
            C["ws"].numel(), nv._stream()))

    stream = torch.cuda.Stream(device)
    graphs = []
    with torch.cuda.stream(stream):
        for C in calls:
            call(C)
        torch.cuda.synchronize()
        assert nv.device_status() == 0
        for w in range(len(wcopies)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for C in calls:
                    call(C, w)
            graphs.append(g)
    torch.cuda.synchronize()
    for C in calls:
        # algorithmic bytes: the routed experts' FC1 + FC2 weights (0.5625 B per weight)
        # plus the BF16 input and output rows
        counts = np.diff(C["offs"].cpu().numpy())
        C["experts"] = int((counts > 0).sum())
        C["bytes"] = C["experts"] * (3 * MOE_I * MOE_H) * 9 // 16 + 2 * 2 * C["T"] * MOE_H
        C["flops"] = C["T"] * MOE_TOPK * (2 * 2 * MOE_I * MOE_H + 2 * MOE_H * MOE_I)
    bytes_step = sum(C["bytes"] for C in calls)
    flops_step = sum(C["flops"] for C in calls)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_index())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            graphs[i % len(graphs)].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_step = max_over_ranks(ev0.elapsed_time(ev1), world) / args.steps
    per = {}
    for C in calls:
        with torch.cuda.stream(stream):
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg, stream=stream):
                for i in range(12):
                    call(C, i)
            gg.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gg.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 12
        per[f"T={C['T']}"] = {"us": round(us, 2), "experts": C["experts"],
                              "GB/s": round(C["bytes"] / us / 1e3, 1), "TFLOP/s": round(C["flops"] / us / 1e6, 2)}
    pk = peaks()
    value = world * bytes_step / (ms_step * 1e-3) / 1e9
    return {
        "metric": "W4A16 NVFP4 GEMM TFLOPS & weight GB/s (1 GB300) and % of roofline",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ACT, "data": "synthetic (seeded)",
        "config": {"workload": "MoE layer E=128 top-8 H=2048 I=768 at T{1,16,256,4096}",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: the 128 experts hold 340 MB of weights, and four copies of "
                         "them are rotated between steps and between the repeated calls of the per-call timing"},
        "tflops": round(world * flops_step / (ms_step * 1e-3) / 1e12, 2),
        "roofline": {"bound": "hbm", "achieved": round(value, 2), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(value / pk["hbm"], 4), "traffic": None, "peak_source": pk["source"],
                     "kernel": "nvfp4::tc_gemm_kernel (MoE FC1 tile mode at T=4096, the largest share of a "
                               "step); T=16 and 256 run nvfp4::moe_persist_kernel, T=1 nvfp4::moe_linear_kernel",
                     "per_call": per},
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"]},
        "gpu_launches": sum(moe_launches(C["T"], MOE_E, MOE_TOPK, MOE_I) for C in calls) * args.steps,
        "_base": None,
        "_moe": (fc1, fc2, calls[0]["case"]),
    }


def gemm_launches(M, N, K, awq=False):
    """Library kernels one gemm call launches (the library's own plan: the
    GEMM, a split-K reduction pass on the tile kernels, the AWQ activation
    pass)."""
    import w4a16_nvfp4_weight_gb300 as nv
    return nv.gemm_plan(M, N, K, awq)["launches"]


def launch_count(nv, L):
    return gemm_launches(L["M"], L["N"], L["K"], L["pqs"] is not None)


def moe_launches(T, E, topk, I):
    """Kernels of one MoE call: routing + permutation (one fused kernel up to 64
    tokens, two up to 512, three chunked ones above), FC1 and FC2 (on the tile
    path plus the row gather and the two streaming waves of the experts'
    tails), combine; one token: two kernels."""
    if T == 1 and topk <= 8:
        return 2                      # single token: FC1 and FC2 (+ combine), each routing itself
    per_expert = T * topk // E
    tile = per_expert >= 32 and I % 128 == 0
    routing = 1 if T <= 64 else 2 if T <= 512 else 3
    return routing + (5 if tile else 2) + 1


def mlp_launches(T, H, I):
    """Kernels of one dense MLP call: FC1 (streaming or tile) and the FC2 GEMM."""
    return 1 + gemm_launches(T, H, I)


def kernel_timing(nv, launches, base, stream, device, reps=30):
    """Average device time per launch of each shape, from CUDA events around a
    graph of back-to-back launches that rotate over enough weight copies to
    exceed 4x L2 (so each launch streams its weights from HBM)."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size if hasattr(
        torch.cuda.get_device_properties(device), "L2_cache_size") else 128 << 20
    total_s, total_b, total_f = 0.0, 0, 0
    per = {}
    for L in launches:
        key = (L["M"], L["K"], L["N"])
        wb = weight_bytes(L["N"], L["K"])
        copies = max(2, min(64, int(np.ceil(4 * l2 / wb))))
        bufs = [L["w"]] + [nv.NVFP4Weight(L["w"].buf.clone(), L["N"], L["K"]) for _ in range(copies - 1)]
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(reps):
                    nv.gemm(L["x"], bufs[i % copies], pre_quant_scale=L["pqs"], out=L["y"], workspace=L["ws"])
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(3):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) * 1e-3 / (3 * reps)
        per[f"{key[0]}x{key[1]}x{key[2]}"] = round(sec * 1e6, 3)
        total_s += sec
        total_b += algo_bytes(*key)
        total_f += flops(*key)
        del g, bufs
    torch.cuda.empty_cache()
    return dict(seconds=total_s, bytes=total_b, flops=total_f, per_shape_us=per)


MLP_H, MLP_I = 4096, 14336
MLP_T = (1, 16, 512, 2048)


def run_mlp(args, rank, world, device, nv, synth):
    """The dense gated MLP (H=4096, I=14336: FC1 [28672 x 4096], FC2 [4096 x 14336])
    at T = 1, 16, 512, 2048 tokens, one call each per step."""
    r = synth.rng(synth.seed_for(6, 0))
    fc1 = synth.quantize(synth.normal_weight(r, 2 * MLP_I, MLP_H))
    fc2 = synth.quantize(synth.normal_weight(r, MLP_H, MLP_I))

    def rep(w, N, K):
        p, sc, d = w
        return nv.repack(torch.from_numpy(p).to(device), torch.from_numpy(sc).to(device), float(d), N, K)

    w1, w2 = rep(fc1, 2 * MLP_I, MLP_H), rep(fc2, MLP_H, MLP_I)
    # four weight copies (4 x 99 MB), rotated between steps and repeated calls
    wcopies = [(w1, w2)] + [(nv.NVFP4Weight(w1.buf.clone(), w1.N, w1.K), nv.NVFP4Weight(w2.buf.clone(), w2.N, w2.K))
                            for _ in range(3)]
    calls = []
    for T in MLP_T:
        x = bits_tensor(synth.normal_act(synth.rng(synth.seed_for(6, T)), (T, MLP_H), ACT), device)
        ws = torch.empty(nv.mlp_workspace_size(T, MLP_H, MLP_I), dtype=torch.uint8, device=device)
        out = torch.empty((T, MLP_H), dtype=act_torch(), device=device)
        calls.append(dict(T=T, x=x, ws=ws, out=out))

    def call(C, w=0):
        a, b = wcopies[w % len(wcopies)]
        nv.mlp(C["x"], a, b, out=C["out"], workspace=C["ws"])

    stream = torch.cuda.Stream(device)
    graphs = []
    with torch.cuda.stream(stream):
        for C in calls:
            call(C)
        torch.cuda.synchronize()
        assert nv.device_status() == 0
        for w in range(len(wcopies)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for C in calls:
                    call(C, w)
            graphs.append(g)
    torch.cuda.synchronize()
    wbytes = weight_bytes(2 * MLP_I, MLP_H) + weight_bytes(MLP_H, MLP_I)
    for C in calls:
        T = C["T"]
        C["bytes"] = wbytes + 2 * 2 * T * MLP_H
        C["flops"] = flops(T, 2 * MLP_I, MLP_H) + flops(T, MLP_H, MLP_I)
    bytes_step = sum(C["bytes"] for C in calls)
    flops_step = sum(C["flops"] for C in calls)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_index())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            graphs[i % len(graphs)].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_step = max_over_ranks(ev0.elapsed_time(ev1), world) / args.steps
    assert nv.device_status() == 0
    per = {}
    for C in calls:
        with torch.cuda.stream(stream):
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg, stream=stream):
                for i in range(12):
                    call(C, i)
            gg.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gg.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 12
        per[f"T={C['T']}"] = {"us": round(us, 2), "GB/s": round(C["bytes"] / us / 1e3, 1),
                              "TFLOP/s": round(C["flops"] / us / 1e6, 2)}
    pk = peaks()
    value = world * bytes_step / (ms_step * 1e-3) / 1e9
    return {
        "metric": "W4A16 NVFP4 GEMM TFLOPS & weight GB/s (1 GB300) and % of roofline",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ACT, "data": "synthetic (seeded)",
        "config": {"workload": "dense gated MLP H=4096 I=14336 at T{1,16,512,2048}",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: four copies of the 99 MB weight pair rotated between steps "
                         "and between the repeated calls of the per-call timing"},
        "tflops": round(world * flops_step / (ms_step * 1e-3) / 1e12, 2),
        "roofline": {"bound": "hbm", "achieved": round(value, 2), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(value / pk["hbm"], 4), "traffic": None, "peak_source": pk["source"],
                     "note": "whole layer per step; T=512 and 2048 are tensor-bound, see per_call"},
        "per_call": per,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"]},
        "gpu_launches": sum(mlp_launches(C["T"], MLP_H, MLP_I) for C in calls) * args.steps,
    }


def run_e2e(nv, launches, stream, args, bw_unit):
    """Same step through the public API with the activations coming from pinned
    host memory and the outputs going back to it, copies inside the timed
    region: one host-to-device copy of all of the step's activations, the
    GEMMs (nv.gemm on device views of that buffer), one device-to-host copy of
    all outputs; the step is captured in a CUDA graph, as a decode loop would
    run it."""
    def layout(shapes):
        offs, off = [], 0
        for (r, c) in shapes:
            offs.append(off)
            off += (2 * r * c + 255) // 256 * 256
        return offs, off

    xo, xbytes = layout([(L["M"], L["K"]) for L in launches])
    yo, ybytes = layout([(L["M"], L["N"]) for L in launches])
    hx = torch.empty(xbytes, dtype=torch.uint8).pin_memory()
    hy = torch.empty(ybytes, dtype=torch.uint8).pin_memory()
    dx = torch.empty(xbytes, dtype=torch.uint8, device=launches[0]["x"].device)
    dy = torch.empty(ybytes, dtype=torch.uint8, device=launches[0]["x"].device)
    xs, ys = [], []
    for L, ox, oy in zip(launches, xo, yo):
        nx, ny = 2 * L["M"] * L["K"], 2 * L["M"] * L["N"]
        hx[ox:ox + nx].copy_(L["x"].cpu().contiguous().view(torch.uint8).reshape(-1))
        xs.append(dx[ox:ox + nx].view(act_torch()).view(L["M"], L["K"]))
        ys.append(dy[oy:oy + ny].view(act_torch()).view(L["M"], L["N"]))
    steps = max(3, min(args.steps, 200))

    def step():
        dx.copy_(hx, non_blocking=True)
        for L, x, y in zip(launches, xs, ys):
            nv.gemm(x, L["w"], pre_quant_scale=L["pqs"], out=y, workspace=L["ws"])
        hy.copy_(dy, non_blocking=True)

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    # the host copy of the last step's output matches the device result
    assert torch.equal(hy, dy.cpu())
    ms = e0.elapsed_time(e1) / steps
    h2d, d2h = hx.numel(), hy.numel()          # the copied buffers (256-byte aligned slots)
    bytes_step = sum(algo_bytes(L["M"], L["N"], L["K"]) for L in launches)
    flops_step = sum(flops(L["M"], L["N"], L["K"]) for L in launches)
    v = bytes_step / (ms * 1e-3) / 1e9 if bw_unit else flops_step / (ms * 1e-3) / 1e12
    return {"value": round(v, 2), "unit": "GB/s" if bw_unit else "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms, 4), "steps": steps,
            "path": "pinned host X -> device in one copy per step, nvfp4_w4a16_gemm via the Python binding "
                    "(the step captured in a CUDA graph), device Y -> pinned host in one copy per step"}


def run_e2e_per_call(nv, launches, stream, args, bw_unit):
    """The step as a user calls it, with nothing captured: each step copies its
    activations from pinned host memory to the device (one copy), calls
    nvfp4_w4a16_gemm once per GEMM through the Python binding (argument checks,
    the launch plan, the ctypes call and the launches all run every step), and
    copies all outputs back to pinned host memory (one copy)."""
    def layout(shapes):
        offs, off = [], 0
        for (r, c) in shapes:
            offs.append(off)
            off += (2 * r * c + 255) // 256 * 256
        return offs, off

    xo, xbytes = layout([(L["M"], L["K"]) for L in launches])
    yo, ybytes = layout([(L["M"], L["N"]) for L in launches])
    dev = launches[0]["x"].device
    hx = torch.empty(xbytes, dtype=torch.uint8).pin_memory()
    hy = torch.empty(ybytes, dtype=torch.uint8).pin_memory()
    dx = torch.empty(xbytes, dtype=torch.uint8, device=dev)
    dy = torch.empty(ybytes, dtype=torch.uint8, device=dev)
    xs, ys = [], []
    for L, ox, oy in zip(launches, xo, yo):
        nx, ny = 2 * L["M"] * L["K"], 2 * L["M"] * L["N"]
        hx[ox:ox + nx].copy_(L["x"].cpu().contiguous().view(torch.uint8).reshape(-1))
        xs.append(dx[ox:ox + nx].view(act_torch()).view(L["M"], L["K"]))
        ys.append(dy[oy:oy + ny].view(act_torch()).view(L["M"], L["N"]))
    steps = max(3, min(args.steps, 200))

    def step():
        dx.copy_(hx, non_blocking=True)
        for L, x, y in zip(launches, xs, ys):
            nv.gemm(x, L["w"], pre_quant_scale=L["pqs"], out=y, workspace=L["ws"])
        hy.copy_(dy, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    assert torch.equal(hy, dy.cpu())
    ms = e0.elapsed_time(e1) / steps
    bytes_step = sum(algo_bytes(L["M"], L["N"], L["K"]) for L in launches)
    flops_step = sum(flops(L["M"], L["N"], L["K"]) for L in launches)
    v = bytes_step / (ms * 1e-3) / 1e9 if bw_unit else flops_step / (ms * 1e-3) / 1e12
    return {"value": round(v, 2), "unit": "GB/s" if bw_unit else "TFLOP/s",
            "h2d_bytes_per_step": hx.numel(), "d2h_bytes_per_step": hy.numel(),
            "ms_per_step": round(ms, 4), "steps": steps,
            "path": "every step: pinned host X -> device (one copy), one nvfp4_w4a16_gemm call per GEMM "
                    "through the Python binding (no graph capture), device Y -> pinned host (one copy)"}


# ----------------------------------------------------------- CPU baseline --
def _baseline_cases(base, rows_per_gemm):
    """The oracle's sample of the decode workload: every GEMM of a step
    restricted to a seeded subset of output rows."""
    from w4a16_nvfp4_weight_gb300 import synth

    r = synth.rng(4242)
    cases = []
    for si, (K, N) in enumerate(DECODE_SHAPES):
        if base is not None:
            _, packed, scales, d = base[(K, N)]
        else:
            packed, scales, d = synth.weight_only(K, N, synth.seed_for(1, si))
        rows = np.sort(r.choice(N, size=rows_per_gemm, replace=False))
        sub_p, sub_s = packed[rows], scales[rows]
        for M in DECODE_M:
            cases.append((M, K, sub_p, sub_s, d, synth.normal_act(r, (M, K), ACT)))
    return cases


def _oracle_sweeps(job):
    """Sweep the oracle over the sample for `seconds` (or `reps` sweeps);
    returns (algorithmic bytes, elapsed s, sweeps)."""
    cases, seconds, reps, act = job
    from oracle import dense

    rows = len(cases[0][2])
    t0 = time.perf_counter()
    n_sweeps = 0
    b = 0
    while True:
        for (M, K, p, s, d, x) in cases:
            dense.linear(x, p, s, d, True, act=act)
            b += algo_bytes(M, rows, K)
        n_sweeps += 1
        el = time.perf_counter() - t0
        if (reps is not None and n_sweeps >= reps) or (reps is None and el >= seconds):
            return b, el, n_sweeps


def cpu_baseline(seconds_target=15.0, reps=None, base=None, rows_per_gemm=256):
    """The oracle, as it stands, single-threaded on a bounded sample of the
    decode workload."""
    cases = _baseline_cases(base, rows_per_gemm)
    b, el, n_sweeps = _oracle_sweeps((cases, seconds_target, reps, ACT))
    return {"value": round(b / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_sweeps} sweep(s) of the 20 decode GEMMs restricted to {rows_per_gemm} seeded "
                      f"output rows each (numpy float64 oracle, single thread), {el:.1f} s"}


def cpu_baseline_all_cores(seconds_target=10.0, base=None, rows_per_gemm=256):
    """The same sample on every host core: one single-threaded oracle process
    per core (spawned, so no process is forked from one that holds a CUDA
    context), all sweeping at once; value = their bytes / the wall time."""
    import multiprocessing as mp

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    cores = min(cores, 64)          # each process imports torch: bound the memory and start-up
    cases = _baseline_cases(base, rows_per_gemm)
    with mp.get_context("spawn").Pool(cores) as pool:
        pool.map(_oracle_sweeps, [(cases[:1], 0.0, 1, ACT)] * cores)       # start every worker first
        t0 = time.perf_counter()
        res = pool.map(_oracle_sweeps, [(cases, seconds_target, None, ACT)] * cores, chunksize=1)
        wall = time.perf_counter() - t0
    total = sum(r[0] for r in res)
    return {"value": round(total / wall / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes x {min(r[2] for r in res)}+ sweep(s) of the single-thread sample "
                      f"(20 decode GEMMs, {rows_per_gemm} seeded output rows each), {wall:.1f} s wall"}


def cpu_baseline_dense(cases, base, bw_unit, seconds_target=12.0):
    """The oracle, single-threaded, on the prefill / LM-head / odd-shape
    workloads: every GEMM of a step with its full activations but restricted to
    a seeded subset of output rows (16 per GEMM for the byte-bound shapes, 4
    for the tensor-bound ones); value in the workload's unit."""
    from oracle import dense
    from w4a16_nvfp4_weight_gb300 import synth

    r = synth.rng(4243)
    per = 16 if bw_unit else 4
    work = []
    for (M, K, N, x_bits, pqs_bits) in cases:
        _, packed, scales, d = base[(K, N)]
        rows = np.sort(r.choice(N, size=min(per, N), replace=False))
        work.append((M, K, len(rows), packed[rows], scales[rows], d, x_bits, pqs_bits))
    t0 = time.perf_counter()
    n_sweeps, amount = 0, 0
    while True:
        for (M, K, nr, p, sc, d, x, pqs) in work:
            dense.linear(x, p, sc, d, True, pqs_bits=pqs, act=ACT)
            amount += algo_bytes(M, nr, K) if bw_unit else flops(M, nr, K)
        n_sweeps += 1
        el = time.perf_counter() - t0
        if el >= seconds_target:
            break
    return {"value": round(amount / el / (1e9 if bw_unit else 1e12), 6), "unit": "GB/s" if bw_unit else "TFLOP/s",
            "cores": 1, "kind": "oracle",
            "sample": f"{n_sweeps} sweep(s) of the {len(work)} GEMMs with full activations, {per} seeded output "
                      f"rows each (numpy float64 oracle, single thread), {el:.1f} s"}


def cpu_baseline_moe(fc1, fc2, case, seconds_target=12.0):
    """The oracle, single-threaded, on the T = 1 MoE layer (routing,
    permutation, the 8 routed experts' FC1 + SwiGLU and FC2, combine); value
    in GB/s of the routed experts' weights plus the input and output rows."""
    from oracle import moe as omoe

    w1 = [(p, sc, d, True) for (p, sc, d) in fc1]
    w2 = [(p, sc, d, True) for (p, sc, d) in fc2]
    T = case.x_bits.shape[0]
    t0 = time.perf_counter()
    n, amount = 0, 0
    while True:
        res = omoe.moe_layer(case.x_bits, case.logits, w1, w2, MOE_TOPK, act=ACT)
        experts = int((np.asarray(res["counts"]) > 0).sum())
        amount += experts * (3 * MOE_I * MOE_H) * 9 // 16 + 2 * 2 * T * MOE_H
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds_target:
            break
    return {"value": round(amount / el / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} call(s) of the whole T={T} layer ({experts} routed experts; numpy float64 oracle, "
                      f"single thread), {el:.1f} s"}


def strip_host_data(res):
    """Remove the host-side inputs run_* hands to the baselines; returns them."""
    return res.pop("_base", None), res.pop("_cases", None), res.pop("_moe", None)


def attach_cpu_baselines(res, workload, world, skip, seconds=None):
    """Time the oracle beside the GPU line (rank 0 of a one-GPU run only) and
    drop the host data; `seconds` shortens every sample (tests)."""
    base, cases, moe_host = strip_host_data(res)
    if skip or world != 1:
        return res
    kw = {} if seconds is None else {"seconds_target": seconds}
    if workload == "decode":
        res["cpu_baseline"] = cpu_baseline(base=base, **kw)
        res["cpu_baseline_all_cores"] = cpu_baseline_all_cores(base=base, **kw)
    elif workload in ("prefill", "lmhead", "tails", "toy"):
        res["cpu_baseline"] = cpu_baseline_dense(cases, base, workload != "prefill", **kw)
    elif workload == "moe":
        res["cpu_baseline"] = cpu_baseline_moe(*moe_host, **kw)
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from w4a16_nvfp4_weight_gb300 import synth
    base = {}
    for si, (K, N) in enumerate(DECODE_SHAPES):
        base[(K, N)] = (None,) + tuple(synth.weight_only(K, N, synth.seed_for(1, si)))
    # size each step's sample so the whole run stays within about 90 s
    t0 = time.perf_counter()
    cpu_baseline(reps=1, base=base, rows_per_gemm=8)
    per_row = (time.perf_counter() - t0) / 8
    rows = int(max(1, min(256, 90.0 / (args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        cpu_baseline(reps=1, base=base, rows_per_gemm=rows)
    t0 = time.perf_counter()
    res = cpu_baseline(reps=args.steps, base=base, rows_per_gemm=rows)
    el = time.perf_counter() - t0
    return {
        "metric": "W4A16 NVFP4 GEMM TFLOPS & weight GB/s (1 GB300) and % of roofline",
        "impl": "reference", "value": res["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"decode dense linears (bounded sample: {rows} output rows per GEMM)"},
        "cpu_baseline": {"value": res["value"], "unit": "GB/s", "kind": "oracle", "cores": 1,
                         "sample": res["sample"]},
        "e2e": {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_case(args):
    """One GEMM shape, 3 warm-up + 3 launches, for an ncu capture of its kernel."""
    import w4a16_nvfp4_weight_gb300 as nv
    from w4a16_nvfp4_weight_gb300 import synth
    M, K, N = (int(v) for v in args.profile.split(","))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(9, 0))
    w = nv.repack(torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda(), float(d), N, K)
    r = synth.rng(7)
    x = bits_tensor(synth.normal_act(r, (M, K), ACT), "cuda")
    pqs = bits_tensor(synth.awq_scale_bits(r, K, ACT), "cuda") if args.awq else None
    for _ in range(6):
        y = nv.gemm(x, w, pre_quant_scale=pqs)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    print(json.dumps({"profile": [M, K, N], "awq": bool(args.awq), "ok": True}))


def profile_moe_case(args):
    """The MoE layer (128 experts, top-8, hidden 2048, intermediate 768) at T
    tokens, 3 warm-up + 3 calls, for an ncu capture of its kernels."""
    import w4a16_nvfp4_weight_gb300 as nv
    from w4a16_nvfp4_weight_gb300 import synth
    T = int(args.profile_moe)
    fc1, fc2 = synth.moe_weights(MOE_E, MOE_H, MOE_I, synth.seed_for(3, 500))

    def experts(ws, N, K):
        size = nv.repack_size(N, K)
        buf = torch.empty(len(ws) * size, dtype=torch.uint8, device="cuda")
        for e, (p, sc, d) in enumerate(ws):
            nv.repack(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), float(d), N, K,
                      out=buf[e * size:(e + 1) * size])
        return buf

    d1, d2 = experts(fc1, 2 * MOE_I, MOE_H), experts(fc2, MOE_H, MOE_I)
    c = synth.moe_case(T, synth.seed_for(3, T), E=MOE_E, topk=MOE_TOPK, H=MOE_H, I=MOE_I, weights=(fc1, fc2))
    x = bits_tensor(c.x_bits, "cuda")
    lg = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    for _ in range(6):
        nv.moe_grouped(x, lg, d1, d2, MOE_TOPK, MOE_I)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    print(json.dumps({"profile_moe": T, "ok": True}))


# ------------------------------------------------------------ distributed --
def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "lmhead", "tails", "toy", "moe", "mlp"])
    ap.add_argument("--awq", action="store_true")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16"],
                    help="activation type: BF16 (default) or FP16 activations, weights and output")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None, metavar="M,K,N",
                    help="run one GEMM shape 3 times after 3 warm-ups (for ncu captures); no timing")
    ap.add_argument("--profile-moe", default=None, metavar="T",
                    help="run the MoE layer at T tokens 3 times after 3 warm-ups (for ncu captures); no timing")
    args = ap.parse_args()
    global ACT
    ACT = args.dtype
    if args.profile:
        profile_case(args)
        return
    if args.profile_moe:
        profile_moe_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("gloo")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    device = torch.device("cuda", local)
    res = run_ours(args, rank, world, device)
    if rank == 0:
        attach_cpu_baselines(res, args.workload, world, args.no_cpu_baseline)
        print(json.dumps(res), flush=True)
    else:
        strip_host_data(res)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
