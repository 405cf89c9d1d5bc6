"""Benchmark of the FP4 hot path on GB300 (one JSON line on rank 0).

Step (N = 1 workload): one pass of the FP8 activation pipeline on an
8192 x 7168 E4M3 tensor with one FP32 scale per 1x128 tile (0.5 % outlier
columns x40): direct FP8 -> MXFP4 quantization, then scaled MXFP4 -> FP8
conversion.  `value` is algorithmic GB/s of the step (bytes each kernel must
read and write, summed over both kernels) with inputs resident in HBM; input
sets rotate through 4 copies (608 MB > the 126 MB L2) so every step reads
cold data.  `e2e` is the same metric through the C ABI with pinned host
buffers: host->device copy of the step's inputs, both kernels, device->host
copy of both outputs, all inside the timed region.

The other hot-path rows are measured after the timed region and reported
under "rows": MXFP4 round trip of BF16 256x4096; NVFP4 (RHT + SR, then RNE)
of a BF16 8192x14336 gradient; block-scaled FP4 GEMM 8192^3 (MXFP4, and NVFP4
with RHT operands).

The roofline object is for the dominant kernel of the step, timed alone:
N back-to-back launches of that kernel over the rotating input sets between
two CUDA events on its stream.  Every other row flushes L2 before each timed
call by READING a buffer twice the L2 size, so the timed kernel finds no dirty
lines to write back.  CPU baselines (the oracle as it stands, on a bounded
sample) are timed for every config on one core and on all host cores, each in
a subprocess whose thread count is fixed by its environment.

--impl reference times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload and prints the same kind of line.
Multi-GPU (torchrun): every rank runs its own copy of the workload (weak
scaling, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantize/convert GB/s (frac. HBM peak); FP4 block-scaled GEMM TFLOPS vs peak"
WORKLOAD = "fp8_e4m3[8192x7168]+fp32 1x128 tile scales -> MXFP4 -> FP8_e4m3 (0.5% outlier cols x40)"
ROWS, COLS = 8192, 7168
NSETS = 4
L2_BYTES = 126 * 2 ** 20

# DRAM traffic per launch measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum)
# for the named kernel on the workload above, with a hash of the kernel's source
# files at capture time; reported as null once any of those sources has changed.
TRAFFIC = {
    "fp8_to_mx": {"bytes_per_launch": 60579584 + 2470144, "src_sha": "cc401b8614be28fe",
                  "src": ["mx_quant.cu", "common.cuh", "ring.cuh", "tc.cuh"],
                  "profile": "profiles/fp8_pipeline_8192x7168.md"},
    "mx_to_fp8": {"bytes_per_launch": 31214592 + 5374976, "src_sha": "7bb34dc406d17efc",
                  "src": ["fp4_to_fp8.cu", "common.cuh", "ring.cuh", "tc.cuh"],
                  "profile": "profiles/fp8_pipeline_8192x7168.md"},
}


def _src_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "micro_scaled_fp4_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str):
    t = TRAFFIC.get(kernel)
    if not t or t.get("src_sha") != _src_hash(t["src"]):
        return None
    return t.get("bytes_per_launch")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured (MEASURED_PEAKS.json)"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback (6.8 TB/s, 1.9 PF bf16)"}


FP4_OVER_BF16 = 13.5 / 2.25      # nominal dense FP4 : BF16 tensor ratio on GB300


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def bytes_fp8_to_mx(r, c):       # e4m3 + tile scales in, codes + E8M0 out
    return r * c + r * (c // 128) * 4 + r * c // 2 + r * (c // 32)


def bytes_mx_to_fp8(r, c):       # codes + E8M0 in, e4m3 + tile scales out
    return r * c // 2 + r * (c // 32) + r * c + r * (c // 128) * 4


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[4], f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        mx = max(r[1] for r in rows)
        load = [r for r in rows if r[0] > 0.5 * mx] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in load:
            for n, v in zip(names, r[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(load)}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def _timed_loop(fn, seconds: float, max_passes: int = 1000):
    """Runs fn until `seconds` have passed (at least once); seconds per pass, passes."""
    n = 0
    t0 = time.perf_counter()
    while True:
        fn()
        n += 1
        if time.perf_counter() - t0 >= seconds or n >= max_passes:
            break
    return (time.perf_counter() - t0) / n, n


CPU_LEGS = ("c1", "c2", "c3", "c4", "c5")


def cpu_leg(cfg: str, seconds: float, c2_rows: int = 256) -> dict:
    """The oracle as it stands on a bounded sample of one config, repeated for
    about `seconds`; the thread count is whatever this process's environment
    sets (OMP_NUM_THREADS for the C oracle's OpenMP loops, the BLAS variables
    for NumPy's float64 matmul).  Returns value / unit / sample."""
    import oracle
    from micro_scaled_fp4_gb300 import workloads as W
    oracle.build()
    if cfg == "c1":
        x = W.activation_bf16()

        def f():
            q, s = oracle.mx_quantize(x)
            oracle.mx_dequantize(q, s)
        dt, n = _timed_loop(f, seconds)
        nb = 2 * 256 * 4096 * (2 + 0.5 + 1 / 32)
        return {"value": nb / dt / 1e9, "unit": "GB/s",
                "sample": f"the whole 256x4096 round trip (quantize + dequantize), {n} passes"}
    if cfg == "c2":
        e4, ts = W.fp8_activation(c2_rows, COLS, seed=1, outlier_seed=2)

        def f():
            q, s = oracle.fp8_to_mx(e4, ts)
            oracle.mx_to_fp8(q, s)
        dt, n = _timed_loop(f, seconds)
        nb = bytes_fp8_to_mx(c2_rows, COLS) + bytes_mx_to_fp8(c2_rows, COLS)
        return {"value": nb / dt / 1e9, "unit": "GB/s",
                "sample": f"{c2_rows} of {ROWS} rows (a3 + a4), {n} passes"}
    if cfg == "c3":
        r, c = 64, 14336
        x = W.gradient_bf16(r, c)

        def f():
            am = oracle.nv_amax(x, 1, 7)
            oracle.nv_quantize(x, rht=1, rht_seed=7, rounding="sr", sr_seed=1234, amax=am)
            oracle.nv_quantize(x, rht=1, rht_seed=7, amax=am)
        dt, n = _timed_loop(f, seconds)
        nb = r * c * (2 + 2 * (2 + 0.5 + 1 / 16))
        return {"value": nb / dt / 1e9, "unit": "GB/s",
                "sample": f"{r} of 8192 rows x {c} (amax pass + SR pass + RNE pass, RHT), {n} passes"}
    if cfg == "c4":
        m = 256
        a, b = W.gemm_operands(m=m)
        qa, sa = oracle.mx_quantize(a)
        qb, sb = oracle.mx_quantize(b)
        dt, n = _timed_loop(lambda: oracle.mx_gemm_ref(qa, sa, qb, sb), seconds)
        return {"value": 2.0 * m * 8192 * 8192 / dt / 1e12, "unit": "TFLOPS",
                "sample": f"{m} of 8192 rows of A x all of B (MXFP4, dequantize + float64 matmul), {n} passes"}
    if cfg == "c5":
        import torch
        T, H, I, E, k, rows = 4096, 7168, 2048, 64, 8, 256
        x = W.moe_activations(T, H, seed=8)
        topk = W.moe_routing(tokens=T, experts=E, top_k=k, seed=9)
        w1 = W.moe_weights_torch(1, 2 * I, H, 10, "cpu")[0].view(torch.int16).numpy().view(np.uint16)
        w2 = W.moe_weights_torch(1, H, I, 11, "cpu")[0].view(torch.int16).numpy().view(np.uint16)
        r1, r2 = oracle.nv_quantize(w1), oracle.nv_quantize(w2)       # offline, not timed
        w1d = oracle.nv_dequantize_f64(r1["q"], r1["s"], r1["s_t"])
        w2d = oracle.nv_dequantize_f64(r2["q"], r2["s"], r2["s_t"])

        def f():
            qx, sx = oracle.mx_quantize(x)
            order, offs = oracle.moe_dispatch(topk, E)
            tok = order[offs[0]:offs[0] + rows]
            h = oracle.moe_up_gate(oracle.mx_dequantize_f64(qx[tok], sx[tok]), w1d, I)
            qh, sh = oracle.mx_quantize(h.astype(np.float32))
            oracle.gemm_ref(oracle.mx_dequantize_f64(qh, sh), w2d)
        dt, n = _timed_loop(f, seconds)
        flops = 2.0 * rows * H * 2 * I + 2.0 * rows * I * H
        return {"value": flops / dt / 1e12, "unit": "TFLOPS",
                "sample": f"{T} tokens quantized and routed, {rows} dispatched rows of expert 0 through "
                          f"up-proj + SiLU gate + MXFP4 of h + down-proj (float64), {n} passes"}
    raise ValueError(cfg)


def host_cores() -> int:
    return os.cpu_count() or 1


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
    except (OSError, subprocess.SubprocessError):
        return "unknown"
    for line in out.splitlines():
        if line.startswith("Model name:"):
            return line.split(":", 1)[1].strip()
    return "unknown"


def cpu_baseline(cfg: str, threads: int, seconds: float) -> dict:
    """cpu_leg in a fresh Python process whose OpenMP and BLAS thread counts are
    `threads` (set before the process starts, so they hold for the libraries
    it loads); the result as a cpu_baseline object."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-leg", cfg, "--cpu-seconds", str(seconds)]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        out = json.loads(res.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"value": None, "cores": threads, "kind": "oracle", "error": str(e)[:160]}
    return {"value": round(out["value"], 4), "unit": out["unit"], "cores": threads, "kind": "oracle",
            "sample": out["sample"]}


def cpu_baselines(cfg: str, seconds: float) -> dict:
    """The oracle on all host cores (the object's own value) and on one core."""
    allc = cpu_baseline(cfg, host_cores(), seconds)
    allc["one_core"] = cpu_baseline(cfg, 1, seconds)
    return allc


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (the job's time is its slowest
    rank's); x itself without a process group."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(nbytes_per_rank_step: int, ms_step: float, world: int) -> float:
    """GB/s of the whole job: every rank moves its own replica's bytes per step."""
    return world * nbytes_per_rank_step / ms_step / 1e6


def step_config(world: int) -> dict:
    """The workload of the step, shared by both arms."""
    nbytes = bytes_fp8_to_mx(ROWS, COLS) + bytes_mx_to_fp8(ROWS, COLS)
    return {"workload": WORKLOAD, "rows": ROWS, "cols": COLS, "parallelism": f"replicas{world}",
            "l2": f"{NSETS} rotating input sets ({NSETS * (nbytes // 2**20)} MB > L2)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    sample = 256
    for _ in range(args.warmup):
        cpu_leg("c2", 0.0, sample)
    vals, t_total = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        vals.append(cpu_leg("c2", 0.0, sample)["value"])
        t_total += time.perf_counter() - t0
    value = statistics.mean(vals)
    cores = int(os.environ.get("OMP_NUM_THREADS", host_cores()))
    desc = f"{sample} of {ROWS} rows of the workload per step (a3 + a4, scalar C oracle, OpenMP)"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": step_config(world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


ROW_NAMES = ("c1", "c3", "gemm", "moe", "col", "nv2d", "fp8")


def main_rows(fq, W, torch, peaks, which=ROW_NAMES, moe_tokens=65536):
    """The other hot-path rows, each timed with CUDA events (inputs > L2 or L2 flushed).
    `which` selects the rows: c1 (MXFP4 round trip), c3 (NVFP4 of a gradient),
    gemm (dense block-scaled GEMM), moe (MoE expert FFN), col (column path:
    FP4RowToFP8Col, column-wise quantize, Wgrad GEMM with the deterministic
    H16), nv2d (16x16-scaled NVFP4 weights), fp8 (MXFP8 GEMM on FP4 -> FP8
    outputs)."""
    rows = {}
    stream = torch.cuda.current_stream()
    # L2 flush by reading a buffer twice the L2 size: the lines it leaves are
    # clean, so the timed kernel writes back nothing that is not its own
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
    flush_out = torch.empty((), dtype=torch.int32, device="cuda")
    lib = fq.load()

    def timed(fn, iters, do_flush):
        ts = []
        for i in range(iters + 3):
            if do_flush:
                torch.amax(flush, dim=0, out=flush_out)
            e0, e1 = _events(torch, 2)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= 3:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    def b2b(launch, n=200):
        """n back-to-back launches (launch(i) picks input set i), CUDA events on
        the stream around the whole run: the streaming kernels' steady rate, as
        for the step's kernels.  Each row's sets together exceed L2, so every
        launch reads its inputs from HBM; a single call after an L2 flush also
        pays the kernel's start and drain (~3 us on a 20 us kernel)."""
        for i in range(3):
            launch(i)
        e0, e1 = _events(torch, 2)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            launch(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n
    timed.b2b = b2b

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    if "c1" in which:
        c1_row(fq, W, torch, peaks, timed, dev_bf16, rows)
    if "c3" in which:
        c3_row(fq, W, torch, peaks, timed, dev_bf16, rows)
    if "gemm" in which and getattr(lib, "fp4q_block_scaled_gemm", None) is not None:
        gemm_row(fq, W, torch, peaks, timed, dev_bf16, rows)
    if "col" in which and getattr(lib, "fp4q_fp4_row_to_fp8_col", None) is not None:
        col_rows(fq, W, torch, peaks, timed, dev_bf16, rows)
    if "nv2d" in which and getattr(lib, "fp4q_nv_quantize_2d", None) is not None:
        nv2d_row(fq, W, torch, peaks, timed, rows)
    if "fp8" in which and getattr(lib, "fp4q_fp8_tile_scales_to_e8m0", None) is not None:
        fp8_row(fq, W, torch, peaks, timed, dev_bf16, rows)
    torch.cuda.empty_cache()
    if "moe" in which and getattr(lib, "fp4q_grouped_gemm", None) is not None:
        rows[f"moe_ffn_{moe_tokens}x7168_top8_of_64"] = moe_row(fq, W, torch, peaks, timed, moe_tokens)
    return rows


def c1_row(fq, W, torch, peaks, timed, dev_bf16, rows):
    """C1: MXFP4 round trip, BF16 256x4096 (5 MB: L2-resident, launch-latency bound)."""
    stream = torch.cuda.current_stream()
    x = dev_bf16(W.activation_bf16())
    q = torch.empty((256, 2048), dtype=torch.uint8, device="cuda")
    s = torch.empty((256, 128), dtype=torch.uint8, device="cuda")
    y = torch.empty((256, 4096), dtype=torch.bfloat16, device="cuda")

    def c1():
        fq.fp4q_mx_quantize(x, fq.FP4Q_BF16, None, 256, 4096, 4096, 1, q, s, 0, stream)
        fq.fp4q_mx_dequantize(q, s, 256, 4096, 1, y, fq.FP4Q_BF16, stream)
    ms = timed(c1, 50, True)
    nb = 2 * (256 * 4096 * 2 + 256 * 2048 + 256 * 128)
    rows["mx_roundtrip_bf16_256x4096"] = {"ms": round(ms, 4), "GB_per_s": round(nb / ms / 1e6, 1),
                                          "frac_hbm": round(nb / ms / 1e6 / peaks["hbm_gbs"], 3),
                                          "note": "5.3 MB, L2 flushed before each pass; launch-latency bound"}
    g = graph_c1 = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(20):
                fq.fp4q_mx_quantize(x, fq.FP4Q_BF16, None, 256, 4096, 4096, 1, q, s, 0,
                                    torch.cuda.current_stream())
                fq.fp4q_mx_dequantize(q, s, 256, 4096, 1, y, fq.FP4Q_BF16, torch.cuda.current_stream())
        ms_g = timed(g.replay, 20, False) / 20
        rows["mx_roundtrip_bf16_256x4096"]["graph_ms"] = round(ms_g, 4)
        rows["mx_roundtrip_bf16_256x4096"]["graph_GB_per_s"] = round(nb / ms_g / 1e6, 1)
    except Exception as e:  # noqa: BLE001 - graph capture is an optional extra figure
        rows["mx_roundtrip_bf16_256x4096"]["graph_error"] = str(e)[:120]
    del x, q, s, y, g, graph_c1


def c3_row(fq, W, torch, peaks, timed, dev_bf16, rows):
    """C3: NVFP4 of a BF16 8192x14336 Student-t gradient, RHT, SR then RNE (235 MB > L2)."""
    stream = torch.cuda.current_stream()
    R3, C3 = 8192, 14336
    xg = dev_bf16(W.gradient_bf16(R3, C3))
    q3 = torch.empty((R3, C3 // 2), dtype=torch.uint8, device="cuda")
    s3 = torch.empty((R3, C3 // 16), dtype=torch.uint8, device="cuda")
    st = torch.empty(1, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")

    def c3(rounding, amax_in=None):
        fq.fp4q_nv_quantize(xg, R3, C3, C3, 1, 1, 7, rounding, 1234, amax_in, am, st, q3, s3, 0, ws, 256, stream)
    b_amax = R3 * C3 * 2
    b_quant = R3 * C3 * 2 + R3 * C3 // 2 + R3 * C3 // 16
    ms_sr = timed(lambda: c3(fq.FP4Q_SR), 10, True)
    ms_rne = timed(lambda: c3(fq.FP4Q_RNE), 10, True)
    amax_dev = am.clone()
    ms_sr1 = timed(lambda: c3(fq.FP4Q_SR, amax_dev), 10, True)
    ms_rne1 = timed(lambda: c3(fq.FP4Q_RNE, amax_dev), 10, True)
    # both roundings from one read (fp4q_nv_quantize_sr_rne): the amax pass plus
    # one quantize pass writing the SR and the RNE codes over one set of scales
    q3b = torch.empty_like(q3)

    def c3_both(amax_in=None):
        fq.fp4q_nv_quantize_sr_rne(xg, R3, C3, C3, 1, 7, 1234, amax_in, am, st, q3, q3b, s3, 0, ws, 256, stream)
    b_both = R3 * C3 * 2 + 2 * (R3 * C3 // 2) + R3 * C3 // 16
    ms_both = timed(c3_both, 10, True)
    ms_both1 = timed(lambda: c3_both(amax_dev), 10, True)
    # back to back (the 235 MB input exceeds L2)
    hbm = peaks["hbm_gbs"]
    bb_rne1 = timed.b2b(lambda i: c3(fq.FP4Q_RNE, amax_dev), 100)
    bb_both1 = timed.b2b(lambda i: c3_both(amax_dev), 100)
    rows["nvfp4_rht_8192x14336"] = {
        "back_to_back": {"rne_quant_pass_ms": round(bb_rne1, 4),
                         "frac_hbm_rne_quant_pass": round(b_quant / bb_rne1 / 1e6 / hbm, 3),
                         "sr_rne_quant_pass_ms": round(bb_both1, 4),
                         "frac_hbm_sr_rne_quant_pass": round(b_both / bb_both1 / 1e6 / hbm, 3)},
        "sr_and_rne_one_call_ms": round(ms_both, 4),
        "sr_and_rne_one_call_GB_per_s": round((b_amax + b_both) / ms_both / 1e6, 1),
        "sr_and_rne_separate_calls_ms": round(ms_sr + ms_rne, 4),
        "sr_rne_quant_pass_ms": round(ms_both1, 4),
        "sr_rne_quant_pass_GB_per_s": round(b_both / ms_both1 / 1e6, 1),
        "frac_hbm_sr_rne_quant_pass": round(b_both / ms_both1 / 1e6 / peaks["hbm_gbs"], 3),
        "sr_two_pass_ms": round(ms_sr, 4), "rne_two_pass_ms": round(ms_rne, 4),
        "sr_two_pass_GB_per_s": round((b_amax + b_quant) / ms_sr / 1e6, 1),
        "rne_two_pass_GB_per_s": round((b_amax + b_quant) / ms_rne / 1e6, 1),
        "sr_quant_pass_ms": round(ms_sr1, 4), "rne_quant_pass_ms": round(ms_rne1, 4),
        "sr_quant_pass_GB_per_s": round(b_quant / ms_sr1 / 1e6, 1),
        "rne_quant_pass_GB_per_s": round(b_quant / ms_rne1 / 1e6, 1),
        "frac_hbm_rne_quant_pass": round(b_quant / ms_rne1 / 1e6 / peaks["hbm_gbs"], 3),
        "frac_hbm_sr_quant_pass": round(b_quant / ms_sr1 / 1e6 / peaks["hbm_gbs"], 3)}
    del xg, q3, q3b, s3


def gemm_row(fq, W, torch, peaks, timed, dev_bf16, rows):
    """C4: block-scaled GEMM 8192^3, MXFP4 and NVFP4 (RHT), BF16 out."""
    stream = torch.cuda.current_stream()
    a, b = W.gemm_operands()
    ad, bd = dev_bf16(a), dev_bf16(b)
    qa, sa = fq.mx_quantize(ad, layout=fq.FP4Q_SCALES_MMA)
    qb, sb = fq.mx_quantize(bd, layout=fq.FP4Q_SCALES_MMA)
    ms_qa = timed(lambda: fq.mx_quantize(ad, layout=fq.FP4Q_SCALES_MMA), 10, True)
    D = torch.empty((8192, 8192), dtype=torch.bfloat16, device="cuda")
    A = fq.make_operand(qa, sa, fq.FP4Q_MXFP4)
    B = fq.make_operand(qb, sb, fq.FP4Q_MXFP4)
    flops = 2.0 * 8192 ** 3
    ms_mx = timed(lambda: fq.fp4q_block_scaled_gemm(A, B, 8192, 8192, 8192, D, fq.FP4Q_BF16, 8192, stream), 10,
                  True)
    ra = fq.nv_quantize(ad, rht=True, rht_seed=7, layout=fq.FP4Q_SCALES_MMA)
    rb = fq.nv_quantize(bd, rht=True, rht_seed=7, layout=fq.FP4Q_SCALES_MMA)
    An = fq.make_operand(ra["q"], ra["scales"], fq.FP4Q_NVFP4, ra["s_t"])
    Bn = fq.make_operand(rb["q"], rb["scales"], fq.FP4Q_NVFP4, rb["s_t"])
    ms_nv = timed(lambda: fq.fp4q_block_scaled_gemm(An, Bn, 8192, 8192, 8192, D, fq.FP4Q_BF16, 8192, stream),
                  10, True)
    peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    rows["gemm_fp4_8192^3"] = {
        "mxfp4_ms": round(ms_mx, 4), "mxfp4_TFLOPS": round(flops / ms_mx / 1e9, 1),
        "mxfp4_frac_peak": round(flops / ms_mx / 1e9 / peak, 3),
        "nvfp4_ms": round(ms_nv, 4), "nvfp4_TFLOPS": round(flops / ms_nv / 1e9, 1),
        "nvfp4_frac_peak": round(flops / ms_nv / 1e9 / peak, 3),
        "peak_TFLOPS": round(peak, 1),
        "peak_source": f"{peaks['source']} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16)",
        "mx_quantize_operand_ms": round(ms_qa, 4)}
    del ad, bd, qa, sa, qb, sb, D, ra, rb


def col_rows(fq, W, torch, peaks, timed, dev_bf16, rows):
    """Column path (the weight-gradient operands): FP4RowToFP8Col on the FP8
    activation's MXFP4 form (8192x7168), column-wise NVFP4 of the 8192x14336
    gradient with the deterministic H16 (SR and RNE passes) and column-wise
    MXFP4 of a BF16 8192x8192 tensor, and the Wgrad GEMM dW = dY^T X
    (8192 tokens, 8192 x 8192) on column-wise H16 NVFP4 operands."""
    hbm = peaks["hbm_gbs"]
    stream = torch.cuda.current_stream()
    e4, ts = W.fp8_activation(ROWS, COLS)
    x8, t8 = torch.from_numpy(e4).cuda(), torch.from_numpy(ts).cuda()
    q, s = fq.mx_quantize(x8, tile_scale=t8)
    y = torch.empty((COLS, ROWS), dtype=torch.uint8, device="cuda")
    yt = torch.empty((COLS, ROWS // 128), dtype=torch.float32, device="cuda")
    ms = timed(lambda: fq.fp4q_fp4_row_to_fp8_col(q, s, ROWS, COLS, y, yt, stream), 10, True)
    nb = bytes_mx_to_fp8(ROWS, COLS)
    row_ms = timed(lambda: fq.fp4q_fp4_to_fp8(q, s, ROWS, COLS, 1, y, yt, stream), 10, True)
    # back to back over NSETS copies of the input (NSETS x 31 MB in, 59 MB out per launch)
    sets = [(q, s)] + [(q.clone(), s.clone()) for _ in range(NSETS - 1)]
    bb = timed.b2b(lambda i: fq.fp4q_fp4_row_to_fp8_col(sets[i % NSETS][0], sets[i % NSETS][1], ROWS, COLS, y, yt,
                                                       stream))
    rows["f1_fp4_row_to_fp8_col_8192x7168"] = {
        "back_to_back": {"ms": round(bb, 4), "GB_per_s": round(nb / bb / 1e6, 1),
                         "frac_hbm": round(nb / bb / 1e6 / hbm, 3)},
        "ms": round(ms, 4), "GB_per_s": round(nb / ms / 1e6, 1), "frac_hbm": round(nb / ms / 1e6 / hbm, 3),
        "row_layout_ms": round(row_ms, 4), "row_layout_GB_per_s": round(nb / row_ms / 1e6, 1)}
    del x8, t8, q, s, y, yt, sets

    # the same on ragged expert groups: the 2048-wide expert activation of 8192
    # tokens routed top-8 over 64 experts (65536 dispatched rows), each group
    # padded to whole 128-row tiles in the output
    topk = W.moe_routing(tokens=8192, experts=64, top_k=8, seed=33)
    goffs = np.zeros(65, dtype=np.int64)
    goffs[1:] = np.cumsum(np.bincount(topk.reshape(-1), minlength=64))
    RG, CG = int(goffs[-1]), 2048
    tiles = int(sum((goffs[g + 1] - goffs[g] + 127) // 128 for g in range(64)))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(36)
    gsets = [(torch.randint(0, 256, (RG, CG // 2), dtype=torch.uint8, device="cuda", generator=gen),
              torch.randint(110, 140, (RG, CG // 32), dtype=torch.uint8, device="cuda", generator=gen))
             for _ in range(NSETS)]
    go = torch.from_numpy(goffs).cuda()
    ld = fq.fp4q_fp4_row_to_fp8_col_grouped_ld(RG, 64)
    gy = torch.empty((CG, ld), dtype=torch.uint8, device="cuda")
    gt = torch.empty((CG, ld // 128), dtype=torch.float32, device="cuda")
    nbg = RG * (CG // 2 + CG // 32) + CG * 128 * tiles + 4 * CG * tiles
    gms = timed(lambda: fq.fp4q_fp4_row_to_fp8_col_grouped(gsets[0][0], gsets[0][1], RG, CG, go, 64, gy, gt,
                                                           stream), 10, True)
    gbb = timed.b2b(lambda i: fq.fp4q_fp4_row_to_fp8_col_grouped(gsets[i % NSETS][0], gsets[i % NSETS][1], RG, CG,
                                                                 go, 64, gy, gt, stream))
    rows["f1_fp4_row_to_fp8_col_grouped_65536x2048_64experts"] = {
        "back_to_back": {"ms": round(gbb, 4), "GB_per_s": round(nbg / gbb / 1e6, 1),
                         "frac_hbm": round(nbg / gbb / 1e6 / hbm, 3)},
        "ms": round(gms, 4), "GB_per_s": round(nbg / gms / 1e6, 1), "frac_hbm": round(nbg / gms / 1e6 / hbm, 3),
        "tiles": tiles, "bytes": nbg}
    del gsets, go, gy, gt

    R3, C3 = 8192, 14336
    xg = dev_bf16(W.gradient_bf16(R3, C3))
    q3 = torch.empty((C3, R3 // 2), dtype=torch.uint8, device="cuda")
    s3 = torch.empty((C3, R3 // 16), dtype=torch.uint8, device="cuda")
    st = torch.empty(1, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")

    def c3col(rounding, amax_in=None):
        fq.fp4q_nv_quantize(xg, R3, C3, C3, 0, 2, 0, rounding, 1234, amax_in, am, st, q3, s3, 0, ws, 256, stream)
    b_amax = R3 * C3 * 2
    b_quant = R3 * C3 * 2 + R3 * C3 // 2 + R3 * C3 // 16
    ms_sr = timed(lambda: c3col(fq.FP4Q_SR), 10, True)
    ms_rne = timed(lambda: c3col(fq.FP4Q_RNE), 10, True)
    amax_dev = am.clone()
    ms_sr1 = timed(lambda: c3col(fq.FP4Q_SR, amax_dev), 10, True)
    ms_rne1 = timed(lambda: c3col(fq.FP4Q_RNE, amax_dev), 10, True)
    bb_rne1 = timed.b2b(lambda i: c3col(fq.FP4Q_RNE, amax_dev), 100)       # 235 MB input > L2
    rows["f1_f3_nvfp4_col_h16_8192x14336"] = {
        "back_to_back": {"rne_quant_pass_ms": round(bb_rne1, 4),
                         "frac_hbm_rne_quant_pass": round(b_quant / bb_rne1 / 1e6 / hbm, 3)},
        "sr_two_pass_ms": round(ms_sr, 4), "rne_two_pass_ms": round(ms_rne, 4),
        "sr_quant_pass_GB_per_s": round(b_quant / ms_sr1 / 1e6, 1),
        "rne_quant_pass_GB_per_s": round(b_quant / ms_rne1 / 1e6, 1),
        "rne_two_pass_GB_per_s": round((b_amax + b_quant) / ms_rne / 1e6, 1),
        "frac_hbm_rne_quant_pass": round(b_quant / ms_rne1 / 1e6 / hbm, 3),
        "frac_hbm_sr_quant_pass": round(b_quant / ms_sr1 / 1e6 / hbm, 3)}
    del xg, q3, s3

    a, b = W.gemm_operands()
    ad, bd = dev_bf16(a), dev_bf16(b)
    qa = torch.empty((8192, 4096), dtype=torch.uint8, device="cuda")
    sa = torch.empty((8192, 256), dtype=torch.uint8, device="cuda")
    ms_mx = timed(lambda: fq.fp4q_mx_quantize(ad, fq.FP4Q_BF16, None, 8192, 8192, 8192, 0, qa, sa, 0, stream), 10,
                  True)
    nbq = 8192 * 8192 * (2 + 0.5 + 1 / 32)
    ad2 = ad.clone()                                                        # two 134 MB inputs
    bb_mx = timed.b2b(lambda i: fq.fp4q_mx_quantize(ad if i % 2 == 0 else ad2, fq.FP4Q_BF16, None, 8192, 8192, 8192, 0,
                                                    qa, sa, 0, stream), 100)
    del ad2
    rows["f1_mxfp4_col_bf16_8192x8192"] = {"back_to_back": {"ms": round(bb_mx, 4),
                                                            "frac_hbm": round(nbq / bb_mx / 1e6 / hbm, 3)},
                                           "ms": round(ms_mx, 4), "GB_per_s": round(nbq / ms_mx / 1e6, 1),
                                           "frac_hbm": round(nbq / ms_mx / 1e6 / hbm, 3)}
    # Wgrad: tokens along K for both operands (rows of a and b are the tokens here)
    ra = fq.nv_quantize(ad, rht=2, layout=fq.FP4Q_SCALES_MMA, block_axis=0)
    rb = fq.nv_quantize(bd, rht=2, layout=fq.FP4Q_SCALES_MMA, block_axis=0)
    D = torch.empty((8192, 8192), dtype=torch.bfloat16, device="cuda")
    An = fq.make_operand(ra["q"], ra["scales"], fq.FP4Q_NVFP4, ra["s_t"])
    Bn = fq.make_operand(rb["q"], rb["scales"], fq.FP4Q_NVFP4, rb["s_t"])
    ms_g = timed(lambda: fq.fp4q_block_scaled_gemm(An, Bn, 8192, 8192, 8192, D, fq.FP4Q_BF16, 8192, stream), 10, True)
    peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    flops = 2.0 * 8192 ** 3
    rows["f3_wgrad_h16_gemm_8192^3"] = {"ms": round(ms_g, 4), "TFLOPS": round(flops / ms_g / 1e9, 1),
                                        "frac_peak": round(flops / ms_g / 1e9 / peak, 3)}
    del ad, bd, qa, sa, ra, rb, D


def fp8_row(fq, W, torch, peaks, timed, dev_bf16, rows):
    """The FP8 consumer: C4's operands stored MXFP4, expanded to FP8 by the
    bit-remap conversion, multiplied as MXFP8 (kind::mxf8f6f4) 8192^3."""
    stream = torch.cuda.current_stream()
    a, b = W.gemm_operands()
    qa, sa = fq.mx_quantize(dev_bf16(a))
    qb, sb = fq.mx_quantize(dev_bf16(b))
    ya, tsa = fq.fp4_to_fp8(qa, sa)
    yb, tsb = fq.fp4_to_fp8(qb, sb)
    ea, eb = fq.fp8_mma_scales(tsa), fq.fp8_mma_scales(tsb)
    D = torch.empty((8192, 8192), dtype=torch.bfloat16, device="cuda")
    A = fq.make_operand(ya, ea, fq.FP4Q_MXFP8)
    B = fq.make_operand(yb, eb, fq.FP4Q_MXFP8)
    ms = timed(lambda: fq.fp4q_block_scaled_gemm(A, B, 8192, 8192, 8192, D, fq.FP4Q_BF16, 8192, stream), 10, True)
    ms_s = timed(lambda: fq.fp4q_fp8_tile_scales_to_e8m0(tsa, 8192, 8192, ea, fq.FP4Q_SCALES_MMA, stream), 10, True)
    peak8 = peaks["bf16_tflops"] * 2.0
    flops = 2.0 * 8192 ** 3
    rows["f4_mxfp8_gemm_8192^3"] = {"ms": round(ms, 4), "TFLOPS": round(flops / ms / 1e9, 1),
                                    "frac_peak_fp8": round(flops / ms / 1e9 / peak8, 3),
                                    "peak_TFLOPS": round(peak8, 1),
                                    "peak_source": f"{peaks['source']} bf16 burst x 2 (nominal FP8:BF16)",
                                    "scale_conversion_ms": round(ms_s, 4)}
    del qa, sa, qb, sb, ya, yb, D


def nv2d_row(fq, W, torch, peaks, timed, rows):
    """16x16-scaled NVFP4 of BF16 weights: one expert's W1 slab, 4096 x 7168,
    times 8 (a 32768 x 7168 stack), RNE, two passes and quantize pass."""
    stream = torch.cuda.current_stream()
    R, C = 8 * 4096, 7168
    w = W.moe_weights_torch(1, R, C, 10, "cuda")[0]
    q = torch.empty((R, C // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((R, C // 16), dtype=torch.uint8, device="cuda")
    st = torch.empty(1, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    ms2 = timed(lambda: fq.fp4q_nv_quantize_2d(w, R, C, C, fq.FP4Q_RNE, 0, None, am, st, q, s, 0, ws, 256, stream),
                10, True)
    amax_dev = am.clone()
    ms1 = timed(lambda: fq.fp4q_nv_quantize_2d(w, R, C, C, fq.FP4Q_RNE, 0, amax_dev, am, st, q, s, 0, ws, 256,
                                               stream), 10, True)
    b_quant = R * C * (2 + 0.5 + 1 / 16)
    bb1 = timed.b2b(lambda i: fq.fp4q_nv_quantize_2d(w, R, C, C, fq.FP4Q_RNE, 0, amax_dev, am, st, q, s, 0, ws, 256,
                                                     stream), 50)           # 470 MB input > L2
    rows["f2_nvfp4_2d_weights_32768x7168"] = {
        "back_to_back": {"quant_pass_ms": round(bb1, 4),
                         "frac_hbm_quant_pass": round(b_quant / bb1 / 1e6 / peaks["hbm_gbs"], 3)},
        "two_pass_ms": round(ms2, 4), "quant_pass_ms": round(ms1, 4),
        "quant_pass_GB_per_s": round(b_quant / ms1 / 1e6, 1),
        "frac_hbm_quant_pass": round(b_quant / ms1 / 1e6 / peaks["hbm_gbs"], 3)}
    del w, q, s


def moe_row(fq, W, torch, peaks, timed, T=65536):
    """MoE expert FFN forward in FP4: T tokens x 7168, top-8 of 64 experts
    (Zipf 1.1), experts 7168 -> 2x2048 (SiLU gate) -> 7168, NVFP4 weights."""
    H, I, E, k = 7168, 2048, 64, 8
    R = T * k
    stream = torch.cuda.current_stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(8)
    x = torch.randn((T, H), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    topk = torch.from_numpy(W.moe_routing(tokens=T, experts=E, top_k=k, seed=9)).cuda()
    w1 = W.moe_weights_torch(E, 2 * I, H, 10, "cuda")
    w2 = W.moe_weights_torch(E, H, I, 11, "cuda")

    def quant_weights(w, rows, cols):
        q = torch.empty((E * rows, cols // 2), dtype=torch.uint8, device="cuda")
        per = fq.fp4q_scales_bytes(rows, cols // 16, fq.FP4Q_SCALES_MMA)
        sc = torch.empty(E * per, dtype=torch.uint8, device="cuda")
        st = torch.empty(E, dtype=torch.float32, device="cuda")
        wsb = fq.fp4q_nv_quantize_workspace_bytes(rows, cols)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        for e in range(E):
            fq.fp4q_nv_quantize(w[e], rows, cols, cols, 1, 0, 0, fq.FP4Q_RNE, 0, None, None, st.data_ptr() + 4 * e,
                                q.data_ptr() + e * rows * (cols // 2), sc.data_ptr() + e * per, fq.FP4Q_SCALES_MMA,
                                ws, wsb, stream)
        return q, sc, st
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    w1q, w1s, w1t = quant_weights(w1, 2 * I, H)
    w2q, w2s, w2t = quant_weights(w2, H, I)
    e1.record(stream)
    torch.cuda.synchronize()
    wq_ms = e0.elapsed_time(e1)
    del w1, w2
    torch.cuda.empty_cache()

    # buffers
    xq = torch.empty((T, H // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int64, device="cuda")
    rtok = torch.empty(R, dtype=torch.int32, device="cuda")
    dq = torch.empty((R, H // 2), dtype=torch.uint8, device="cuda")
    ds = torch.empty((R, H // 32), dtype=torch.uint8, device="cuda")
    wsb = fq.fp4q_moe_dispatch_workspace_bytes(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    ue1 = torch.empty(fq.fp4q_rebased_scales_bytes(R, H, E), dtype=torch.uint8, device="cuda")
    rs1 = torch.empty(R, dtype=torch.float32, device="cuda")
    hq = torch.empty((R, I // 2), dtype=torch.uint8, device="cuda")
    hs = torch.empty((R, I // 32), dtype=torch.uint8, device="cuda")
    ue2 = torch.empty(fq.fp4q_rebased_scales_bytes(R, I, E), dtype=torch.uint8, device="cuda")
    rs2 = torch.empty(R, dtype=torch.float32, device="cuda")
    y = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
    viol = torch.zeros(2, dtype=torch.int32, device="cuda")

    stages = [
        ("a1_quantize_tokens", lambda: fq.fp4q_mx_quantize(x, fq.FP4Q_BF16, None, T, H, H, 1, xq, xs, 0, stream)),
        ("a9_dispatch", lambda: fq.fp4q_moe_dispatch(topk, T, k, E, xq, xs, H, offs, rtok, dq, ds, ws, wsb, stream)),
        ("rebase_tokens", lambda: fq.fp4q_mx_rebase_scales(ds, R, H, offs, E, ue1, rs1, viol, stream)),
        ("a10_up_silu_gate_mxfp4", lambda: fq.fp4q_grouped_gemm(dq, ue1, rs1, w1q, w1s, w1t, offs, R, E, 2 * I, H,
                                                              fq.FP4Q_EPI_SILU_GATE_MXFP4, hq, hs, None, stream)),
        ("rebase_h", lambda: fq.fp4q_mx_rebase_scales(hs, R, I, offs, E, ue2, rs2, viol[1:], stream)),
        ("a11_down", lambda: fq.fp4q_grouped_gemm(hq, ue2, rs2, w2q, w2s, w2t, offs, R, E, H, I,
                                                fq.FP4Q_EPI_STORE_BF16, y, None, None, stream)),
    ]
    for _, fn in stages:          # warm-up pass (the dispatch must precede the rest)
        fn()
    torch.cuda.synchronize()
    out = {}
    total = 0.0
    for name, fn in stages:
        ms = timed(fn, 5, True)
        out[name + "_ms"] = round(ms, 4)
        total += ms
    f_up = 2.0 * R * H * (2 * I)
    f_down = 2.0 * R * I * H
    peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    out["total_ms"] = round(total, 4)
    out["TFLOPS_end_to_end"] = round((f_up + f_down) / total / 1e9, 1)
    out["up_TFLOPS"] = round(f_up / out["a10_up_silu_gate_mxfp4_ms"] / 1e9, 1)
    out["down_TFLOPS"] = round(f_down / out["a11_down_ms"] / 1e9, 1)
    out["up_frac_peak"] = round(f_up / out["a10_up_silu_gate_mxfp4_ms"] / 1e9 / peak, 3)
    out["down_frac_peak"] = round(f_down / out["a11_down_ms"] / 1e9 / peak, 3)
    nb_q = T * H * 2 + T * H // 2 + T * H // 32
    out["a1_GB_per_s"] = round(nb_q / out["a1_quantize_tokens_ms"] / 1e6, 1)
    nb_d = 2 * R * (H // 2 + H // 32) + T * k * 4
    out["a9_GB_per_s"] = round(nb_d / out["a9_dispatch_ms"] / 1e6, 1)
    out["rebase_violations"] = int(viol.sum().item())
    out["weight_quantize_ms_offline"] = round(wq_ms, 3)
    out["tokens_per_expert_min_max"] = [int(v) for v in torch.diff(offs).aminmax()]
    return out


def run_gpu(args, rank, world):
    import torch
    import micro_scaled_fp4_gb300.fp4q as fq
    from micro_scaled_fp4_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    fq.load()
    peaks = _peaks()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    # ---- inputs: NSETS rotating copies, resident in HBM ----
    e4, ts = W.fp8_activation(ROWS, COLS)
    stream = torch.cuda.current_stream()
    sets = []
    for i in range(NSETS):
        x = torch.from_numpy(e4).cuda()
        t = torch.from_numpy(ts).cuda()
        q = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device="cuda")
        s = torch.empty((ROWS, COLS // 32), dtype=torch.uint8, device="cuda")
        y = torch.empty((ROWS, COLS), dtype=torch.uint8, device="cuda")
        yt = torch.empty((ROWS, COLS // 128), dtype=torch.float32, device="cuda")
        sets.append((x, t, q, s, y, yt))

    def a3(i):
        x, t, q, s, y, yt = sets[i % NSETS]
        fq.fp4q_mx_quantize(x, fq.FP4Q_E4M3, t, ROWS, COLS, COLS, 1, q, s, fq.FP4Q_SCALES_ROWMAJOR, stream)

    def a4(i):
        x, t, q, s, y, yt = sets[i % NSETS]
        fq.fp4q_fp4_to_fp8(q, s, ROWS, COLS, 1, y, yt, stream)

    def step(i):
        a3(i)
        a4(i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = _events(torch, 1)[0]
    t_end = _events(torch, 1)[0]
    wall0 = time.perf_counter()
    t_start.record(stream)
    for i in range(args.steps):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, dist, "cuda")
    ms_step = ms_total / args.steps
    nbytes = bytes_fp8_to_mx(ROWS, COLS) + bytes_mx_to_fp8(ROWS, COLS)
    value = whole_job_gbs(nbytes, ms_step, world)

    # ---- each kernel alone: n back-to-back launches over the rotating sets,
    # CUDA events on the launching stream around the whole run ----
    def alone(launch, n):
        for i in range(3):
            launch(i)
        e0, e1 = _events(torch, 2)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            launch(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n
    n_alone = max(100, min(args.steps, 2000))
    a3_ms = alone(a3, n_alone)
    a4_ms = alone(a4, n_alone)

    # ---- e2e through the C ABI with pinned host buffers ----
    hx = torch.from_numpy(e4).pin_memory()
    ht = torch.from_numpy(ts).pin_memory()
    hq = torch.empty((ROWS, COLS // 2), dtype=torch.uint8).pin_memory()
    hs = torch.empty((ROWS, COLS // 32), dtype=torch.uint8).pin_memory()
    hy = torch.empty((ROWS, COLS), dtype=torch.uint8).pin_memory()
    hyt = torch.empty((ROWS, COLS // 128), dtype=torch.float32).pin_memory()
    # one call of the library's host-buffer entry point per step: chunked
    # copies in and out overlapped with the two conversions on three streams
    del sets
    torch.cuda.empty_cache()
    wsb = fq.fp4q_fp8_pipeline_host_workspace_bytes(COLS, args.e2e_chunk)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def e2e_step():
        fq.fp4q_fp8_pipeline_host(hx, ht, ROWS, COLS, hq, hs, hy, hyt, args.e2e_chunk, ws, wsb, stream)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = _events(torch, 2)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda") / e2e_steps
    h2d = hx.numel() + ht.numel() * 4
    d2h = hq.numel() + hs.numel() + hy.numel() + hyt.numel() * 4
    clk = clocks.stop()

    # ---- roofline of the dominant kernel ----
    dom = ("fp8_to_mx", a3_ms, bytes_fp8_to_mx(ROWS, COLS), "mx_quant.cu") if a3_ms >= a4_ms else \
          ("mx_to_fp8", a4_ms, bytes_mx_to_fp8(ROWS, COLS), "fp4_to_fp8.cu")
    achieved = dom[2] / dom[1] / 1e6
    if dom[1] > ms_step:
        print(f"bench: the dominant kernel alone ({dom[1]:.5f} ms) is slower than the whole step "
              f"({ms_step:.5f} ms)", file=sys.stderr)
    roof = {"kernel": dom[0], "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 3), "traffic": _traffic(dom[0]),
            "algorithmic_bytes_per_launch": dom[2], "ms_per_launch": round(dom[1], 5),
            "timing": f"{n_alone} back-to-back launches of the kernel alone over the {NSETS} rotating input sets, "
                      "CUDA events on its stream around the whole run",
            "kernel_ms_within_step": bool(dom[1] <= ms_step),
            "peak_source": peaks["source"],
            "kernels": {"fp8_to_mx": {"ms": round(a3_ms, 5), "GB_per_s": round(bytes_fp8_to_mx(ROWS, COLS) / a3_ms / 1e6, 1)},
                        "mx_to_fp8": {"ms": round(a4_ms, 5), "GB_per_s": round(bytes_mx_to_fp8(ROWS, COLS) / a4_ms / 1e6, 1)}}}

    rows = None
    cpu = None
    if rank == 0 and not args.no_rows:
        del ws
        torch.cuda.empty_cache()
        rows = main_rows(fq, W, torch, peaks, args.rows.split(","), args.moe_tokens)
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baselines("c2", args.cpu_seconds)
        if rows is not None:
            for key, cfg in (("mx_roundtrip_bf16_256x4096", "c1"), ("nvfp4_rht_8192x14336", "c3"),
                             ("gemm_fp4_8192^3", "c4"), (f"moe_ffn_{args.moe_tokens}x7168_top8_of_64", "c5")):
                if key in rows:
                    rows[key]["cpu_baseline"] = cpu_baselines(cfg, args.cpu_seconds)
    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": step_config(world),
            "frac_hbm": round(value / world / peaks["hbm_gbs"], 3),
            "host": {"nproc": host_cores(), "cpu": _cpu_model()},
            "wall_s_timed_region": round(wall, 4),
            "e2e": {"value": round(whole_job_gbs(nbytes, e2e_ms, world), 1), "unit": "GB/s",
                    "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
                    "call": "fp4q_fp8_pipeline_host", "chunk_rows": args.e2e_chunk},
            "gpu_launches": 2 * args.steps, "roofline": roof, "cpu_baseline": cpu, "clocks": clk, "rows": rows}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="fp4q", choices=["fp4q", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="skip the other hot-path rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--rows", default=",".join(ROW_NAMES),
                    help="comma-separated rows to report besides the step: " + ", ".join(ROW_NAMES))
    ap.add_argument("--moe-tokens", type=int, default=65536, help="tokens of the MoE row")
    ap.add_argument("--e2e-chunk", type=int, default=2048, help="rows per chunk of the host-buffer (e2e) call")
    ap.add_argument("--cpu-seconds", type=float, default=4.0, help="seconds of oracle work per CPU baseline leg")
    ap.add_argument("--cpu-leg", choices=CPU_LEGS, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_leg:
        print(json.dumps(cpu_leg(args.cpu_leg, args.cpu_seconds)), flush=True)
        return
    bad = [r for r in args.rows.split(",") if r not in ROW_NAMES]
    if bad:
        ap.error(f"unknown rows {bad}")
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)


if __name__ == "__main__":
    main()
