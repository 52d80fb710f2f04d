#!/usr/bin/env python3
"""Benchmark of the NVFP4 quantized linear layer on one GB300.

A step is one pass of the whole hot path over one batch of the FFN up-projection
shaped like the 5120-hidden model of the NVFP4 pretraining news page (¶1):
M = 8192 tokens, K = 5120, N = 20480, bf16 inputs X ~ N(0,1), W ~ N(0,0.02),
dY ~ N(0,1e-3):
  quantize W (16x16, RNE, with W^T)            -- weights [page ¶2]
  Fprop : quantize X (1x16, RNE)     ; Y  = X . W^T     (tcgen05 FP4 GEMM, bf16 out)
  Dgrad : quantize dY (1x16, SR)     ; dX = dY . W
  Wgrad : quantize dY^T, X^T (1x16 along M, shared-sign RHT; SR / RNE) ; dW = dY^T . X
value = 3 * 2MNK / step time (TFLOP/s, quantizers included).  One JSON line.

--impl reference times the CPU oracle (test infrastructure) on a bounded sample of
the same workload; it is the reference arm because the pages ship no code.
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
sys.path.insert(0, ROOT)

M, K, N = 8192, 5120, 20480
METRIC = "NVFP4 GEMM TFLOPS (Fprop/Dgrad/Wgrad at 8192x5120x20480); quantize GB/s"
WORKLOAD = "ffn_up_8192x5120x20480"
GEMM_KERNEL = "gemm_nvfp4_pair_kernel"
FP4_PER_BF16 = 13.5 / 2.25          # nominal dense FP4 : BF16 tensor rate on GB300


def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def rank_seed(rank: int) -> int:
    """Data seed of a rank's token batch (data parallel over M: every rank owns its batch)."""
    return 1000 * rank


def max_over_ranks(ms: float, world: int, device="cpu") -> float:
    """The slowest rank's time (the job's time) via an all-reduce MAX; no-op on one rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job TFLOP/s: the units all ranks processed / the slowest rank's time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def gemm_traffic_bytes():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was taken
    on the current gemm.cu (else None: the counters are stale)."""
    import hashlib
    import re
    try:
        src = open(os.path.join(ROOT, "nvfp4_bit_quantized_gb300", "csrc", "gemm.cu"), "rb").read()
        txt = open(os.path.join(ROOT, "profiles", "gemm_nvfp4_ffn_up_8192x5120x20480.md")).read()
    except OSError:
        return None
    sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    tr = re.search(r"traffic_bytes_per_launch:\s*(\d+)", txt)
    if not sha or not tr or sha.group(1) != hashlib.sha256(src).hexdigest():
        return None
    return int(tr.group(1))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons of the GPU, read through NVML
    (read-only queries) every ~2 ms by a background thread while armed, so even a 25 ms
    timed region gets a dozen readings; falls back to ``nvidia-smi -lms 10`` when NVML
    cannot be loaded.  ``summary()`` covers the samples taken since the last ``take()``."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h)
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, cuda_index: int, interval_s: float = 0.002):
        import threading
        self.cuda_index = cuda_index
        self.interval = interval_s
        self.samples = []                  # (sm_mhz, power_w, reasons bitmask)
        self.max_mhz = None
        self.source = None
        self._armed = threading.Event()
        self._stop = threading.Event()
        self._lock = threading.Lock()
        self._thread = None
        self._smi = None
        self._nvml = self._open_nvml()

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            ok = False
            try:
                import torch
                u = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
                u = u if u.startswith("GPU-") else "GPU-" + u
                ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok and not os.environ.get("CUDA_VISIBLE_DEVICES"):
                ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(h)) == 0
            if not ok:
                return None
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:       # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._h = h
            self.source = "nvml"
            return lib
        except Exception:
            return None

    def _read_nvml(self):
        import ctypes
        c, p, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        lib = self._nvml
        if lib.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(c)) != 0:
            return None
        pw = p.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(self._h, ctypes.byref(p)) == 0 else None
        rs = r.value if self._reasons_fn(self._h, ctypes.byref(r)) == 0 else 0
        return (float(c.value), pw, int(rs))

    def _loop(self):
        import time as _t
        while not self._stop.is_set():
            if not self._armed.wait(0.05):
                continue
            s = self._read_nvml()
            if s is not None:
                with self._lock:
                    self.samples.append(s)
            _t.sleep(self.interval)

    def __enter__(self):
        import threading
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._armed.set()
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self._smi is not None:
            self._smi_stop()

    # -- timed regions ----------------------------------------------------------------
    def _sample_now(self):
        s = self._read_nvml()
        if s is not None:
            with self._lock:
                self.samples.append(s)

    def arm(self):
        """Start sampling (one reading right away, so even a short region has some)."""
        if self._nvml is not None:
            self._sample_now()
            self._armed.set()
        else:
            self._smi_start()

    def disarm(self):
        """Stop sampling (call right after the closing synchronize: one last reading under load)."""
        if self._nvml is not None:
            self._armed.clear()
            self._sample_now()
        else:
            self._smi_stop()

    def _smi_start(self):
        try:
            self._smi = subprocess.Popen(["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except Exception:
            self._smi = None

    def _smi_stop(self):
        if self._smi is None:
            return
        self._smi.terminate()
        try:
            out, _ = self._smi.communicate(timeout=5)
        except Exception:
            self._smi.kill()
            out = ""
        self._smi = None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in out.splitlines():
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            self.max_mhz = mx
            bits = 0
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    bits |= self.REASON_BITS[n]
            pw = None
            try:
                pw = float(f[3])
            except ValueError:
                pass
            with self._lock:
                self.samples.append((sm, pw, bits))

    def take(self):
        """Summary of the samples since the last take(), which it clears."""
        with self._lock:
            smp, self.samples = self.samples, []
        if not smp:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source}
        reasons = sorted({n for n, b in self.REASON_BITS.items() for _, _, r in smp if r & b})
        pw = [p for _, p, _ in smp if p is not None]
        return {"sm_mhz": statistics.median(s for s, _, _ in smp), "sm_min_mhz": min(s for s, _, _ in smp),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(smp),
                "power_w_max": round(max(pw), 1) if pw else None, "source": self.source}

    summary = take


# --------------------------------------------------------------------------- our arm

def run_kernel_only(args):
    """One kernel family alone on the Fprop-shaped operands (for profiling): the
    GEMM (operands quantized once, untimed) or the five quantizer passes."""
    import torch
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs

    torch.cuda.set_device(0)
    X, W, dY = inputs.linear_layer(M, K, N, seed=0, dtype=torch.bfloat16, device="cuda")
    nv.reset_status()
    if args.kernel == "gemm":
        xq = nv.quantize(X, nv.ROW, nv.RNE, scales=False)
        wq = nv.quantize(W, nv.TILE16, nv.RNE, scales=False, transpose=False)
        del dY
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        work = lambda: nv.gemm(xq, wq, out=out, split_tail=True)
        unit, per = "TFLOP/s", 2.0 * M * N * K / 1e12
    else:
        def work():
            nv.quantize(W, nv.TILE16, nv.RNE, scales=False, transpose=True)
            nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=11, scales=False)
            nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=7, rht_seed=11, scales=False)
        unit = "GB/s"
        per = (N * K * (4 + 2 * 0.5625) + (M * K + M * N) * (4 + 2 * 0.5625)) / 1e9
    for _ in range(args.warmup):
        work()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        clk.arm()
        e0.record()
        for _ in range(args.steps):
            work()
        e1.record()
        torch.cuda.synchronize()
        clk.disarm()
        clocks = clk.take()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"kernel": args.kernel, "value": round(per / (ms * 1e-3), 1), "unit": unit,
                      "ms_per_iter": round(ms, 4), "steps": args.steps, "device_status": nv.status_query(),
                      "clocks": clocks, "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N}}))


_CLK = None          # the ClockSampler of a --config run: armed inside every timed region


def _clocks():
    """Clock summary of the timed regions since the last JSON line (None without a sampler)."""
    return _CLK.take() if _CLK is not None else None


def _timed(fn, steps: int, warmup: int) -> float:
    """ms per call of fn (CUDA events on the current stream, after warm-up); the clock
    sampler, when there is one, is armed for the timed region only."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if _CLK is not None:
        _CLK.arm()
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    if _CLK is not None:
        _CLK.disarm()
    return e0.elapsed_time(e1) / steps


def _graph_timed(fn, reps: int, warmup: int) -> float:
    """ms per call of fn with the host out of the loop: reps calls captured once into a CUDA
    graph, the graph replayed twice and timed with CUDA events (the clock sampler armed for the
    replays).  Small tensors would otherwise measure the Python and launch overhead per call."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if _CLK is not None:
        _CLK.arm()
    e0.record()
    g.replay()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    if _CLK is not None:
        _CLK.disarm()
    del g
    return e0.elapsed_time(e1) / (2 * reps)


def run_sweep(args):
    """Quantizer bandwidth sweep: bf16 [R, C], R*C ~ 2^p, C in {5120, 20480}, 0.1% outlier
    columns x100; four modes.  One JSON line per case (GB/s of algorithmic bytes, timed by CUDA
    graph replay; the plain per-call loop, host overhead included, beside it)."""
    import torch
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs
    peaks, src = measured_peaks()
    modes = [("row_rne", nv.ROW, nv.RNE, False, 4.5625), ("row_sr", nv.ROW, nv.SR, False, 4.5625),
             ("tile16_rne_with_transpose", nv.TILE16, nv.RNE, False, 5.125),
             ("col_rht_sr", nv.COL, nv.SR, True, 4.5625)]
    for C in (5120, 20480):
        for p in range(args.sweep_min, args.sweep_max + 1):
            R = inputs.sweep_rows(p, C)
            x = inputs.sweep_tensor(R, C, seed=p, device="cuda")
            for name, block, rnd, rht, bpe in modes:
                fn = lambda: nv.quantize(x, block, rnd, rht=rht, sr_seed=1, rht_seed=2, scales=False,
                                         transpose=(block == nv.TILE16))
                ms_host = _timed(fn, max(3, args.steps), args.warmup)
                ms = _graph_timed(fn, max(3, args.steps), args.warmup)
                gbs = R * C * bpe / (ms * 1e-3) / 1e9
                # the one-read lower bound: the input read once plus the outputs (2D: W and W^T)
                one = 2 + (bpe - 4)
                print(json.dumps({"config": "quantizer_sweep", "mode": name, "R": R, "C": C, "elements": R * C,
                                  "log2_elements": p, "ms": round(ms, 4), "timing": "cuda graph replay",
                                  "ms_host_loop": round(ms_host, 4), "GB/s": round(gbs, 1),
                                  "hbm_frac": round(gbs / peaks["hbm_gbs"], 3), "peak_source": src,
                                  "bytes_per_element": bpe, "inputs_exceed_l2": R * C * 2 > 129e6,
                                  "one_read_bytes_per_element": one,
                                  "one_read_frac": round(R * C * one / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                                  "clocks": _clocks()}))
            del x
            torch.cuda.empty_cache()


def run_mlp(args):
    """One dense MLP block step (5120 -> 20480 -> 5120, squared-ReLU, 16384 tokens), all six
    GEMMs in NVFP4 with re-quantization between them: step time and per-GEMM TFLOP/s.  The
    activation A = relu(H)^2 is quantized straight from H and never stored, from tensor maxima
    the fwd1 GEMM's epilogue leaves (no amax read of H); dH = dA * 2 relu(H) and its tensor maxima
    come out of the dgrad2 GEMM's epilogue (dA is never stored; dH's quantization reads it once)."""
    import torch
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs
    T, d, f = 16384, 5120, 20480
    X = inputs.normal((T, d), 1.0, 10, device="cuda")
    W1 = inputs.normal((f, d), 0.02, 11, device="cuda")
    W2 = inputs.normal((d, f), 0.02, 12, device="cuda")
    dY = inputs.normal((T, d), 1e-3, 13, device="cuda")
    stream = torch.cuda.current_stream()
    names = ["fwd1", "fwd2", "dgrad2", "wgrad2", "dgrad1", "wgrad1"]

    def step(i, ev=None):
        g = []
        w1q, w2q = nv.quantize_weight(W1), nv.quantize_weight(W2)
        xq, xt = nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=9, scales=False)

        def gemm(a, b, k, h=None, maxima=False):
            if ev is not None:
                ev[k][0].record(stream)
            if h is not None:
                out = nv.gemm_sqrelu_backward(a, b, h, maxima=maxima, rht_seed=9)
            elif maxima:
                out = nv.gemm_sqrelu_maxima(a, b, rht_seed=9)
            else:
                out = nv.gemm(a, b, torch.bfloat16, split_tail=True)
            if ev is not None:
                ev[k][1].record(stream)
            return out
        H, maxima = gemm(xq, w1q, 0, maxima=True)          # + relu(H)^2's tensor maxima in the epilogue
        # A = relu(H)^2 is quantized straight from H (the activation is applied as H is loaded)
        aq, at = nv.quantize_dual(H, nv.RNE, nv.RNE, rht=True, rht_seed=9, scales=False, pre="sqrelu",
                                  maxima=maxima)
        gemm(aq, w2q, 1)
        dyq, dyt = nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=5, sr_offset=2 * i, rht_seed=9, scales=False)
        dH, dh_maxima = gemm(dyq, w2q.transposed(), 2, h=H, maxima=True)   # dH = dA * 2 relu(H) + its maxima
        gemm(dyt, at, 3)
        dhq, dht = nv.quantize_dual(dH, nv.SR, nv.SR, rht=True, sr_seed=5, sr_offset=2 * i + 1, rht_seed=9,
                                    scales=False, maxima=dh_maxima)
        gemm(dhq, w1q.transposed(), 4)
        gemm(dht, xt, 5)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in names] for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if _CLK is not None:
        _CLK.arm()
    e0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    if _CLK is not None:
        _CLK.disarm()
    ms = e0.elapsed_time(e1) / args.steps
    # per-GEMM times from a second pass with events around each GEMM
    for i in range(args.steps):
        step(args.warmup + args.steps + i, evs[i])
    torch.cuda.synchronize()
    flop = 2.0 * T * d * f
    per = {n: flop / (statistics.mean(evs[i][k][0].elapsed_time(evs[i][k][1]) for i in range(args.steps)) * 1e-3) / 1e12
           for k, n in enumerate(names)}
    print(json.dumps({"config": "mlp_block_16384x5120x20480_sqrelu", "ms_per_step": round(ms, 4),
                      "tflops_step": round(6 * flop / (ms * 1e-3) / 1e12, 1),
                      "gemm_tflops": {k: round(v, 1) for k, v in per.items()},
                      # W1, W2 (amax + encode each), X and dY duals (amax + fused encode each),
                      # A and dH duals from epilogue maxima (one fused encode each), six GEMMs
                      "launches_per_step": 2 * 2 + 2 * 2 + 2 * 1 + 6, "clocks": _clocks(),
                      "device_status": nv.status_query()}))


def run_heavy(args):
    """Heavy-tailed layer (M=16384, K=4096, N=14336; Student-t inputs, outlier channels):
    the NVFP4 step against the same three GEMMs in BF16 on cuBLAS (torch.matmul): speedup
    (GEMM-only and with quantization) and the NVFP4 error relative to BF16."""
    import torch
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs
    Mh, Kh, Nh = 16384, 4096, 14336
    X, W, dY = inputs.heavy_tailed_layer(Mh, Kh, Nh, seed=0, device="cuda")
    wq_op_w = nv.quantize(W, nv.TILE16, nv.RNE, scales=False, transpose=True)
    xq, xt = nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=11, scales=False)
    dyq, dyt = nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=7, rht_seed=11, scales=False)

    def gemms():
        return (nv.gemm(xq, wq_op_w, torch.bfloat16, split_tail=True),
                nv.gemm(dyq, wq_op_w.transposed(), torch.bfloat16, split_tail=True),
                nv.gemm(dyt, xt, torch.bfloat16, split_tail=True))

    def full():
        w = nv.quantize(W, nv.TILE16, nv.RNE, scales=False, transpose=True)
        a, at = nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=11, scales=False)
        g, gt = nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=7, rht_seed=11, scales=False)
        return (nv.gemm(a, w, torch.bfloat16, split_tail=True),
                nv.gemm(g, w.transposed(), torch.bfloat16, split_tail=True),
                nv.gemm(gt, at, torch.bfloat16, split_tail=True))

    def bf16():
        return X @ W.t(), dY @ W, dY.t() @ X

    t_g, t_f, t_b = (_timed(fn, args.steps, args.warmup) for fn in (gemms, full, bf16))
    fp4, ref = full(), bf16()
    err = {n: round(((a.float() - b.float()).norm() / b.float().norm()).item(), 4)
           for n, a, b in zip(("fprop", "dgrad", "wgrad"), fp4, ref)}
    clk = _clocks()
    # the RHT's effect on the Wgrad product alone, with and without the transform: both operands
    # RNE, and the recipe's rounding (dY stochastic, X RNE); on this layer (outliers are whole
    # channels, which the transform along tokens cannot spread) and on the same layer with its
    # outliers along the tokens instead (the Wgrad contraction axis)
    def wgrad_rht_effect(Xw, dYw, refw):
        out = {}
        for name, rnd in (("rne", nv.RNE), ("recipe_sr_dy", nv.SR)):
            out[name] = {}
            for rht in (True, False):
                gt = nv.quantize(dYw, nv.COL, rnd, rht=rht, sr_seed=7, rht_seed=11, scales=False)
                at = nv.quantize(Xw, nv.COL, nv.RNE, rht=rht, rht_seed=11, scales=False)
                d = nv.gemm(gt, at, torch.bfloat16).float()
                out[name]["rht" if rht else "no_rht"] = round(((d - refw.float()).norm() / refw.float().norm()).item(), 4)
        return out
    wq = {"channel_outliers": wgrad_rht_effect(X, dY, ref[2])}
    del fp4, ref, X, dY, wq_op_w
    torch.cuda.empty_cache()
    Xt, _, dYt = inputs.heavy_tailed_token_outliers(Mh, Kh, Nh, seed=0, device="cuda")
    wq["token_outliers"] = wgrad_rht_effect(Xt, dYt, dYt.t() @ Xt)
    flop = 3 * 2.0 * Mh * Kh * Nh
    print(json.dumps({"config": "heavy_tailed_16384x4096x14336", "nvfp4_gemm_ms": round(t_g, 4),
                      "nvfp4_step_ms": round(t_f, 4), "bf16_cublas_ms": round(t_b, 4),
                      "speedup_gemm_only": round(t_b / t_g, 2), "speedup_with_quantization": round(t_b / t_f, 2),
                      "nvfp4_tflops_gemm": round(flop / (t_g * 1e-3) / 1e12, 1),
                      "bf16_tflops": round(flop / (t_b * 1e-3) / 1e12, 1),
                      "rel_error_vs_bf16": err, "wgrad_rht_effect_rel_error_vs_bf16": wq,
                      "clocks": clk, "device_status": nv.status_query()}))


def run_yardstick(args):
    """Library yardsticks at the three GEMM shapes of the bench workload (context, not the
    target): the same NVFP4 operands through torch._scaled_mm's block-scaled FP4 path
    (cuBLASLt) where this torch offers it -- also a cross-check of the result -- and FP8 (e4m3)
    GEMMs through torch._scaled_mm, with a per-tensor scale and block-scaled (MXFP8: one UE8M0
    scale per 32 elements along K), against this library's GEMM."""
    import torch
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs
    shapes = {"fprop": (M, K, N), "dgrad": (M, N, K), "wgrad": (N, M, K)}     # (rows of A, K, rows of B)
    out = {"config": "gemm_yardsticks", "shapes_MKN": {}, "ours_tflops": {}, "cublaslt_nvfp4_tflops": {},
           "cublaslt_fp8_tflops": {}, "cublaslt_mxfp8_tflops": {}, "mxfp8_vs_fp8_rel_diff": {},
           "nvfp4_vs_cublaslt_rel_diff": {}, "notes": []}
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    for name, (m, k, n) in shapes.items():
        out["shapes_MKN"][name] = [m, k, n]
        flop = 2.0 * m * n * k
        a = inputs.normal((m, k), 1.0, 1, device="cuda").to(torch.bfloat16)
        b = inputs.normal((n, k), 0.02, 2, device="cuda").to(torch.bfloat16)
        qa = nv.quantize(a, nv.ROW, nv.RNE, scales=False)
        qb = nv.quantize(b, nv.ROW, nv.RNE, scales=False)
        d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        t = _timed(lambda: nv.gemm(qa, qb, out=d, split_tail=True), args.steps, args.warmup)
        out["ours_tflops"][name] = round(flop / (t * 1e-3) / 1e12, 1)
        try:
            if fp4 is None:
                raise RuntimeError("torch has no float4_e2m1fn_x2")
            af = qa.codes.view(fp4)
            bf = qb.codes.view(fp4).t()
            sa = qa.scales_mma.view(torch.float8_e4m3fn)
            sb = qb.scales_mma.view(torch.float8_e4m3fn)
            fn = lambda: torch._scaled_mm(af, bf, sa, sb, out_dtype=torch.bfloat16)
            r = fn()
            torch.cuda.synchronize()
            alpha = (qa.s_dec[0] * qb.s_dec[0]).float()
            ref = r.float() * alpha
            out["nvfp4_vs_cublaslt_rel_diff"][name] = round(((d.float() - ref).norm() / ref.norm()).item(), 6)
            t = _timed(fn, args.steps, args.warmup)
            out["cublaslt_nvfp4_tflops"][name] = round(flop / (t * 1e-3) / 1e12, 1)
        except Exception as e:                                    # not offered by this torch / cuBLASLt
            out["cublaslt_nvfp4_tflops"][name] = None
            out["notes"].append(f"nvfp4 {name}: {type(e).__name__}: {str(e)[:160]}")
        a8 = a.to(torch.float8_e4m3fn)
        b8 = b.to(torch.float8_e4m3fn).t()
        r8 = None
        try:
            one = torch.ones((), dtype=torch.float32, device="cuda")
            fn = lambda: torch._scaled_mm(a8, b8, one, one, out_dtype=torch.bfloat16)
            r8 = fn()
            t = _timed(fn, args.steps, args.warmup)
            out["cublaslt_fp8_tflops"][name] = round(flop / (t * 1e-3) / 1e12, 1)
        except Exception as e:
            out["cublaslt_fp8_tflops"][name] = None
            out["notes"].append(f"fp8 {name}: {type(e).__name__}: {str(e)[:160]}")
        try:
            # block-scaled FP8 (MXFP8): the same e4m3 codes with every block scale 2^0 (UE8M0 code
            # 127), so the result must equal the per-tensor one; the scale layout is cuBLASLt's
            # 128 x 4 tiling, whose content is uniform here
            e8m0 = getattr(torch, "float8_e8m0fnu", None)
            if e8m0 is None:
                raise RuntimeError("torch has no float8_e8m0fnu")
            kb = ((k // 32) + 3) // 4 * 4
            sa8 = torch.full((((m + 127) // 128) * 128 * kb,), 127, dtype=torch.uint8, device="cuda").view(e8m0)
            sb8 = torch.full((((n + 127) // 128) * 128 * kb,), 127, dtype=torch.uint8, device="cuda").view(e8m0)
            fn = lambda: torch._scaled_mm(a8, b8, sa8, sb8, out_dtype=torch.bfloat16)
            rm = fn()
            torch.cuda.synchronize()
            if r8 is not None:
                out["mxfp8_vs_fp8_rel_diff"][name] = round(((rm.float() - r8.float()).norm() / r8.float().norm()).item(), 6)
            t = _timed(fn, args.steps, args.warmup)
            out["cublaslt_mxfp8_tflops"][name] = round(flop / (t * 1e-3) / 1e12, 1)
        except Exception as e:
            out["cublaslt_mxfp8_tflops"][name] = None
            out["notes"].append(f"mxfp8 {name}: {type(e).__name__}: {str(e)[:160]}")
        del a, b, qa, qb, d, a8, b8
        torch.cuda.empty_cache()
    out["clocks"] = _clocks()
    out["device_status"] = nv.status_query()
    print(json.dumps(out))


def run_mx(args):
    """MXFP4, the comparison format (32-element blocks, UE8M0 scales, no tensor scale):
    its three GEMMs and its quantizer at the FFN up-projection shapes next to NVFP4's,
    and the error of each format's Fprop / Dgrad / Wgrad against BF16 (cuBLAS) on the
    heavy-tailed layer -- NVFP4 both as plain 1x16 RNE (format against format) and as the
    full recipe (16x16 weights, RHT and SR on the Wgrad inputs)."""
    import torch
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs
    peaks, src = measured_peaks()
    out = {"config": "mxfp4_comparison", "gemm_shapes_MKN": {}, "mx_gemm_tflops": {}, "nvfp4_gemm_tflops": {},
           "mx_quantize": {}, "rel_error_vs_bf16_heavy_tailed": {}, "peak_source": src}
    X, W, dY = inputs.linear_layer(M, K, N, seed=0, device="cuda")
    # operands of the three products, each as [rows, K] of its GEMM
    mx_ops = {"fprop": (lambda: nv.mx_quantize(X), lambda: nv.mx_quantize(W)),
              "dgrad": (lambda: nv.mx_quantize(dY), lambda: nv.mx_quantize(W, col=True)),
              "wgrad": (lambda: nv.mx_quantize(dY, col=True), lambda: nv.mx_quantize(X, col=True))}
    nv_ops = {"fprop": (lambda: nv.quantize(X, nv.ROW, nv.RNE, scales=False),
                        lambda: nv.quantize(W, nv.ROW, nv.RNE, scales=False)),
              "dgrad": (lambda: nv.quantize(dY, nv.ROW, nv.RNE, scales=False),
                        lambda: nv.quantize(W, nv.COL, nv.RNE, scales=False)),
              "wgrad": (lambda: nv.quantize(dY, nv.COL, nv.RNE, scales=False),
                        lambda: nv.quantize(X, nv.COL, nv.RNE, scales=False))}
    for name in ("fprop", "dgrad", "wgrad"):
        qa, qb = mx_ops[name][0](), mx_ops[name][1]()
        m, n, k = qa.rows, qb.rows, qa.cols
        out["gemm_shapes_MKN"][name] = [m, k, n]
        flop = 2.0 * m * n * k
        d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        t = _timed(lambda: nv.mx_gemm(qa, qb, out=d), args.steps, args.warmup)
        out["mx_gemm_tflops"][name] = round(flop / (t * 1e-3) / 1e12, 1)
        del qa, qb
        qa, qb = nv_ops[name][0](), nv_ops[name][1]()
        t = _timed(lambda: nv.gemm(qa, qb, out=d), args.steps, args.warmup)
        out["nvfp4_gemm_tflops"][name] = round(flop / (t * 1e-3) / 1e12, 1)
        del qa, qb, d
        torch.cuda.empty_cache()
    # quantizer: bf16 in (2 B), codes (0.5 B) and UE8M0 scales (1/32 B) out per element
    bpe = 2 + 0.5 + 1 / 32
    for mode, col in (("row", False), ("col", True)):
        t = _timed(lambda: nv.mx_quantize(dY, col=col, scales=False), args.steps, args.warmup)
        gbs = dY.numel() * bpe / (t * 1e-3) / 1e9
        out["mx_quantize"][f"{mode}_{M}x{N}"] = {"ms": round(t, 4), "GB/s": round(gbs, 1),
                                                "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)}
    out["clocks"] = _clocks()
    del X, W, dY
    torch.cuda.empty_cache()
    Mh, Kh, Nh = 16384, 4096, 14336
    X, W, dY = inputs.heavy_tailed_layer(Mh, Kh, Nh, seed=0, device="cuda")
    ref = {"fprop": X @ W.t(), "dgrad": dY @ W, "wgrad": dY.t() @ X}

    def rel(name, d):
        r = ref[name].float()
        return round(((d.float() - r).norm() / r.norm()).item(), 5)
    mx = {"fprop": nv.mx_gemm(nv.mx_quantize(X), nv.mx_quantize(W)),
          "dgrad": nv.mx_gemm(nv.mx_quantize(dY), nv.mx_quantize(W, col=True)),
          "wgrad": nv.mx_gemm(nv.mx_quantize(dY, col=True), nv.mx_quantize(X, col=True))}
    out["rel_error_vs_bf16_heavy_tailed"]["mxfp4"] = {k: rel(k, v) for k, v in mx.items()}
    del mx
    q = lambda x, b, r=nv.RNE, rht=False: nv.quantize(x, b, r, rht=rht, sr_seed=7, rht_seed=11, scales=False)
    plain = {"fprop": nv.gemm(q(X, nv.ROW), q(W, nv.ROW)),
             "dgrad": nv.gemm(q(dY, nv.ROW), q(W, nv.COL)),
             "wgrad": nv.gemm(q(dY, nv.COL), q(X, nv.COL))}
    out["rel_error_vs_bf16_heavy_tailed"]["nvfp4_1x16_rne"] = {k: rel(k, v) for k, v in plain.items()}
    del plain
    wq = nv.quantize_weight(W)
    recipe = {"fprop": nv.gemm(q(X, nv.ROW), wq),
              "dgrad": nv.gemm(q(dY, nv.ROW, nv.SR), wq.transposed()),
              "wgrad": nv.gemm(q(dY, nv.COL, nv.SR, True), q(X, nv.COL, nv.RNE, True))}
    out["rel_error_vs_bf16_heavy_tailed"]["nvfp4_recipe"] = {k: rel(k, v) for k, v in recipe.items()}
    out["device_status"] = nv.status_query()
    print(json.dumps(out))


def run_ours(args):
    import torch
    import torch.distributed as dist
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import inputs

    if args.kernel != "step":
        return run_kernel_only(args)
    if args.config != "ffn_up":
        global _CLK
        torch.cuda.set_device(0)
        with ClockSampler(0) as clk:
            _CLK = clk
            try:
                return {"sweep": run_sweep, "mlp": run_mlp, "heavy": run_heavy, "yardstick": run_yardstick,
                        "mxfp4": run_mx}[args.config](args)
            finally:
                _CLK = None

    rank, world, local = env_rank()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    # weak scaling: every rank owns its own token batch (data parallel over M)
    X, W, dY = inputs.linear_layer(M, K, N, seed=rank_seed(rank), dtype=torch.bfloat16, device=dev)
    nv.reset_status()
    stream = torch.cuda.current_stream()

    names = ["quant_W_2d", "quant_X_dual", "gemm_fprop", "quant_dY_dual_sr", "gemm_dgrad", "gemm_wgrad"]

    def step(sr_offset, ev=None):
        # forward: W (16x16, with W^T) and X (1x16 rows for Fprop + RHT columns kept for Wgrad);
        # backward: dY (1x16 rows for Dgrad + RHT columns for Wgrad), stochastic rounding
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        wq = nv.quantize(W, nv.TILE16, nv.RNE, scales=False, transpose=True)
        mark(1)
        xq, xt = nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=11, scales=False)
        mark(2)
        Y = nv.gemm(xq, wq, torch.bfloat16, split_tail=True)
        mark(3)
        dyq, dyt = nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=7, sr_offset=sr_offset, rht_seed=11,
                                    scales=False)
        mark(4)
        dX = nv.gemm(dyq, wq.transposed(), torch.bfloat16, split_tail=True)
        mark(5)
        dW = nv.gemm(dyt, xt, torch.bfloat16, split_tail=True)
        mark(6)
        return Y, dX, dW

    # W (amax + encode), X and dY duals (amax + one encode for both operands), three GEMMs
    launches_per_step = 2 + 2 + 2 + 3
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if nv.status_query() != 0:
        raise RuntimeError("device status error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.arm()
        t0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        t1.record(stream)
        torch.cuda.synchronize()
        clk.disarm()
        clocks = clk.take()
    if world > 1:
        dist.barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # The per-operation breakdown comes from a second pass with events between the operations;
    # the headline time above is taken without them, so nothing sits between the kernels.
    for i in range(args.steps):
        step(args.warmup + args.steps + i, evs[i])
    torch.cuda.synchronize()
    status = nv.status_query()
    ms_step = ms_total / args.steps
    flops_step = 3 * 2.0 * M * N * K
    value = job_throughput(flops_step, ms_step, world)

    per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
           for j, n in enumerate(names)}
    gemm_ms = statistics.mean([per["gemm_fprop"], per["gemm_dgrad"], per["gemm_wgrad"]])
    gemm_tflops = {k: 2.0 * M * N * K / (per[k] * 1e-3) / 1e12 for k in ("gemm_fprop", "gemm_dgrad", "gemm_wgrad")}
    # algorithmic bytes per element: the 2D weight pass reads bf16 twice (amax + encode) and writes
    # W and W^T codes + scales (2 x (0.5 + 1/16) B); a dual pass also reads bf16 twice (one amax
    # read and one encode read for both operands) and writes two operands' codes + scales.  The
    # tensor amax has to be known before any element is encoded, so two reads are the minimum
    # for a tensor larger than L2.
    qbytes = {
        "quant_W_2d": N * K * (2 + 2 + 2 * (0.5 + 1 / 16)),
        "quant_X_dual": M * K * (2 + 2 + 2 * (0.5 + 1 / 16)),
        "quant_dY_dual_sr": M * N * (2 + 2 + 2 * (0.5 + 1 / 16)),
    }
    qbytes_sep = dict(qbytes, quant_X_dual=M * K * (2 + 2 * 2 + 2 * (0.5 + 1 / 16)),
                      quant_dY_dual_sr=M * N * (2 + 2 * 2 + 2 * (0.5 + 1 / 16)))
    quant_gbs = {k: qbytes[k] / (per[k] * 1e-3) / 1e9 for k in qbytes}
    quant_ms = sum(per[k] for k in qbytes)
    peaks, peak_src = measured_peaks()
    # The timed region is a short burst (tens of ms at the maximum SM clock), so the burst
    # bf16 figure applies; FP4 dense peak = that x the nominal FP4 : BF16 rate ratio.
    fp4_peak = peaks["bf16_tflops"] * FP4_PER_BF16
    achieved = 2.0 * M * N * K / (gemm_ms * 1e-3) / 1e12
    # A second, hardware figure: ncu's sm__pipe_tensor_cycles_active counts 100 % at
    # 16384 FP4 MACs (32768 flop) per SM per cycle, so at the sampled median SM clock the
    # tensor pipes of all SMs top out at this rate.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pipe_mhz = clocks.get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    pipe_ceiling = sms * 32768 * pipe_mhz * 1e6 / 1e12

    # End to end through the public API with host buffers: every step copies its inputs in
    # from pinned host memory, runs the layer and copies its results out.  Three streams and
    # two device input sets, so step i's H2D copy, step i-1's compute and step i-2's D2H copy
    # overlap (the copy engines and the SMs run at once), as a training pipeline feeds a layer.
    hX = X.cpu().pin_memory()
    hW = W.cpu().pin_memory()
    hdY = dY.cpu().pin_memory()
    hY = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    hdX = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
    hdW = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
    h2d = (hX.numel() + hW.numel() + hdY.numel()) * 2
    d2h = (hY.numel() + hdX.numel() + hdW.numel()) * 2
    sets = [(X, W, dY), tuple(torch.empty_like(t) for t in (X, W, dY))]
    # two device output sets as well: nothing is allocated inside the timed pipeline
    outs = [tuple(torch.empty(s_, dtype=torch.bfloat16, device=dev) for s_ in ((M, N), (M, K), (N, K)))
            for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run_e2e(nsteps, first):
        done = [None, None]                       # compute-finished event of the step that last used each set
        out_done = [None, None]                   # D2H-finished event of the step that last used each output set
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        for i in range(nsteps):
            xs, ws, ys = sets[i % 2]
            with torch.cuda.stream(s_in):
                if done[i % 2] is not None:
                    s_in.wait_event(done[i % 2])
                xs.copy_(hX, non_blocking=True)
                ws.copy_(hW, non_blocking=True)
                ys.copy_(hdY, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s_in)
            stream.wait_event(landed)
            if out_done[i % 2] is not None:
                stream.wait_event(out_done[i % 2])
            Yd, dXd, dWd = outs[i % 2]
            wq = nv.quantize(ws, nv.TILE16, nv.RNE, scales=False, transpose=True)
            xq, xt = nv.quantize_dual(xs, nv.RNE, nv.RNE, rht=True, rht_seed=11, scales=False)
            nv.gemm(xq, wq, out=Yd, split_tail=True)
            dyq, dyt = nv.quantize_dual(ys, nv.SR, nv.SR, rht=True, sr_seed=7, sr_offset=first + i,
                                        rht_seed=11, scales=False)
            nv.gemm(dyq, wq.transposed(), out=dXd, split_tail=True)
            nv.gemm(dyt, xt, out=dWd, split_tail=True)
            fin = torch.cuda.Event()
            fin.record(stream)
            done[i % 2] = fin
            with torch.cuda.stream(s_out):
                s_out.wait_event(fin)
                for d, h in ((Yd, hY), (dXd, hdX), (dWd, hdW)):
                    h.copy_(d, non_blocking=True)
                copied = torch.cuda.Event()
                copied.record(s_out)
                out_done[i % 2] = copied
        end.record(s_out)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    e2e_ms = e2e_value = None
    if not args.no_e2e:
        run_e2e(2, 0)
        e2e_steps = max(4, args.steps)                # steady state: fill and drain amortised over the steps
        e2e_ms = run_e2e(e2e_steps, 2) / e2e_steps
        e2e_value = round(job_throughput(flops_step, e2e_ms, world), 2)
        e2e_ms = round(e2e_ms, 3)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1/e4m3 operands, fp32 accumulate, bf16 in/out",
        "data": "synthetic (seeded normal; X N(0,1), W N(0,0.02), dY N(0,1e-3))",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "in_dtype": "bf16", "out_dtype": "bf16",
                   "step": "quantize W (16x16, +W^T), X dual (1x16 rows + RHT columns), dY dual (SR) + Fprop/Dgrad/Wgrad GEMMs",
                   "l2": "inputs larger than L2 (the step streams >1 GB; 129 MB L2)",
                   "parallelism": f"dp{world} (independent token batches, no collective)"},
        "gemm_tflops": {k: round(v, 1) for k, v in gemm_tflops.items()},
        "quantize_gbs": {k: round(v, 1) for k, v in quant_gbs.items()},
        "ms_breakdown": {k: round(v, 4) for k, v in per.items()},
        "quantize_ms_per_step": round(quant_ms, 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp4_peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / fp4_peak, 4), "traffic": gemm_traffic_bytes(),
                     "kernel": GEMM_KERNEL,
                     "peak_source": f"{peak_src} bf16 burst x {FP4_PER_BF16:g} (nominal dense FP4:BF16)",
                     "tensor_pipe_ceiling": {"value": round(pipe_ceiling, 1), "unit": "TFLOP/s",
                                             "frac": round(achieved / pipe_ceiling, 4),
                                             "basis": f"{sms} SMs x 32768 FP4 flop/cycle (ncu tensor-pipe 100 %) "
                                                      f"x {pipe_mhz:g} MHz (median sampled SM clock)"}},
        "quantize_roofline": {"bound": "hbm", "achieved": round(sum(qbytes.values()) / (quant_ms * 1e-3) / 1e9, 1),
                              "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": round(sum(qbytes.values()) / (quant_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                              # the same time with each dual counted as two separate encode passes
                              # (7.125 B/elem, the count before the fused encode), for comparison
                              "separate_encodes": {
                                  "achieved": round(sum(qbytes_sep.values()) / (quant_ms * 1e-3) / 1e9, 1),
                                  "frac": round(sum(qbytes_sep.values()) / (quant_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "overlap": "H2D copies, the layer step and D2H copies on three streams, two device input sets"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "device_status": status,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))


# --------------------------------------------------------------------------- oracle (CPU) arm

def oracle_sample(budget_s: float = 15.0, reps: int | None = None, rotate: bool = False, threads: int = 1):
    """Times the CPU oracle on a bounded sample of the step: one output block of
    each GEMM with the full contraction length of the workload, the oracle
    quantizing the operand rows that block needs:
      Fprop  64x128 block of Y,  K = 5120   (X rows 1x16 RNE, W rows 16x16)
      Dgrad  64x128 block of dX, N = 20480  (dY rows 1x16 SR, W^T rows 16x16)
      Wgrad 128x64  block of dW, M = 8192   (dY^T, X^T columns with the RHT; SR / RNE)
    With ``rotate`` a rep is one of the three blocks in turn (a third of the work).
    ``threads`` > 1 splits each quantization's rows and each GEMM block's rows among
    that many threads (the oracle's threaded entry points; identical results).
    value = sampled GEMM flops / oracle time."""
    import numpy as np
    import oracle
    import torch
    from nvfp4_bit_quantized_gb300 import inputs

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    mb, nb = 64, 128
    xs = bits(inputs.normal((mb, K), 1.0, 0))            # X rows
    ws = bits(inputs.normal((nb, K), 0.02, 1))           # W rows
    dys = bits(inputs.normal((mb, N), 1e-3, 2))          # dY rows
    wts = bits(inputs.normal((nb, N), 0.02, 3))          # W^T rows (= W columns)
    dyc = bits(inputs.normal((M, nb), 1e-3, 4))          # dY columns
    xc = bits(inputs.normal((M, mb), 1.0, 5))            # X columns
    deq, th = oracle.dequant, threads
    q = lambda *a, **k: oracle.quantize(*a, threads=th, **k)
    gemm = lambda a, b: oracle.gemm_f64(a, b, threads=th)
    blocks = [
        (lambda: gemm(deq(q(xs, oracle.ROW)), deq(q(ws, oracle.TILE16))), K),
        (lambda: gemm(deq(q(dys, oracle.ROW, oracle.SR, sr_seed=7)), deq(q(wts, oracle.TILE16))), N),
        (lambda: gemm(deq(q(dyc, oracle.COL, oracle.SR, rht=True, sr_seed=7, rht_seed=11)),
                      deq(q(xc, oracle.COL, oracle.RNE, rht=True, rht_seed=11))), M),
    ]
    n, flops, t0 = 0, 0.0, time.perf_counter()
    while True:
        for fn, klen in (blocks[n % 3:n % 3 + 1] if rotate else blocks):
            fn()
            flops += 2.0 * mb * nb * klen
        n += 1
        el = time.perf_counter() - t0
        if (reps is not None and n >= reps) or (reps is None and el >= budget_s):
            break
    what = "one output block in turn of" if rotate else "three output blocks"
    how = "single-threaded C" if threads <= 1 else f"C on {threads} threads"
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": max(1, threads), "kind": "oracle",
            "sample": f"{n} x {what} (Fprop 64x128 K={K}, Dgrad 64x128 K={N}, Wgrad 128x64 K={M}) "
                      f"with their operand rows quantized by the oracle; {how}; {el:.1f} s",
            "flops_per_rep": round(flops / n), "seconds": round(el, 3)}


# Algorithmic bytes per element of one quantization with bf16 input, as the GPU sweep counts them:
# the input read twice (tensor amax, then encode), codes 0.5 B, scales 1/16 B (16x16: 1/256 B).
ORACLE_QUANT_MODES = [("row_rne", dict(block=0), 4.5625), ("row_sr", dict(block=0, round_mode=1, sr_seed=1), 4.5625),
                      ("tile16_rne", dict(block=2), 2 + 2 + 0.5 + 1 / 256),
                      ("col_rht_sr", dict(block=1, round_mode=1, rht=True, sr_seed=1, rht_seed=2), 4.5625)]


def oracle_quantize_rates(rows: int, cols: int, threads: int) -> dict:
    """GB/s (algorithmic bytes, as the GPU's) of the oracle quantizing a bf16 [rows, cols]
    tensor shaped like dY (N(0, 1e-3)) in the four modes, on ``threads`` threads."""
    import numpy as np
    import oracle
    import torch
    from nvfp4_bit_quantized_gb300 import inputs
    x = inputs.normal((rows, cols), 1e-3, 6).contiguous().view(torch.int16).numpy().view(np.uint16)
    out = {}
    for name, kw, bpe in ORACLE_QUANT_MODES:
        t0 = time.perf_counter()
        oracle.quantize(x, threads=threads, **kw)
        el = time.perf_counter() - t0
        out[name] = round(x.size * bpe / el / 1e9, 3)
    return out


def cpu_baseline(budget_s: float) -> dict:
    """The oracle on this host's cores (sched_getaffinity count) and on one core: sampled GEMM
    blocks (TFLOP/s; ``value``) and the four quantizer modes (GB/s; full dY size on all cores,
    a 1/cores slice of its columns on one core)."""
    import oracle
    oracle.build()
    cores = oracle.host_cores()
    t0 = time.perf_counter()
    g_all = oracle_sample(budget_s=budget_s / 4, threads=cores)
    g_one = oracle_sample(budget_s=budget_s / 4, threads=1)
    q_all = oracle_quantize_rates(M, N, cores)
    q_one = oracle_quantize_rates(M, max(16, (N // cores) // 16 * 16), 1)
    return {"value": g_all["value"], "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": g_all["sample"],
            "one_core": {"value": g_one["value"], "unit": "TFLOP/s", "sample": g_one["sample"]},
            "quantize_gbs": {"all_cores": q_all, "one_core": q_one,
                             "tensor_all_cores": f"bf16 [{M}, {N}] (dY-shaped, N(0, 1e-3))",
                             "tensor_one_core": f"bf16 [{M}, {max(16, (N // cores) // 16 * 16)}]",
                             "bytes_per_element": {n: round(b, 4) for n, _, b in ORACLE_QUANT_MODES}},
            "seconds": round(time.perf_counter() - t0, 1)}


def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.host_cores()
    # a step is one of the three sampled GEMM blocks in turn, on all of this host's cores
    for _ in range(args.warmup):
        oracle_sample(reps=1, rotate=True, threads=cores)
    t0 = time.perf_counter()
    r = oracle_sample(reps=args.steps, rotate=True, threads=cores)
    el = time.perf_counter() - t0
    value = r["value"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N,
                                            "sample": "per step: one output block of one GEMM (Fprop, Dgrad, Wgrad in turn), full contraction"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400,
                    help="timed steps (the default, ~0.5 s of the headline step, lets the clock sampler "
                         "take several readings under load)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernel", choices=["step", "gemm", "quantize"], default="step",
                    help="step: the whole hot path (the bench line); gemm / quantize: one kernel family alone")
    ap.add_argument("--config", choices=["ffn_up", "mlp", "sweep", "heavy", "yardstick", "mxfp4"], default="ffn_up",
                    help="ffn_up: the headline workload (default); mlp / sweep / heavy / yardstick / mxfp4: the other "
                         "workloads, one JSON line each (not the headline metric)")
    ap.add_argument("--sweep-min", type=int, default=20)
    ap.add_argument("--sweep-max", type=int, default=28)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
