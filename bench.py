"""Benchmark: NVFP4 linear layer (quantise + GEMM), fprop + dgrad + wgrad.

One step = one pass of the whole hot path over the 12B-hybrid-shaped MLP
up-projection (tokens 8192 = 4 x 2048, hidden 5120, FFN 20480): quantise
each of X, W, dY once into both orientations the GEMMs need (1x16
activations/gradients, 16x16 weights, transform + stochastic rounding on the
wgrad operands), then the three block-scaled FP4 GEMMs with BF16 outputs.  Inputs are synthetic
BF16 tensors resident in HBM (629 MB per step, larger than L2).

Prints one JSON line.  `--impl reference` times the CPU oracle (the plain C
statement of the same arithmetic) on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 linear TFLOP/s (quantize+GEMM) and quantize GB/s, % of GB300 roofline"
T, HID, FFN = 8192, 5120, 20480
GEMM_FLOP = 2.0 * T * HID * FFN  # each of fprop, dgrad, wgrad
STEP_FLOP = 3 * GEMM_FLOP
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio on GB300
QUANT_OUT_BYTES_PER_ELT = 0.5 + 1.0 / 16  # codes + block scales of one quantised output
QUANT_BYTES_PER_ELT = 2.0 + QUANT_OUT_BYTES_PER_ELT  # read BF16, write one output
# one dual quantise per tensor and step: read BF16 once, write two quantised outputs
QUANT_STEP_BYTES = (T * HID + FFN * HID + T * FFN) * (2.0 + 2 * QUANT_OUT_BYTES_PER_ELT)
WORKLOAD = ("12B-hybrid MLP up-projection fprop+dgrad+wgrad, tokens 8192 (4x2048), hidden 5120, FFN 20480; "
            "X N(0,1), W N(0,0.02), dY N(0,1e-3); W 16x16, X/dY 1x16, wgrad operands RHT+SR")


# DRAM bytes per GEMM call (dram__bytes_read.sum + dram__bytes_write.sum from
# one ncu capture of each of the step's three GEMM shapes -- the GEMM kernel
# plus, for dgrad and wgrad, the reduction of their last wave's K pieces --
# averaged like the achieved rate), keyed by the SHA-256 prefix of the GEMM
# kernel's sources: a changed kernel reports null until it is measured again.
GEMM_TRAFFIC = {"ce9d4ccb74722c30": 365575680}


def _gemm_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "block_scaled_gemm_nvfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return GEMM_TRAFFIC.get(h.hexdigest()[:16])


def _config():
    return {"workload": WORKLOAD, "tokens": T, "hidden": HID, "ffn": FFN, "out_dtype": "bf16",
            "l2": "inputs larger than L2 (X+W+dY = 629 MB BF16 per step)"}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        smax.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        loaded = sorted(sm)[len(sm) // 4:] or sm  # drop the idle head of the window
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _max_over_ranks(ms, pg, dev):
    """The slowest rank's time (every rank gets it); ms itself when alone."""
    if pg is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.item()


def _tflops(world, ms_per_step):
    """Whole-job throughput: every rank runs one step of the workload (weak
    scaling, independent replicas), timed by the slowest rank."""
    return world * STEP_FLOP / (ms_per_step * 1e-3) / 1e12


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------- ours
def run_ours(args):
    import torch

    import block_scaled_gemm_nvfp4_gb300 as nv
    from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    nv.lib()

    x_c, w_c, dy_c = syn.config2()
    x, w, dy = x_c.to(dev), w_c.to(dev), dy_c.to(dev)

    plan = _step_plan(nv, torch, x, w, dy, dev)
    stream = torch.cuda.current_stream()
    gemm_events = []
    quant_events = []

    def step(record):
        _run_step(nv, plan, stream, quant_events if record else None, gemm_events if record else None)

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step(True)
        t1.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
    ms_total = t0.elapsed_time(t1)
    st = nv.nvfp4_check_device_status(plan["ws"])
    if st != nv.NVFP4_OK:
        raise RuntimeError("device status %s" % nv.nvfp4_status_string(st))
    ms_total = _max_over_ranks(ms_total, pg, dev)
    ms_step = ms_total / args.steps
    value = _tflops(world, ms_step)

    gemm_ms = statistics.mean(a.elapsed_time(b) for a, b in gemm_events)  # per GEMM
    quant_ms = sum(a.elapsed_time(b) for a, b in quant_events) / args.steps  # three dual quantises per step
    peaks, src = _peaks()
    peak_fp4 = peaks["bf16_tflops"] * FP4_OVER_BF16
    achieved = GEMM_FLOP / (gemm_ms * 1e-3) / 1e12
    quant_gbs = QUANT_STEP_BYTES / (quant_ms * 1e-3) / 1e9
    clock = clocks.summary()

    # launches per step: three dual quantises (amax + encode kernels), three
    # GEMMs, and the reduction of each GEMM whose last wave is cut along K
    tails = sum(nv.nvfp4_gemm_plan(M, N, K, plan["ws"].numel())["tail_tiles"] > 0
                for M, N, K in ((T, FFN, HID), (T, HID, FFN), (FFN, HID, T)))
    launches_per_step = 3 * 2 + 3 + tails

    e2e = run_e2e(args, nv, torch, x_c, w_c, dy_c, dev, world, pg)
    # the GEMM's own instruction issued back to back in isolation (after the
    # timed regions): the ceiling its tensor-pipe time can approach
    mma_tf, mma_cyc = nv.nvfp4_debug_mma_rate(0, 4096)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 codes, e4m3 block scales, fp32 accumulate)",
        "data": "synthetic", "config": _config(),
        "roofline": {"bound": "tensor", "kernel": "nvfp4_gemm (tcgen05 mxf4nvf4)", "achieved": round(achieved, 1),
                     "peak": round(peak_fp4, 1), "unit": "TFLOP/s", "frac": round(achieved / peak_fp4, 4),
                     "traffic": _gemm_traffic(),
                     "peak_source": "%s bf16 %.1f TFLOP/s x nominal FP4/BF16 ratio %.1f" % (
                         src, peaks["bf16_tflops"], FP4_OVER_BF16),
                     "gemm_ms": round(gemm_ms, 4),
                     "instruction_ceiling": {
                         "tflops": round(mma_tf, 1), "frac": round(achieved / mma_tf, 4),
                         "cycles_per_mma": round(mma_cyc, 2),
                         "what": "tcgen05.mma kind::mxf4nvf4 scale_vec::4X cta_group::2 256x256x64 issued back to "
                                 "back in isolation (bench.py --case mma)"}},
        "quantize": {"bound": "hbm", "achieved": round(quant_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(quant_gbs / peaks["hbm_gbs"], 4), "ms_per_step": round(quant_ms, 4),
                     "bytes_model": "per tensor (X, W, dY): read BF16 once + two outputs of codes and scales "
                                    "= 2 + 2 x 0.5625 B/element"},
        "clocks": clock,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def _step_plan(nv, torch, x, w, dy, dev):
    """Preallocated quantised operands, outputs and one workspace for the
    training step of the linear layer (the library never allocates)."""
    s = nv.NVFP4_DEFAULT_RHT_SEED
    cfg = {
        "x": nv.quant_cfg(block=0),  # fprop A: X [T, hidden] along hidden
        "xt": nv.quant_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=6),  # wgrad B: X^T along T
        "w": nv.quant_cfg(block=1),  # fprop B: W [ffn, hidden] along hidden
        "wt": nv.quant_cfg(block=1, transpose=1),  # dgrad B: W^T along ffn
        "dy": nv.quant_cfg(block=0),  # dgrad A: dY [T, ffn] along ffn
        "dyt": nv.quant_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=5),  # wgrad A: dY^T along T
    }
    src = {"x": x, "xt": x, "w": w, "wt": w, "dy": dy, "dyt": dy}
    q = {k: nv.nvfp4_empty(src[k], cfg[k]) for k in cfg}
    out = {"y": torch.empty((T, FFN), dtype=torch.bfloat16, device=dev),
           "dx": torch.empty((T, HID), dtype=torch.bfloat16, device=dev),
           "dw": torch.empty((FFN, HID), dtype=torch.bfloat16, device=dev)}
    # one workspace for every call of the step: the quantisers' scratch, or
    # the largest GEMM partial-sum scratch (the last wave's tiles cut along K)
    ws_bytes = max(nv.nvfp4_quantize_workspace_size(T, FFN, cfg["x"]) + (1 << 16),
                   *(nv.nvfp4_gemm_workspace_size(M, N, K) for M, N, K in ((T, FFN, HID), (T, HID, FFN),
                                                                           (FFN, HID, T))))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    return {"cfg": cfg, "q": q, "out": out, "ws": ws, "src": {"x": x, "w": w, "dy": dy}}


def _run_step(nv, plan, stream, quant_events=None, gemm_events=None):
    """fprop, dgrad, wgrad of Y = X W^T: each BF16 tensor is quantised once
    into both orientations the GEMMs need, then the three GEMMs run."""
    import torch

    c, q, o, ws, src = plan["cfg"], plan["q"], plan["out"], plan["ws"], plan["src"]
    rec = quant_events is not None

    def ev():
        if not rec:
            return None
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    e0 = ev()
    nv.nvfp4_quantize_dual(src["x"], c["x"], c["xt"], q["x"], q["xt"], workspace=ws)
    nv.nvfp4_quantize_dual(src["w"], c["w"], c["wt"], q["w"], q["wt"], workspace=ws)
    e1 = ev()
    nv.nvfp4_gemm(q["x"], q["w"], nv.NVFP4_OUT_BF16, d=o["y"], workspace=ws)
    e2 = ev()
    nv.nvfp4_quantize_dual(src["dy"], c["dy"], c["dyt"], q["dy"], q["dyt"], workspace=ws)
    e3 = ev()
    nv.nvfp4_gemm(q["dy"], q["wt"], nv.NVFP4_OUT_BF16, d=o["dx"], workspace=ws)
    e4 = ev()
    nv.nvfp4_gemm(q["dyt"], q["xt"], nv.NVFP4_OUT_BF16, d=o["dw"], workspace=ws)
    e5 = ev()
    if rec:
        quant_events += [(e0, e1), (e2, e3)]
        gemm_events += [(e1, e2), (e3, e4), (e4, e5)]


def run_e2e(args, nv, torch, x_c, w_c, dy_c, dev, world, pg):
    """The same step through the public API with pinned host buffers: every
    step copies X, W, dY host->device and Y, dX, dW device->host inside the
    timed region.  Copies run on their own streams and overlap the compute of
    neighbouring steps (device tensors double-buffered by step parity); each
    step's compute waits for its inputs, fprop starts once X and W have
    arrived, and each result is copied out as soon as it is produced."""
    xh, wh, dyh = x_c.pin_memory(), w_c.pin_memory(), dy_c.pin_memory()
    yh = torch.empty((T, FFN), dtype=torch.bfloat16).pin_memory()
    dxh = torch.empty((T, HID), dtype=torch.bfloat16).pin_memory()
    dwh = torch.empty((FFN, HID), dtype=torch.bfloat16).pin_memory()
    slots = []
    for _ in range(2):
        xd, wd, dyd = (torch.empty_like(x_c, device=dev), torch.empty_like(w_c, device=dev),
                       torch.empty_like(dy_c, device=dev))
        slots.append({"x": xd, "w": wd, "dy": dyd, "plan": _step_plan(nv, torch, xd, wd, dyd, dev),
                      "ev": {k: torch.cuda.Event() for k in ("xw", "dy", "y", "dx", "done", "out")},
                      "used": False})
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def step(i):
        sl = slots[i % 2]
        ev, plan = sl["ev"], sl["plan"]
        c, q, o, ws, src = plan["cfg"], plan["q"], plan["out"], plan["ws"], plan["src"]
        with torch.cuda.stream(s_in):
            if sl["used"]:
                s_in.wait_event(ev["done"])  # the previous step on this slot has read its inputs
            sl["x"].copy_(xh, non_blocking=True)
            sl["w"].copy_(wh, non_blocking=True)
            ev["xw"].record(s_in)
            sl["dy"].copy_(dyh, non_blocking=True)
            ev["dy"].record(s_in)
        with torch.cuda.stream(s_comp):
            if sl["used"]:
                s_comp.wait_event(ev["out"])  # its outputs have been copied out
            s_comp.wait_event(ev["xw"])
            nv.nvfp4_quantize_dual(src["x"], c["x"], c["xt"], q["x"], q["xt"], workspace=ws)
            nv.nvfp4_quantize_dual(src["w"], c["w"], c["wt"], q["w"], q["wt"], workspace=ws)
            nv.nvfp4_gemm(q["x"], q["w"], nv.NVFP4_OUT_BF16, d=o["y"], workspace=ws)
            ev["y"].record(s_comp)
            s_comp.wait_event(ev["dy"])
            nv.nvfp4_quantize_dual(src["dy"], c["dy"], c["dyt"], q["dy"], q["dyt"], workspace=ws)
            nv.nvfp4_gemm(q["dy"], q["wt"], nv.NVFP4_OUT_BF16, d=o["dx"], workspace=ws)
            ev["dx"].record(s_comp)
            nv.nvfp4_gemm(q["dyt"], q["xt"], nv.NVFP4_OUT_BF16, d=o["dw"], workspace=ws)
            ev["done"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["y"])
            yh.copy_(o["y"], non_blocking=True)
            s_out.wait_event(ev["dx"])
            dxh.copy_(o["dx"], non_blocking=True)
            s_out.wait_event(ev["done"])
            dwh.copy_(o["dw"], non_blocking=True)
            ev["out"].record(s_out)
        sl["used"] = True

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    n = max(2, args.steps)
    t0.record(s_in)
    for i in range(n):
        step(i)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    ms = _max_over_ranks(ms, pg, dev)
    ms /= n
    for sl in slots:
        st = nv.nvfp4_check_device_status(sl["plan"]["ws"])
        if st != nv.NVFP4_OK:
            raise RuntimeError("device status %s (end-to-end run)" % nv.nvfp4_status_string(st))
    h2d = (T * HID + FFN * HID + T * FFN) * 2
    d2h = (T * FFN + T * HID + FFN * HID) * 2
    return {"value": round(_tflops(world, ms), 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "api": "nvfp4_quantize_dual + nvfp4_gemm with pinned host buffers; copy-in, compute and copy-out "
                   "streams overlap neighbouring steps"}


# ------------------------------------------------------------- CPU oracle
def _oracle_sample(rows=64):
    """The oracle on a bounded sample of the workload: for each of fprop,
    dgrad and wgrad, quantise the operand rows behind a rows x rows output
    block (the tensor scale still needs the whole operand) and accumulate
    that block in FP64.  Returns (flop, seconds)."""
    import oracle
    from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

    x, w, dy = syn.config2()
    xu, wu, dyu = syn.as_u16(x), syn.as_u16(w), syn.as_u16(dy)
    s = 0x5EEDC0DE0F4
    jobs = [
        (xu, oracle.make_cfg(block=0), wu, oracle.make_cfg(block=1), HID),
        (dyu, oracle.make_cfg(block=0), wu, oracle.make_cfg(block=1, transpose=1), FFN),
        (dyu, oracle.make_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=5),
         xu, oracle.make_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=6), T),
    ]
    t0 = time.perf_counter()
    flop = 0.0
    for a, ca, b, cb, K in jobs:
        qa = oracle.quantize_rows(a, ca, 0, rows)
        qb = oracle.quantize_rows(b, cb, 0, rows)
        oracle.gemm_f64(qa, qb, rows, rows, K)
        flop += 2.0 * rows * rows * K
    return flop, time.perf_counter() - t0


def cpu_baseline(args, rows=64):
    flop, sec = _oracle_sample(rows)
    return {"value": round(flop / sec / 1e12, 9), "unit": "TFLOP/s", "cores": 1, "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": "fprop+dgrad+wgrad, one %dx%d output block each at full K, with the operand rows "
                      "quantised from the full tensors (single-threaded C on one of the host's %d cores, %.1f s)"
                      % (rows, rows, os.cpu_count() or 1, sec)}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    times = []
    flop = 0.0
    for _ in range(args.warmup):
        _oracle_sample(16)
    for _ in range(args.steps):
        f, sec = _oracle_sample(16)
        flop = f
        times.append(sec)
    sec = sum(times) / len(times)
    value = flop / sec / 1e12
    line = {"metric": METRIC, "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (oracle: fp32 encode, fp64 accumulate)",
            "data": "synthetic", "config": _config(), "impl": "reference",
            "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "kind": "oracle", "cores": 1,
                             "host_cores": os.cpu_count(),
                             "sample": "per step: fprop+dgrad+wgrad, one 16x16 output block each at full K, "
                                       "single-threaded"},
            "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------- single kernels
def run_case(args):
    """Time one library call on one shape (for sweeps and ncu captures):
    ``gemm:M,N,K`` (BF16 output), ``quantize:R,C[,mode]`` with mode one of
    row, col, row16, col16, colsr (transform + stochastic rounding), or
    ``dual:R,C[,act|weight]`` (row + colsr, or row16 + col16, from one read),
    ``given:R,C[,mode]`` (one-pass quantiser with a supplied amax) or
    ``gemmq:M,N,K[,nod]`` (GEMM whose epilogue also quantises D along N under
    a supplied amax; ``nod``: D itself is not stored) or
    ``qadamw:R,C,m|v|mdec|vdec`` (optimizer-state codec on an FP32 state).
    Prints a JSON line with the mean time per call over --steps calls.
    ``mma[:iters]`` instead prints the isolated tensor-core instruction rates
    (block-scaled E2M1 and BF16, pair and single CTA)."""
    import torch

    import block_scaled_gemm_nvfp4_gb300 as nv
    from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

    kind, _, rest = args.case.partition(":")
    parts = rest.split(",")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    nv.lib()
    if kind == "mma":
        # the isolated tensor-core instruction rate: the ceiling of the GEMM's
        # tensor pipe (no counterpart in the pages; a roofline measurement)
        iters = int(parts[0]) if parts[0] else 4096
        out = {"case": args.case, "iters": iters, "unit": "TFLOP/s"}
        for k, name in nv.MMA_RATE_KINDS.items():
            tf, cyc = nv.nvfp4_debug_mma_rate(k, iters)
            out[name] = {"tflops": round(tf, 1), "cycles_per_mma": round(cyc, 2)}
        print(json.dumps(out), flush=True)
        return
    s = nv.NVFP4_DEFAULT_RHT_SEED
    modes = {"row": nv.quant_cfg(), "col": nv.quant_cfg(transpose=1), "row16": nv.quant_cfg(block=1),
             "col16": nv.quant_cfg(block=1, transpose=1),
             "colsr": nv.quant_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=5)}
    if kind == "gemm":
        M, N, K = (int(v) for v in parts[:3])
        qa = nv.nvfp4_quantize(syn.normal_bf16((M, K), seed=1).to(dev), nv.quant_cfg())
        qb = nv.nvfp4_quantize(syn.normal_bf16((N, K), seed=2).to(dev), nv.quant_cfg())
        d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(nv.nvfp4_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_gemm(qa, qb, nv.NVFP4_OUT_BF16, d=d, workspace=ws)
        work, unit = 2.0 * M * N * K / 1e12, "TFLOP/s"
    elif kind == "gemmq":
        M, N, K = (int(v) for v in parts[:3])
        store_d = not (len(parts) > 3 and parts[3] == "nod")
        qa = nv.nvfp4_quantize(syn.normal_bf16((M, K), seed=1).to(dev), nv.quant_cfg())
        qb = nv.nvfp4_quantize(syn.normal_bf16((N, K), seed=2).to(dev), nv.quant_cfg())
        amax_in = torch.full((1,), 40.0, dtype=torch.float32, device=dev)
        amax_out = torch.zeros(1, dtype=torch.float32, device=dev)
        d, q = nv.nvfp4_gemm_quantize(qa, qb, amax_in, store_d=store_d, amax_out=amax_out)
        ws = torch.zeros(4096, dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_gemm_quantize(qa, qb, amax_in, d=d, store_d=store_d, amax_out=amax_out, out=q, workspace=ws)
        work, unit = 2.0 * M * N * K / 1e12, "TFLOP/s"
    elif kind == "lora":
        # LoRA-SVD projection forward: U = BF16(X L1^T), then the NVFP4 GEMM with
        # the rank-r branch in the same accumulator (work counted: the NVFP4
        # GEMM's 2 M N K plus the branch's 2 T r (din + dout))
        T, din, dout, r = (int(v) for v in parts[:4])
        xq = nv.nvfp4_quantize(syn.normal_bf16((T, din), seed=1).to(dev), nv.quant_cfg())
        wq = nv.nvfp4_quantize(syn.normal_bf16((dout, din), std=0.02, seed=2).to(dev), nv.quant_cfg(block=1))
        x = syn.normal_bf16((T, din), seed=1).to(dev)
        l1 = syn.normal_bf16((r, din), std=0.02, seed=3).to(dev)
        l2 = syn.normal_bf16((dout, r), std=0.02, seed=4).to(dev)
        y, u = nv.nvfp4_lora_forward(xq, wq, x, l1, l2, 1.0)
        ws = torch.zeros(nv.nvfp4_lora_workspace_size(T, r), dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_lora_forward(xq, wq, x, l1, l2, 1.0, y=y, u=u, workspace=ws)
        work, unit = (2.0 * T * dout * din + 2.0 * T * r * (din + dout)) / 1e12, "TFLOP/s"
    elif kind == "ns":
        # one Newton-Schulz step with NVFP4 products on an iterate X [m, n]
        # (quintic coefficients); work counted: the three products'
        # 2 m m n + 2 m m m + 2 m m n FLOP
        m, n = int(parts[0]), int(parts[1])
        g = syn.normal_bf16((m, n), seed=5).float()
        x = (g / g.norm()).to(torch.bfloat16).to(dev)
        out = torch.empty_like(x)
        ws = torch.zeros(nv.nvfp4_ns_workspace_size(m, n), dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_ns_step(x, 15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0, out=out, workspace=ws)
        work, unit = (4.0 * m * m * n + 2.0 * m * m * m) / 1e12, "TFLOP/s"
    elif kind == "given":
        R, C = int(parts[0]), int(parts[1])
        cfg = modes[parts[2] if len(parts) > 2 else "row"]
        x = syn.normal_bf16((R, C), seed=3).to(dev)
        amax_in = x.abs().max().float().reshape(1)
        out = nv.nvfp4_quantize_given_amax(x, cfg, amax_in)
        ws = torch.zeros(nv.nvfp4_quantize_workspace_size(R, C, cfg), dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_quantize_given_amax(x, cfg, amax_in, out=out, workspace=ws)
        work, unit = R * C * QUANT_BYTES_PER_ELT / 1e9, "GB/s"
    elif kind == "qadamw":
        # optimizer-state codec: m | v (encode, two passes) or mdec | vdec
        R, C = int(parts[0]), int(parts[1])
        what = parts[2] if len(parts) > 2 else "m"
        g = torch.Generator().manual_seed(7)
        state = (torch.randn((R, C), generator=g) * 1e-3)
        if what in ("v", "vdec"):
            state = state * state
        state = state.to(dev)
        ws = torch.zeros(nv.nvfp4_qadamw_workspace_size(), dtype=torch.uint8, device=dev)
        s = nv.NVFP4_DEFAULT_RHT_SEED
        if what in ("m", "mdec"):
            enc = nv.nvfp4_qadamw_m_encode(state, s, 5, workspace=ws)
        else:
            enc = nv.nvfp4_qadamw_v_encode(state, s, workspace=ws)
        packed = QUANT_OUT_BYTES_PER_ELT + (2.0 / 256 if what in ("v", "vdec") else 0.0)
        if what == "m":
            def call():
                nv.nvfp4_qadamw_m_encode(state, s, 5, out=enc, workspace=ws)
        elif what == "v":
            def call():
                nv.nvfp4_qadamw_v_encode(state, s, out=enc, workspace=ws)
        elif what == "mdec":
            def call():
                nv.nvfp4_qadamw_m_decode(enc, s, out=state)
        else:
            def call():
                nv.nvfp4_qadamw_v_decode(enc, s, out=state)
        work, unit = R * C * (4.0 + packed) / 1e9, "GB/s"
    elif kind == "dual":
        R, C = int(parts[0]), int(parts[1])
        pair = {"act": (modes["row"], modes["colsr"]), "weight": (modes["row16"], modes["col16"])}
        ca, cb = pair[parts[2] if len(parts) > 2 else "act"]
        x = syn.normal_bf16((R, C), seed=3).to(dev)
        oa, ob = nv.nvfp4_quantize_dual(x, ca, cb)
        ws = torch.zeros(nv.nvfp4_quantize_workspace_size(R, C, ca), dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_quantize_dual(x, ca, cb, oa, ob, workspace=ws)
        work, unit = R * C * (2.0 + 2 * QUANT_OUT_BYTES_PER_ELT) / 1e9, "GB/s"
    elif kind == "quantize":
        R, C = int(parts[0]), int(parts[1])
        cfg = modes[parts[2] if len(parts) > 2 else "row"]
        x = syn.normal_bf16((R, C), seed=3).to(dev)
        out = nv.nvfp4_quantize(x, cfg)
        ws = torch.zeros(nv.nvfp4_quantize_workspace_size(R, C, cfg), dtype=torch.uint8, device=dev)

        def call():
            nv.nvfp4_quantize(x, cfg, out=out, workspace=ws)
        work, unit = R * C * QUANT_BYTES_PER_ELT / 1e9, "GB/s"
    else:
        raise SystemExit("unknown --case %r" % args.case)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    run = call
    if args.graph:
        # replay a captured CUDA graph of the call: no host launch cost
        # between calls (short kernels are otherwise host-bound)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        torch.cuda.synchronize()
        run = g.replay
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        run()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    st = nv.nvfp4_check_device_status(ws)
    if st != nv.NVFP4_OK:
        raise RuntimeError("device status %s" % nv.nvfp4_status_string(st))
    print(json.dumps({"case": args.case, "ms": round(ms, 5), "value": round(work / (ms * 1e-3), 1),
                      "unit": unit, "steps": args.steps, "warmup": args.warmup, "graph": bool(args.graph)}),
          flush=True)


# ------------------------------------------------------ measurement suite
def _suite_timer(torch, dev):
    """Per-call device time with L2 flushed before every call (a 256 MB
    write), so that inputs smaller than L2 are read from HBM."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def timed(call, iters=10, warmup=3):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        # The call is captured once in a CUDA graph and replayed, so the
        # timed region holds its kernels only (no host-side launch cost), and
        # everything is enqueued before the one synchronisation.
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        torch.cuda.synchronize()
        evs = []
        for _ in range(iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / iters

    return timed


def _oracle_quant_slice(args):
    """Worker: the oracle's encode of rows [r0, r1) of Q under the whole
    operand's amax (the delayed-scale entry point with amax = the operand's
    own amax gives the same output as a full quantisation)."""
    import oracle
    xs, cfg, amax = args
    return oracle.quantize_given_amax(xs, cfg, amax)[2]


def _oracle_amax_slice(args):
    import oracle
    xs, cfg = args
    return oracle.amax(xs, cfg)


def _oracle_suite(emit):
    """The oracle on full tensors of the quantise sweep's larger shape,
    single-threaded and on every host core (row slices in a spawn pool), and
    its FP64 GEMM on an output block of the MLP up-projection, extrapolated."""
    import multiprocessing as mp

    import oracle
    from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

    cores = os.cpu_count() or 1
    x = syn.as_u16(syn.config1(1))  # 8192 x 20480 with outliers
    R, C = x.shape
    for name, cfg in (("1x16 rne", oracle.make_cfg()),
                      ("1x16 sr+rht", oracle.make_cfg(rounding=1, rht=1, rht_seed=1, sr_seed=2))):
        t0 = time.perf_counter()
        oracle.quantize(x, cfg)
        t1 = time.perf_counter() - t0
        # all cores: amax of row slices, then the encode of row slices (the
        # transform and blocks run along rows, so slices are independent)
        step = (R + cores - 1) // cores
        slices = [(r, min(R, r + step)) for r in range(0, R, step)]
        with mp.get_context("spawn").Pool(cores) as pool:
            pool.map(_oracle_amax_slice, [(x[:16], cfg)] * cores)  # start the workers
            t0 = time.perf_counter()
            amax = max(pool.map(_oracle_amax_slice, [(x[a:b], cfg) for a, b in slices]))
            pool.map(_oracle_quant_slice, [(x[a:b], cfg, amax) for a, b in slices])
            tn = time.perf_counter() - t0
        gb = R * C * QUANT_BYTES_PER_ELT / 1e9
        emit({"suite": "oracle_quantize", "mode": name, "shape": [R, C], "threads_1_s": round(t1, 3),
              "threads_1_GBps": round(gb / t1, 4), "threads_all": cores, "threads_all_s": round(tn, 3),
              "threads_all_GBps": round(gb / tn, 4), "host_cores": cores})
    # FP64 GEMM: a 16 x 64 block of the MLP up-projection fprop at full K
    xw = syn.as_u16(syn.normal_bf16((16, HID), seed=1))
    ww = syn.as_u16(syn.normal_bf16((64, HID), std=0.02, seed=2))
    qa = oracle.quantize(xw, oracle.make_cfg())
    qb = oracle.quantize(ww, oracle.make_cfg(block=1))
    t0 = time.perf_counter()
    oracle.gemm_f64(qa, qb, 16, 64, HID)
    tg = time.perf_counter() - t0
    flop = 2.0 * 16 * 64 * HID
    emit({"suite": "oracle_gemm", "sample": "16x64 output block, K=%d, single thread" % HID,
          "s": round(tg, 4), "TFLOPs": round(flop / tg / 1e12, 9),
          "full_fprop_s_extrapolated": round(tg * (T * FFN) / (16 * 64), 1), "host_cores": cores})


def run_suite(args):
    """Every measurement the hot path's scope table asks for beyond the
    benchmark step, one JSON line each: the 16-mode quantise sweep at both
    sweep shapes (and the one-pass delayed-scale variant of each mode), the
    large and skinny GEMM probes, the 3B projection chain through the linear
    wrappers (split into quantise and GEMM), the LoRA-SVD and Newton-Schulz
    costs, and the oracle on the host cores."""
    import torch

    import block_scaled_gemm_nvfp4_gb300 as nv
    from block_scaled_gemm_nvfp4_gb300 import synthetic as syn

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    nv.lib()
    timed = _suite_timer(torch, dev)
    peaks, src = _peaks()
    hbm = peaks["hbm_gbs"]
    fp4 = peaks["bf16_tflops"] * FP4_OVER_BF16

    def emit(d):
        print(json.dumps(d), flush=True)

    with ClockSampler(0) as clocks:
        _suite_gpu(nv, syn, torch, dev, timed, hbm, fp4, emit)
    emit({"suite": "peaks", "hbm_gbs": hbm, "fp4_tflops": round(fp4, 1), "source": src,
          "clocks": clocks.summary()})
    _oracle_suite(emit)


def _suite_gpu(nv, syn, torch, dev, timed, hbm, fp4, emit):
    # quantise sweep: {1x16, 16x16} x {RNE, SR} x {transform off, on} at both shapes
    for si in range(2):
        xd = syn.config1(si).to(dev)
        R, C = xd.shape
        ws = torch.zeros(nv.nvfp4_quantize_workspace_size(R, C, nv.quant_cfg()), dtype=torch.uint8, device=dev)
        amax = xd.abs().max().float().reshape(1)
        for block in (0, 1):
            for rounding in (0, 1):
                for rht in (0, 1):
                    cfg = nv.quant_cfg(block=block, rounding=rounding, rht=rht, rht_seed=11, sr_seed=12)
                    out = nv.nvfp4_quantize(xd, cfg, workspace=ws)
                    ms = timed(lambda: nv.nvfp4_quantize(xd, cfg, out=out, workspace=ws))
                    gbs = R * C * QUANT_BYTES_PER_ELT / (ms * 1e-3) / 1e9
                    row = {"suite": "quantize", "shape": [R, C], "block": "16x16" if block else "1x16",
                           "rounding": "sr" if rounding else "rne", "rht": bool(rht), "ms": round(ms, 4),
                           "GBps": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                           "actual_two_pass_GBps": round(R * C * (QUANT_BYTES_PER_ELT + 2) / (ms * 1e-3) / 1e9, 1)}
                    if not rht:  # one pass under a supplied amax (delayed scaling)
                        ms1 = timed(lambda: nv.nvfp4_quantize_given_amax(xd, cfg, amax, out=out, workspace=ws))
                        g1 = R * C * QUANT_BYTES_PER_ELT / (ms1 * 1e-3) / 1e9
                        row.update({"given_amax_ms": round(ms1, 4), "given_amax_GBps": round(g1, 1),
                                    "given_amax_frac_hbm": round(g1 / hbm, 4)})
                    emit(row)
        assert nv.nvfp4_check_device_status(ws) == nv.NVFP4_OK
        del xd

    # GEMM probes: 16384^3 (tensor-bound) and the skinny decode shape (HBM-bound)
    for M, N, K in ((16384, 16384, 16384), (128, 8192, 8192)):
        a, b = syn.config4(M, N, K)
        qa = nv.nvfp4_quantize(a.to(dev), nv.quant_cfg())
        qb = nv.nvfp4_quantize(b.to(dev), nv.quant_cfg())
        d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        gws = torch.zeros(nv.nvfp4_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
        ms = timed(lambda: nv.nvfp4_gemm(qa, qb, nv.NVFP4_OUT_BF16, d=d, workspace=gws))
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        byts = (M + N) * K * QUANT_OUT_BYTES_PER_ELT + 2.0 * M * N
        emit({"suite": "gemm", "shape": [M, N, K], "ms": round(ms, 4), "TFLOPs": round(tf, 1),
              "frac_fp4": round(tf / fp4, 4), "algorithmic_MB": round(byts / 1e6, 1),
              "GBps": round(byts / (ms * 1e-3) / 1e9, 1), "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / hbm, 4)})
        del qa, qb, d

    # 3B projection chain through the linear wrappers (quantise both operands + GEMM)
    for name, din, dout in syn.PROJ3B:
        x, w, dy = (t.to(dev) for t in syn.config3(name))
        Tt = x.shape[0]
        for op, fn, a_src, b_src, shape in (
                ("fprop", nv.nvfp4_linear_fprop, x, w, (Tt, dout, din)),
                ("dgrad", nv.nvfp4_linear_dgrad, dy, w, (Tt, din, dout)),
                ("wgrad", nv.nvfp4_linear_wgrad, dy, x, (dout, din, Tt))):
            opc = {"fprop": nv.NVFP4_LINEAR_FPROP, "dgrad": nv.NVFP4_LINEAR_DGRAD, "wgrad": nv.NVFP4_LINEAR_WGRAD}[op]
            ws = torch.zeros(nv.nvfp4_linear_workspace_size(opc, Tt, din, dout), dtype=torch.uint8, device=dev)
            out = fn(a_src, b_src, workspace=ws)
            ms = timed(lambda: fn(a_src, b_src, workspace=ws, **{{"fprop": "y", "dgrad": "dx", "wgrad": "dw"}[op]: out}))
            # the GEMM alone on operands quantised the way the wrapper does
            M, N, K = shape
            if op == "fprop":
                qa = nv.nvfp4_quantize(x, nv.quant_cfg())
                qb = nv.nvfp4_quantize(w, nv.quant_cfg(block=1))
            elif op == "dgrad":
                qa = nv.nvfp4_quantize(dy, nv.quant_cfg())
                qb = nv.nvfp4_quantize(w, nv.quant_cfg(block=1, transpose=1))
            else:
                s = nv.NVFP4_DEFAULT_RHT_SEED
                qa = nv.nvfp4_quantize(dy, nv.quant_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=5))
                qb = nv.nvfp4_quantize(x, nv.quant_cfg(rounding=1, rht=1, transpose=1, rht_seed=s, sr_seed=6))
            msg = timed(lambda: nv.nvfp4_gemm(qa, qb, nv.NVFP4_OUT_BF16, d=out))
            flop = 2.0 * M * N * K
            emit({"suite": "linear3b", "proj": name, "op": op, "gemm_shape": [M, N, K], "ms": round(ms, 4),
                  "TFLOPs": round(flop / (ms * 1e-3) / 1e12, 1), "gemm_ms": round(msg, 4),
                  "gemm_TFLOPs": round(flop / (msg * 1e-3) / 1e12, 1), "gemm_frac_fp4": round(
                      flop / (msg * 1e-3) / 1e12 / fp4, 4), "quantize_ms": round(ms - msg, 4)})
            del qa, qb, out, ws
        del x, w, dy

    # LoRA-SVD forward (r = 64) against the plain GEMM on the 12B MLP-up fprop shape
    Tt, din, dout, r = T, HID, FFN, 64
    x = syn.normal_bf16((Tt, din), seed=1).to(dev)
    xq = nv.nvfp4_quantize(x, nv.quant_cfg())
    wq = nv.nvfp4_quantize(syn.normal_bf16((dout, din), std=0.02, seed=2).to(dev), nv.quant_cfg(block=1))
    l1 = syn.normal_bf16((r, din), std=0.02, seed=3).to(dev)
    l2 = syn.normal_bf16((dout, r), std=0.02, seed=4).to(dev)
    y, u = nv.nvfp4_lora_forward(xq, wq, x, l1, l2, 1.0)
    lws = torch.zeros(nv.nvfp4_lora_workspace_size(Tt, r), dtype=torch.uint8, device=dev)
    ms_l = timed(lambda: nv.nvfp4_lora_forward(xq, wq, x, l1, l2, 1.0, y=y, u=u, workspace=lws))
    ms_g = timed(lambda: nv.nvfp4_gemm(xq, wq, nv.NVFP4_OUT_BF16, d=y))
    emit({"suite": "lora_forward", "shape": [Tt, din, dout, r], "ms": round(ms_l, 4), "gemm_ms": round(ms_g, 4),
          "branch_overhead": round(ms_l / ms_g - 1.0, 4)})
    del x, xq, wq, l1, l2, y, u, lws

    # Newton-Schulz step with NVFP4 products
    for m, n in ((1024, 4096), (3072, 8192), (4096, 4096)):
        g = syn.normal_bf16((m, n), seed=5).float()
        xx = (g / g.norm()).to(torch.bfloat16).to(dev)
        out = torch.empty_like(xx)
        nws = torch.zeros(nv.nvfp4_ns_workspace_size(m, n), dtype=torch.uint8, device=dev)
        ms = timed(lambda: nv.nvfp4_ns_step(xx, 15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0, out=out, workspace=nws))
        flop = 4.0 * m * m * n + 2.0 * m * m * m
        emit({"suite": "ns_step", "shape": [m, n], "ms": round(ms, 4), "TFLOPs": round(flop / (ms * 1e-3) / 1e12, 1)})
        del xx, out, nws


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--graph", action="store_true", help="--case: time replays of a captured CUDA graph")
    ap.add_argument("--suite", action="store_true",
                    help="every scope-table measurement beyond the step: quantise sweep, GEMM probes, 3B chain, "
                         "LoRA, Newton-Schulz, oracle on the host cores")
    ap.add_argument("--case", default=None,
                    help="time one call: gemm:M,N,K, quantize:R,C[,mode] or dual:R,C[,act|weight]")
    args = ap.parse_args()
    if args.suite:
        run_suite(args)
    elif args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
