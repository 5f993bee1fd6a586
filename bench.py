"""Benchmark: W8A8 INT8 linear throughput (quantize + GEMM + epilogue) at Llama-3-8B shapes.

One step = the four linear layers of one Llama-3-8B decoder layer (QKV 6144x4096, O
4096x4096, gate_up 28672x4096, down 4096x14336) applied to M = 4096 token rows: per layer
the per-token activation quantizer and the INT8 GEMM with its fused epilogue.  value =
2*M*sum(N*K) / time, in TOPS, whole job over all ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-components]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no data-path
collective); rank 0 prints one JSON line.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload on the host cores.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

METRIC = "W8A8 linear TOPS (quant+GEMM) at Llama-3-8B shapes; % of INT8 tensor peak"
def engine_rate(key, default):
    """A rate recorded in profiles/engine_rates.md (written from the engine probe's output)."""
    p = os.path.join(HERE, "profiles", "engine_rates.md")
    try:
        for line in open(p):
            if line.startswith(key + ":"):
                return float(line.split(":", 1)[1])
    except (OSError, ValueError):
        pass
    return default


# measured dense rate of the GPU's only INT8 tensor instruction (warp MMA s8)
INT8_MMA_SYNC_TOPS = engine_rate("int8_mma_sync_tops", 158.5)
M_TOKENS = 4096
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def gemm_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was taken with the
    kernel source as it is now (else None: the counters are stale)."""
    import hashlib
    prof = os.path.join(HERE, "profiles", "gemm_tc_kernel_llama3_8b_m4096.md")
    src = os.path.join(HERE, "w8a8_int8_quantized_gb300", "csrc", "gemm_tc.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    text = open(prof).read()
    sha, per = None, {}
    for line in text.splitlines():
        line = line.strip()
        if line.startswith("source_sha256:"):
            sha = line.split(":", 1)[1].strip()
        elif line.startswith("traffic_bytes_per_launch:"):
            for kv in line.split(":", 1)[1].split():
                k, v = kv.split("=")
                per[k] = int(v)
    with open(src, "rb") as f:
        if sha is None or hashlib.sha256(f.read()).hexdigest() != sha or not per:
            return None
    return per


def load_peaks():
    p = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        if torch.cuda.is_available():
            pg.barrier(device_ids=[torch.cuda.current_device()])
        else:
            pg.barrier()


def max_over_ranks(pg, v):
    if pg is None:
        return v
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, v):
    if pg is None:
        return v
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


def bench_config(world):
    """The workload both arms run (the reference arm's bounded sample is stated in its
    cpu_baseline, not here)."""
    from w8a8_int8_quantized_gb300 import workloads as wl
    return {"workload": "llama3-8b-decoder-linears", "M": M_TOKENS,
            "shapes": [[n, N, K] for n, N, K in wl.llama_shapes()],
            "act": "dynamic per-token symmetric int8", "weight": "per-channel symmetric int8",
            "l2": "flushed between steps (256 MiB write outside the timed events)",
            "parallelism": f"replicas x{world} (independent batches)"}


def step_ops(M=M_TOKENS):
    from w8a8_int8_quantized_gb300 import workloads as wl
    return sum(2.0 * M * N * K for _, N, K in wl.llama_shapes())


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms.  Started (and given time to come up) before the
    warm-up, because its start-up stalled GPU work for tens of milliseconds when it began with
    the timed region; only samples stamped inside the timed window are reported."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.out = None
        self.window = None

    def start(self):
        try:
            self.out = open(os.path.join("/tmp", f"w8a8_clocks_{os.getpid()}.csv"), "w+")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(1.0)
        except Exception:
            self.proc = None

    def mark(self, t0, t1):
        """The timed window, as time.time() values."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.strip().split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        self.out.close()
        import datetime

        def in_window(r):
            if self.window is None:
                return True
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except (ValueError, IndexError):
                return False
            return self.window[0] - 0.2 <= ts <= self.window[1] + 0.2

        def summarize(sel):
            sm, smax, reasons = [], 0.0, set()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for r in sel:
                try:
                    sm.append(float(r[1]))
                    smax = max(smax, float(r[2]))
                    for nm, v in zip(names, r[5:9]):
                        if "Active" in v and "Not" not in v:
                            reasons.add(nm)
                except (ValueError, IndexError):
                    continue
            return sm, smax, reasons

        sm, smax, reasons = summarize([r for r in rows if in_window(r)])
        scope = "timed window"
        if not sm:  # no sample stamped inside a short window: report the whole loaded run
            sm, smax, reasons = summarize(rows)
            scope = "warm-up and timed region"
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "scope": scope}


# --------------------------------------------------------------------------- our arm
def run_ours(args, world, rank, pg):
    import w8a8_int8_quantized_gb300 as w8
    from w8a8_int8_quantized_gb300 import workloads as wl
    dev = "cuda"
    peaks, peak_src = load_peaks()
    seed = 1 + rank
    layers = []
    for name, N, K in wl.llama_shapes():
        x = wl.llama_activations(M_TOKENS, K, seed=seed, stream=10 + N % 97).to(dev)
        w = torch.randn(N, K, device=dev, generator=torch.Generator(device=dev).manual_seed(seed * 31 + N),
                        dtype=torch.float32).mul_(0.02).to(torch.bfloat16)
        wq, sw = w8.quantize_weight(w)
        del w
        packed = torch.empty(w8.act_packed_size(M_TOKENS, K), dtype=torch.uint8, device=dev)
        sx = torch.empty(M_TOKENS, dtype=torch.float32, device=dev)
        y = torch.empty((M_TOKENS, N), dtype=torch.bfloat16, device=dev)
        layers.append(dict(name=name, N=N, K=K, x=x, wq=wq, sw=sw, packed=packed, sx=sx, y=y))
    # K-split scratch (the tiles past a launch's last full wave of CTA pairs), shared by the
    # layers: the calls run one after another on one stream
    split_bytes = max(w8.splitk_workspace_size(M_TOKENS, L["N"], L["K"]) for L in layers)
    split_ws = torch.empty(max(split_bytes, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    lib = w8.lib()
    stream = torch.cuda.current_stream()
    sptr = __import__("ctypes").c_void_p(stream.cuda_stream)
    P = __import__("ctypes").c_void_p

    def step(record):
        # per layer: quantizer (packed output) then the GEMM with its fused epilogue; this is
        # exactly what w8a8_linear launches, split in two calls so each kernel can be timed
        for L in layers:
            e0 = torch.cuda.Event(enable_timing=True) if record else None
            e1 = torch.cuda.Event(enable_timing=True) if record else None
            e2 = torch.cuda.Event(enable_timing=True) if record else None
            if record:
                e0.record()
            rc = lib.w8a8_quantize_act_packed(P(L["x"].data_ptr()), M_TOKENS, L["K"], L["K"], 0,
                                              P(L["packed"].data_ptr()), P(L["sx"].data_ptr()), None, sptr)
            if record:
                e1.record()
            rc |= lib.w8a8_scaled_mm_packed(P(L["packed"].data_ptr()), P(L["wq"].data_ptr()), M_TOKENS, L["N"],
                                            L["K"], 0, P(L["sx"].data_ptr()), None, None, 0,
                                            P(L["sw"].data_ptr()), None, None, P(L["y"].data_ptr()),
                                            P(split_ws.data_ptr()), split_bytes, None, sptr)
            if record:
                e2.record()
                L.setdefault("ev", []).append((e0, e1, e2))
            if rc:
                raise RuntimeError("library call failed")

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for _ in range(args.warmup):
        step(False)
        flush.zero_()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    tw0 = time.time()
    step_events = []
    for _ in range(args.steps):
        flush.zero_()           # L2 flush between steps, outside the timed events
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        step(True)
        s1.record()
        step_events.append((s0, s1))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks.mark(tw0, time.time())
    clk = clocks.stop()
    barrier(pg)
    torch.cuda.synchronize()
    ms_total = sum(a.elapsed_time(b) for a, b in step_events)
    ms_total = max_over_ranks(pg, ms_total)
    ops = step_ops() * args.steps * world
    value = ops / (ms_total * 1e-3) / 1e12
    # per-kernel live timings (GEMM = dominant kernel)
    gemm_ms = 0.0
    quant_ms = 0.0
    gemm_flops = 0.0
    quant_bytes = 0.0
    quant_alg_bytes = 0.0
    per_layer = {}
    for L in layers:
        gq = sum(a.elapsed_time(b) for a, b, _ in L["ev"])
        gg = sum(b.elapsed_time(c) for _, b, c in L["ev"])
        n = len(L["ev"])
        quant_ms += gq
        gemm_ms += gg
        gemm_flops += 2.0 * M_TOKENS * L["N"] * L["K"] * n
        quant_bytes += (M_TOKENS * L["K"] * 4 + M_TOKENS * 8) * n   # bf16 in, fp16 codes out, scale + norm
        quant_alg_bytes += (M_TOKENS * L["K"] * 3 + M_TOKENS * 4) * n  # bf16 in, int8 codes out, scale
        per_layer[L["name"]] = {
            "N": L["N"], "K": L["K"],
            "gemm_us": round(gg / n * 1e3, 2), "quant_us": round(gq / n * 1e3, 2),
            "gemm_tflops": round(2.0 * M_TOKENS * L["N"] * L["K"] / (gg / n * 1e-3) / 1e12, 1),
            "linear_tops": round(2.0 * M_TOKENS * L["N"] * L["K"] / ((gg + gq) / n * 1e-3) / 1e12, 1),
        }
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tr = gemm_traffic()
    roofline = {
        "bound": "tensor", "kernel": "gemm_tc_kernel (tcgen05 kind::f16, int8 operands exact in fp16)",
        "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
        # mean DRAM bytes per GEMM launch over the four layer launches of a step (ncu, committed
        # under profiles/), null when the kernel source changed since the capture
        "traffic": (round(sum(tr[L["name"]] for L in layers) / len(layers)) if tr and all(
            L["name"] in tr for L in layers) else None),
        "traffic_per_layer": tr,
        "peak_source": f"{peak_src} bf16 burst (fp16 runs at the bf16 rate)",
        "per_launch_flops": "2*M*N*K of each GEMM launch (M=4096)",
        # sm_103a has no tcgen05 integer MMA kind; its one INT8 tensor path, the warp-level
        # mma.sync.m16n8k32.s8, was probed at this rate on the same GPUs
        # (profiles/engine_rates.md): the int8 products run instead as exact fp16 products
        # on the tcgen05 tensor cores (peak above)
        "int8_mma_sync_tops": INT8_MMA_SYNC_TOPS,
        "int8_mma_sync_source": "profiles/engine_rates.md (engine_probe.cu)",
        "achieved_over_int8_mma_sync": round(achieved / INT8_MMA_SYNC_TOPS, 2),
    }
    quant_gbs = quant_bytes / (quant_ms * 1e-3) / 1e9
    e2e = run_e2e(args, layers, w8, world, pg)
    comps = None
    if not args.no_components and rank == 0:
        comps = components(w8, wl, peaks)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic (seeded; random-init weights)",
        "config": bench_config(world),
        "e2e": e2e,
        # per layer: the quantizer, the GEMM and, when its tiles leave a partial last wave of
        # CTA pairs, the K-split reduce
        "gpu_launches": sum(2 + (1 if w8.splitk_workspace_size(M_TOKENS, L["N"], L["K"]) > 0 else 0)
                            for L in layers) * args.steps,
        "roofline": roofline,
        "kernels": {
            # the in-step quantizer writes the GEMM's fp16 operand (4 B per element moved);
            # the algorithmic figure counts the int8 rule's 3 B per element + 4 B per row
            "quantize_act_gbs": round(quant_gbs, 1),
            "quantize_act_frac_hbm": round(quant_gbs / float(peaks.get("hbm_gbs", 6800.0)), 4),
            "quantize_act_bytes_counted": "4 B/elem (bf16 in, fp16 codes out) + 8 B/row",
            "quantize_act_algorithmic_gbs": round(quant_alg_bytes / (quant_ms * 1e-3) / 1e9, 1),
            "quantize_act_algorithmic_frac_hbm": round(quant_alg_bytes / (quant_ms * 1e-3) / 1e9 / float(
                peaks.get("hbm_gbs", 6800.0)), 4),
            "per_layer": per_layer},
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    if comps is not None:
        line["components"] = comps
    return line


def run_e2e(args, layers, w8, world, pg):
    """Same step through the public API with host buffers: pinned H2D of every layer's x, the
    linear (w8a8_linear), D2H of every layer's y.  Copies run on their own streams and overlap
    the other layers' compute (layer i+1's input lands while layer i computes, y_i returns
    while later layers compute); device buffers are double-buffered across steps and every
    reuse waits on the event of the step that last touched it."""
    dev = "cuda"
    hx = [L["x"].cpu().pin_memory() for L in layers]
    hy = [torch.empty(L["y"].shape, dtype=torch.bfloat16).pin_memory() for L in layers]
    ws = [torch.empty(max(w8.linear_workspace_size(M_TOKENS, L["K"], "dyn_sym", L["N"]), 16), dtype=torch.uint8,
                      device=dev) for L in layers]
    dx = [[torch.empty_like(L["x"]) for L in layers] for _ in range(2)]
    dy = [[torch.empty_like(L["y"]) for L in layers] for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n = len(layers)
    ev_in = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]
    ev_comp = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]
    used = [[False] * n for _ in range(2)]
    step_no = [0]

    def step():
        b = step_no[0] % 2
        for i, L in enumerate(layers):
            with torch.cuda.stream(s_in):
                if used[b][i]:
                    s_in.wait_event(ev_comp[b][i])      # the linear that last read dx[b][i]
                dx[b][i].copy_(hx[i], non_blocking=True)
                ev_in[b][i].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[b][i])
                if used[b][i]:
                    s_comp.wait_event(ev_out[b][i])     # the copy that last read dy[b][i]
                w8.linear(dx[b][i], L["wq"], L["sw"], workspace=ws[i], out=dy[b][i])
                ev_comp[b][i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b][i])
                hy[i].copy_(dy[b][i], non_blocking=True)
                ev_out[b][i].record(s_out)
            used[b][i] = True
        step_no[0] += 1

    cur = torch.cuda.current_stream()

    def join():
        for st in (s_in, s_comp, s_out):
            e = torch.cuda.Event()
            e.record(st)
            cur.wait_event(e)

    for _ in range(max(1, args.warmup)):
        step()
    join()
    torch.cuda.synchronize()
    barrier(pg)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for st in (s_in, s_comp, s_out):
        st.wait_event(e0)
    for _ in range(args.steps):
        step()
    join()
    e1.record(cur)
    torch.cuda.synchronize()
    ms = max_over_ranks(pg, e0.elapsed_time(e1))
    value = step_ops() * args.steps * world / (ms * 1e-3) / 1e12
    return {"value": round(value, 2), "unit": "TOPS",
            "h2d_bytes_per_step": int(sum(L["x"].numel() * 2 for L in layers)),
            "d2h_bytes_per_step": int(sum(L["y"].numel() * 2 for L in layers)),
            "overlap": "copies on separate streams overlap other layers' compute"}


def _time_launches(fn, reps=10, warm=2, rounds=5):
    """Median device time of one fn() call, replayed from a CUDA graph so that host-side
    argument marshalling never shows up as device time.  Each event pair spans `reps`
    back-to-back replays (event timestamps tick in steps of about 2 us, too coarse for one
    launch of a few tens of microseconds); the median is over `rounds` such pairs."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    evs = []
    for _ in range(rounds):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) / reps for a, b in evs)


def components(w8, wl, peaks):
    """Per-row measurements of the other hot-path steps (not part of `value`)."""
    dev = "cuda"
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    tf = float(peaks.get("bf16_tflops", 1900.0))
    out = {}
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_words = flush_buf.view(torch.int32)

    class _Flush:
        """L2 flush before each component launch: a 256 MiB write, then a read of the same
        buffer, so the write's dirty lines are written back before the measured kernel
        instead of during it (a short kernel would otherwise be charged up to ~129 MB of
        write-back that is not its own).  Its own time is subtracted."""

        @staticmethod
        def zero_():
            flush_buf.zero_()
            flush_words.sum()

    flush = _Flush()
    out["flush"] = "256 MiB write + read of the same buffer before each launch, its time subtracted"
    # S1 / S2 quantizers at M = 8192
    for K in (4096, 14336):
        x = wl.llama_activations(8192, K, seed=5).to(dev)
        for mode in ("dyn_sym", "dyn_asym"):
            def f():
                flush.zero_()
            ms_flush = _time_launches(f)
            ms = _time_launches(lambda: (flush.zero_(), w8.quantize_act(x, mode))) - ms_flush
            b = 8192 * K * 3 + 8192 * 4 * (2 if mode == "dyn_asym" else 1)
            out[f"quant_{mode}_M8192_K{K}"] = {"us": round(ms * 1e3, 2), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                                                "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
        del x
        # the affine rule on its own workload, rows ~ N(0.5, 1): bf16 quotients land on or next
        # to half-integers far more often there, and each such value is decided by a division
        x = wl.asym_activations(8192, K, seed=5).to(dev)
        ms = _time_launches(lambda: (flush.zero_(), w8.quantize_act(x, "dyn_asym"))) - ms_flush
        b = 8192 * K * 3 + 8192 * 8
        out[f"quant_dyn_asym_M8192_K{K}_nonzero_mean_rows"] = {
            "us": round(ms * 1e3, 2), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
            "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
        del x
    # S7 weight quantizer (+ azp_adj) on the four Llama-3-8B weights
    for N, K in ((6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336)):
        w = torch.randn(N, K, device=dev, dtype=torch.float32).mul_(0.02).to(torch.bfloat16)
        ms = _time_launches(lambda: (flush.zero_(), w8.quantize_weight(w, with_azp_adj=True))) - ms_flush
        b = N * K * 3 + N * 8
        out[f"quant_weight_{N}x{K}"] = {"us": round(ms * 1e3, 2), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                                        "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
        del w
    # fused Q/K/V weight with per-partition tensor scales -> one (max) scale, in place
    wq = torch.randint(-127, 128, (6144, 4096), dtype=torch.int8, device=dev)
    sc = torch.tensor([1.1e-3, 1.7e-3, 1.3e-3], dtype=torch.float32, device=dev)
    ms = _time_launches(lambda: (flush.zero_(), w8.requantize_max_scale(wq, sc, [4096, 1024, 1024]))) - ms_flush
    b = 6144 * 4096 * 2
    out["requant_max_scale_qkv_6144x4096"] = {"us": round(ms * 1e3, 2), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                                              "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
    del wq
    # S8 requant: 64 x [6144, 4096] + 8 x [3000, 1500], one batched call
    g = torch.Generator(device=dev).manual_seed(7)
    mats = []
    for N, K, cnt in ((6144, 4096, 64), (3000, 1500, 8)):
        for _ in range(cnt):
            c = torch.randn(N, K, device=dev, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
            s = torch.exp(torch.empty((N + 127) // 128, (K + 127) // 128, device=dev).uniform_(
                np.log(1e-4), np.log(1e-2), generator=g))
            mats.append((c, s))
    outs = [(torch.empty(c.shape, dtype=torch.int8, device=dev), torch.empty(c.shape[0], device=dev))
            for c, _ in mats]
    ms = _time_launches(lambda: w8.fp8block_to_int8_rowwise_batched(mats, outs), reps=5)
    b = sum(c.numel() * 2 + c.shape[0] * 4 + s.numel() * 4 for c, s in mats)
    out["requant_64x6144x4096_plus_8x3000x1500"] = {"us": round(ms * 1e3, 1),
                                                    "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                                                    "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
    # the same conversion writing each weight's azp_adj (row sums of the codes) in the pass
    outs = [o + (torch.empty(o[0].shape[0], dtype=torch.int32, device=dev),) for o in outs]
    ms = _time_launches(lambda: w8.fp8block_to_int8_rowwise_batched(mats, outs, azp_adj=True), reps=5)
    b += sum(c.shape[0] * 4 for c, _ in mats)
    out["requant_with_azp_adj_64x6144x4096_plus_8x3000x1500"] = {
        "us": round(ms * 1e3, 1), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
        "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
    del mats, outs
    # S2/S3 asymmetric linears, K = N = 4096
    for M in (128, 4096):
        x = wl.asym_activations(M, 4096, seed=3).to(dev)
        w = torch.randn(4096, 4096, device=dev).mul_(0.02).to(torch.bfloat16)
        wq, sw, adj, wsq = w8.quantize_weight(w, with_azp_adj=True, with_sumsq=True)
        ws = torch.empty(w8.linear_workspace_size(M, 4096, "dyn_asym", 4096), dtype=torch.uint8, device=dev)
        yb = torch.empty(M, 4096, dtype=torch.bfloat16, device=dev)
        ms = _time_launches(lambda: w8.linear(x, wq, sw, act_mode="dyn_asym", azp_adj=adj, workspace=ws, out=yb,
                                              w_sumsq=wsq))
        out[f"linear_dyn_asym_M{M}_4096x4096"] = {"us": round(ms * 1e3, 2),
                                                  "TOPS": round(2 * M * 4096 * 4096 / (ms * 1e-3) / 1e12, 1)}
        if M == 4096:
            # static per-tensor asymmetric (config 3b): scale and int8 zero point of the whole tensor
            xf = x.float()
            lo, hi = float(xf.min()), float(xf.max())
            sc = torch.tensor([(hi - lo) / 255.0], dtype=torch.float32, device=dev)
            zp = torch.tensor([max(-128, min(127, round(-128 - lo / float(sc))))], dtype=torch.int32, device=dev)
            adj_s = w8.azp_adj(wq, zp)
            ws_s = torch.empty(w8.linear_workspace_size(M, 4096, "static_asym"), dtype=torch.uint8, device=dev)
            ms = _time_launches(lambda: w8.linear(x, wq, sw, act_mode="static_asym", input_scale=sc,
                                                  input_zero_point=zp, azp_adj=adj_s, workspace=ws_s, out=yb,
                                                  w_sumsq=wsq))
            out["linear_static_asym_M4096_4096x4096"] = {"us": round(ms * 1e3, 2),
                                                         "TOPS": round(2 * M * 4096 * 4096 / (ms * 1e-3) / 1e12, 1)}
    # the whole Llama-3-8B grid: every linear at M in {1, 16, 128, 1024, 8192} (M = 4096 is the
    # headline step), quantizer + GEMM through w8a8_linear with the K-split scratch, L2
    # flushed before each launch (its own time subtracted).  M <= 16 streams the weight
    # (fraction of HBM over weight + activation + output bytes); larger M is tensor-bound
    # (fraction of the bf16 peak the fp16 products run at).
    f0 = _time_launches(lambda: flush.zero_())
    for name, N, K in wl.llama_shapes():
        wq = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev)
        sw = torch.rand(N, device=dev).mul_(1e-3)
        for M in (1, 16, 128, 1024, 8192):
            x = wl.llama_activations(M, K, seed=4).to(dev)
            ws = torch.empty(max(w8.linear_workspace_size(M, K, "dyn_sym", N), 16), dtype=torch.uint8, device=dev)
            yb = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            ms = _time_launches(lambda: (flush.zero_(), w8.linear(x, wq, sw, workspace=ws, out=yb)), reps=5) - f0
            tops = 2 * M * N * K / (ms * 1e-3) / 1e12
            e = {"us": round(ms * 1e3, 2), "TOPS": round(tops, 2)}
            if M <= 16:
                b = N * K + M * K * 2 + M * N * 2 + N * 4
                e["GBps"] = round(b / (ms * 1e-3) / 1e9, 1)
                e["frac_hbm"] = round(b / (ms * 1e-3) / 1e9 / hbm, 3)
            else:
                e["frac_tensor"] = round(tops / tf, 3)
            out[f"linear_{name}_{N}x{K}_M{M}"] = e
            del x, ws, yb
        del wq, sw
    # S9 MoE layer (4096 tokens, 32 experts, top-4)
    md = moe_device_inputs(w8, wl)
    ms = _time_launches(lambda: w8.moe_forward(*md["args"], **md["kw"]), reps=5)
    out["moe_T4096_E32_top4"] = {"us": round(ms * 1e3, 1), "TOPS": round(md["ops"] / (ms * 1e-3) / 1e12, 1),
                                 "frac_tensor": round(md["ops"] / (ms * 1e-3) / 1e12 / tf, 3)}
    # routing on the GPU (top-4 of 32 + counting sort), alone and in front of the layer
    logits = wl.moe_workload(T=4096, H=64, E=32, topk=4, inter=64, seed=0, with_weights=False)["logits"].to(dev)
    rws = torch.empty(max(w8.lib().w8a8_moe_route_workspace_size(4096, 32, 4), 4), dtype=torch.uint8, device=dev)
    ms = _time_launches(lambda: w8.moe_route(logits, 4, workspace=rws), reps=20)
    out["moe_route_T4096_E32_top4"] = {"us": round(ms * 1e3, 2)}
    x, _, _, _, _, w13, s13, w2, s2 = md["args"]

    def routed_layer():
        ids, tw, seg, row_index, row_of = w8.moe_route(logits, 4, workspace=rws)
        return w8.moe_forward(x, row_index, seg, row_of, tw, w13, s13, w2, s2, **md["kw"])
    ms = _time_launches(routed_layer, reps=5)
    out["moe_T4096_E32_top4_with_routing"] = {"us": round(ms * 1e3, 1),
                                              "TOPS": round(md["ops"] / (ms * 1e-3) / 1e12, 1)}
    return out


def moe_device_inputs(w8, wl, T=4096, H=4096, E=32, topk=4, inter=1408):
    """Routing from the seeded workload, expert weights drawn on the device and prepared once
    (per-channel quantization, row sums of squares), rows sorted by expert."""
    dev = "cuda"
    d = wl.moe_workload(T=T, H=H, E=E, topk=topk, inter=inter, seed=0, with_weights=False)
    ids = d["topk_ids"].numpy().reshape(-1)
    order = np.argsort(ids, kind="stable")
    counts = np.bincount(ids, minlength=E)
    seg = np.zeros(E + 1, np.int64)
    seg[1:] = np.cumsum(counts)
    row_of = np.zeros(T * topk, np.int64)
    row_of[order] = np.arange(T * topk)
    g = torch.Generator(device=dev).manual_seed(11)
    w13 = torch.randn(E * 2 * inter, H, device=dev, generator=g).mul_(0.02).to(torch.bfloat16)
    w2 = torch.randn(E * H, inter, device=dev, generator=g).mul_(0.02).to(torch.bfloat16)
    w13q, s13 = w8.quantize_weight(w13)
    w2q, s2 = w8.quantize_weight(w2)
    del w13, w2
    args = (d["x"].to(dev), torch.from_numpy(order // topk).to(dev), torch.from_numpy(seg).to(dev),
            torch.from_numpy(row_of.reshape(T, topk)).to(dev), d["topk_w"].to(dev),
            w13q.view(E, 2 * inter, H), s13.view(E, 2 * inter), w2q.view(E, H, inter), s2.view(E, H))
    ops = 2.0 * T * topk * (2 * inter * H + H * inter)
    kw = {"w13_sumsq": w8.weight_sumsq(w13q).view(E, 2 * inter), "w2_sumsq": w8.weight_sumsq(w2q).view(E, H)}
    return {"args": args, "ops": ops, "kw": kw}


# --------------------------------------------------------------------------- reference arm (CPU oracle)
def run_reference(args, world, rank):
    import oracle
    from w8a8_int8_quantized_gb300 import workloads as wl
    sample_rows = 32
    prepared = []
    for name, N, K in wl.llama_shapes():
        x = wl.llama_activations(sample_rows, K, seed=1, stream=10 + N % 97)
        w = wl.weight_bf16(N, K, seed=2)
        rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
        prepared.append((wl.bits(x), rq, rs, N, K))
    ops_per_rep = sum(2.0 * sample_rows * N * K for _, _, _, N, K in prepared)

    def rep():
        for xb, rq, rs, N, K in prepared:
            oracle.w8a8_linear(xb, rq, rs)

    for _ in range(args.warmup):
        rep()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rep()
    dt = time.perf_counter() - t0
    value = ops_per_rep * args.steps / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded; random-init weights)",
        "config": bench_config(world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": f"{sample_rows} of {M_TOKENS} token rows per layer, all four layers, per step"},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline_leg():
    """The oracle as it stands, on a bounded sample of the step (about 10 s of host work)."""
    import oracle
    from w8a8_int8_quantized_gb300 import workloads as wl
    sample_rows = 32
    prepared = []
    for name, N, K in wl.llama_shapes():
        x = wl.llama_activations(sample_rows, K, seed=1)
        w = wl.weight_bf16(N, K, seed=2)
        rq, rs = oracle.quantize_weight_per_channel(w.float().numpy())
        prepared.append((wl.bits(x), rq, rs, N, K))
    ops = sum(2.0 * sample_rows * N * K for _, _, _, N, K in prepared)
    reps, t0 = 0, time.perf_counter()
    while True:
        for xb, rq, rs, N, K in prepared:
            oracle.w8a8_linear(xb, rq, rs)
        reps += 1
        if time.perf_counter() - t0 > 8.0:
            break
    dt = time.perf_counter() - t0
    return {"value": round(ops * reps / dt / 1e12, 6), "unit": "TOPS", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{sample_rows} token rows x 4 Llama-3-8B layers, repeated {reps}x (weights pre-quantized)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-components", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # the CPU oracle on rank 0 only; the other ranks exit at once (no collective needed)
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    world, rank, local, pg = dist_setup(args)
    line = run_ours(args, world, rank, pg)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline_leg()
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
