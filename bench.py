#!/usr/bin/env python3
"""Benchmark: scaled FP8 quantize -> FP8 GEMM on one transformer layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fp8q|reference]

One step is one pass of the whole path over one layer's synthetic inputs:
the 12 GEMMs (Fprop / Dgrad / Wgrad of QKV, attention out, MLP up, MLP down;
M = 31 x 512 = 15872 tokens, hidden 4096, FFN 16384) with per-tensor current
scaling, in autocast mode: every step takes the amax of x, w and grad_out,
derives their scales and casts them (E4M3 / E5M2, each with its transposed
copy for the backward GEMMs) before the GEMMs, as the low-precision-training
blog post's autocast timing does for its FP8 CurrentScaling recipe.  The
headline value is whole-job TFLOP/s of that step (2 M N K summed over the 12
GEMMs / step time).  The same line also reports the prequantized step (GEMM
kernels only), delayed scaling of the gradient, the same layer with 1x128 /
128x128 block scaling (autocast and prequant), quantize GB/s on the
8192x4096 activation, the dominant kernels' rooflines, an end-to-end figure
with host buffers, the oracle timed on the host cores, and SM clocks sampled
during the timed region.

Under torchrun each rank runs an independent replica of the step on its own
GPU (no data-path collective; weak scaling); timings are maxed over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 GEMM TFLOP/s (autocast & prequant) + quantize GB/s, % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # nominal dense FP8 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)
L2_BYTES = 126 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["fp8q", "reference"], default="fp8q")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the oracle on the host cores")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                    help="run one kernel on a small case three times for an ncu capture "
                         "(prints no bench line)")
    return ap.parse_args()


# Small cases for ncu captures: operands about L2-sized or larger, a few
# hundred MB on the device, three launches of the kernel under study.
PROFILE_CASES = {
    "gemm_tensor": "8192x8192x8192 per-tensor E4M3 GEMM, bf16 out",
    "gemm_block": "8192x8192x8192 1x128 x 128x128 GEMM, bf16 out",
    "gemm_tile": "8192x8192x8192 1x128 x 1x128 GEMM (wgrad form), bf16 out",
    "gemm_row": "8192x8192x8192 row-scaled x row-scaled E4M3 GEMM, bf16 out",
    "quant_tile_dual": "16384x8192 bf16, 1x128 row and column tiles, E4M3",
    "quant_tile_rows": "16384x8192 bf16, 1x128 row tiles, E4M3",
    "quant_block": "16384x8192 bf16, 128x128 blocks + transposed copy, E4M3",
    "quant_rowwise": "16384x8192 bf16, row-wise scales, q and the transposed copy, E4M3",
    "quant_tensor_dual": "16384x8192 bf16, per-tensor scale, q and the transposed copy, E4M3",
    "amax": "16384x8192 bf16 amax",
    "quant_activation": ("the bench's 8192x4096 activation, 1x128 row tiles, E4M3, L2 flushed "
                         "before each of the three calls"),
    "quant_mx_dual": "16384x8192 bf16, MXFP8 1x32 row and 32x1 column blocks, E4M3",
    "amax_activation": "the bench's 8192x4096 activation, amax, L2 flushed before each of three calls",
    "gemm_mx": "8192x8192x8192 MXFP8 x MXFP8 GEMM, bf16 out",
}
# One linear of the layer, its Fprop, Dgrad and Wgrad once each (three GEMM
# launches after the quantisation): layer_<recipe>_<linear>.
for _rc in ("tensor", "block", "mx"):
    for _ln in ("qkv", "attn_out", "mlp_up", "mlp_down"):
        PROFILE_CASES[f"layer_{_rc}_{_ln}"] = (f"the layer's {_ln} Fprop, Dgrad and Wgrad, "
                                               f"{_rc} scaling, bf16 out")


def run_profile_case(case: str):
    import torch
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    import workloads
    build_lib.build()
    fq.load_library()
    if case.startswith("layer_"):
        recipe, name = case[len("layer_"):].split("_", 1)
        idx = [s.name for s in workloads.LAYER].index(name)
        x, w, g = (t.cuda() for t in workloads.layer_inputs(workloads.LAYER[idx], idx))
        if recipe == "tensor":
            qx, qxt, sx = fq.fp8_quantize_tensor(x, fq.E4M3, fq.fp8_amax(x), want_qt=True)
            qw, qwt, sw = fq.fp8_quantize_tensor(w, fq.E4M3, fq.fp8_amax(w), want_qt=True)
            qg, qgt, sg = fq.fp8_quantize_tensor(g, fq.E5M2, fq.fp8_amax(g), want_qt=True)
            T = fq.GemmOperand.tensor
            ops = [(fq.fp8_gemm_fprop, T(qx, 0, sx), T(qw, 0, sw)),
                   (fq.fp8_gemm_dgrad, T(qg, 1, sg), T(qwt, 0, sw)),
                   (fq.fp8_gemm_wgrad, T(qgt, 1, sg), T(qxt, 0, sx))]
        elif recipe == "block":
            qx, sx, qxt, sxt = fq.fp8_quantize_tile1x128(x, fq.E4M3, rows=True, cols=True)
            qw, qwt, sw = fq.fp8_quantize_block128x128(w, fq.E4M3, want_q=True, want_qt=True)
            qg, sg, qgt, sgt = fq.fp8_quantize_tile1x128(g, fq.E5M2, rows=True, cols=True)
            T, B, BT = fq.GemmOperand.tile, fq.GemmOperand.block, fq.GemmOperand.block_transposed
            ops = [(fq.fp8_gemm_fprop, T(qx, 0, sx), B(qw, 0, sw)),
                   (fq.fp8_gemm_dgrad, T(qg, 1, sg), BT(qwt, 0, sw)),
                   (fq.fp8_gemm_wgrad, T(qgt, 1, sgt), T(qxt, 0, sxt))]
        else:
            qx, sx, qxt, sxt = fq.fp8_quantize_mxfp8(x, fq.E4M3, rows=True, cols=True)
            qw, sw, qwt, swt = fq.fp8_quantize_mxfp8(w, fq.E4M3, rows=True, cols=True)
            qg, sg, qgt, sgt = fq.fp8_quantize_mxfp8(g, fq.E5M2, rows=True, cols=True)
            X = fq.GemmOperand.mx
            ops = [(fq.fp8_gemm_fprop, X(qx, 0, sx), X(qw, 0, sw)),
                   (fq.fp8_gemm_dgrad, X(qg, 1, sg), X(qwt, 0, swt)),
                   (fq.fp8_gemm_wgrad, X(qgt, 1, sgt), X(qxt, 0, sxt))]
        del x, w, g
        for fn, A, B in ops:
            fn(A, B)
    elif case == "quant_mx_dual":
        x = workloads.normal((16384, 8192), 1.0, 902).cuda()
        for _ in range(3):
            fq.fp8_quantize_mxfp8(x, fq.E4M3, rows=True, cols=True)
    elif case.startswith("gemm"):
        M = N = K = 8192
        a = workloads.normal((M, K), 1.0, 900).cuda()
        b = workloads.normal((N, K), 0.02, 901).cuda()
        if case == "gemm_tensor":
            qa, _, sa = fq.fp8_quantize_tensor(a, fq.E4M3, fq.fp8_amax(a))
            qb, _, sb = fq.fp8_quantize_tensor(b, fq.E4M3, fq.fp8_amax(b))
            A, B = fq.GemmOperand.tensor(qa, 0, sa), fq.GemmOperand.tensor(qb, 0, sb)
        elif case == "gemm_mx":
            qa, sa, _, _ = fq.fp8_quantize_mxfp8(a, fq.E4M3)
            qb, sb, _, _ = fq.fp8_quantize_mxfp8(b, fq.E4M3)
            A, B = fq.GemmOperand.mx(qa, 0, sa), fq.GemmOperand.mx(qb, 0, sb)
        elif case == "gemm_row":
            qa, sa, _, _ = fq.fp8_quantize_rowwise(a, fq.E4M3)
            qb, sb, _, _ = fq.fp8_quantize_rowwise(b, fq.E4M3)
            A, B = fq.GemmOperand.row(qa, 0, sa), fq.GemmOperand.row(qb, 0, sb)
        else:
            qa, sa, _, _ = fq.fp8_quantize_tile1x128(a, fq.E4M3)
            A = fq.GemmOperand.tile(qa, 0, sa)
            if case == "gemm_block":
                qb, _, sb = fq.fp8_quantize_block128x128(b, fq.E4M3)
                B = fq.GemmOperand.block(qb, 0, sb)
            else:
                qb, sb, _, _ = fq.fp8_quantize_tile1x128(b, fq.E4M3)
                B = fq.GemmOperand.tile(qb, 0, sb)
        del a, b
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            fq.fp8_gemm(A, B, out=out)
    elif case in ("quant_activation", "amax_activation"):
        x, _ = workloads.quantize_activation()
        x = x.cuda()
        flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        for _ in range(3):
            flush_buf.fill_(1.0)
            if case == "amax_activation":
                fq.fp8_amax(x)
            else:
                fq.fp8_quantize_tile1x128(x, fq.E4M3, rows=True)
    else:
        x = workloads.normal((16384, 8192), 1.0, 902).cuda()
        for _ in range(3):
            if case == "quant_tile_dual":
                fq.fp8_quantize_tile1x128(x, fq.E4M3, rows=True, cols=True)
            elif case == "quant_tile_rows":
                fq.fp8_quantize_tile1x128(x, fq.E4M3, rows=True)
            elif case == "quant_tensor_dual":
                fq.fp8_quantize_tensor(x, fq.E4M3, fq.fp8_amax(x), want_q=True, want_qt=True)
            elif case == "quant_rowwise":
                fq.fp8_quantize_rowwise(x, fq.E4M3, rows=True, cols=True)
            elif case == "quant_block":
                fq.fp8_quantize_block128x128(x, fq.E4M3, want_q=True, want_qt=True)
            else:
                fq.fp8_amax(x)
    torch.cuda.synchronize()
    if fq.device_status() != 0:
        raise SystemExit("profile case: a kernel reported a barrier timeout")
    print(f"profile case {case} done: {PROFILE_CASES[case]}")


KERNEL_SOURCES = {
    "gemm_tensor_pair_kernel": ("fp8q_gemm.cu", "fp8q_gemm_common.cuh", "fp8q_ptx.cuh"),
    "gemm_blockscaled_kernel": ("fp8q_gemm_block.cu", "fp8q_gemm_common.cuh", "fp8q_ptx.cuh"),
    "gemm_mx_kernel": ("fp8q_gemm_mx.cu", "fp8q_gemm_common.cuh", "fp8q_ptx.cuh"),
    "quant2d_tile_rows": ("fp8q_quant.cu", "fp8q_ptx.cuh"),
}


def kernel_source_digest(key: str) -> str:
    """sha256 over the source files a kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[key]:
        with open(os.path.join(ROOT, "scaled_quantize_fp8_warp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(key: str):
    """DRAM bytes per launch for a kernel, from profiles/roofline_traffic.json,
    only if the kernel's sources are unchanged since that capture (their
    sha256 is stored with the figure); otherwise None."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(key)
        digest = kernel_source_digest(key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha256") != digest:
        return None
    return rec.get("bytes_per_launch")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- distributed

class Dist:
    def __init__(self):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi for this process's GPU every 50 ms while the layer
    phases run; time_steps() records the wall-clock window of each timed
    region, and the summary keeps only the samples whose own nvidia-smi
    timestamp falls inside one of those windows."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.windows = []   # (t0, t1) wall-clock seconds of the timed regions

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2 * self.PERIOD_MS / 1000)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    @staticmethod
    def _epoch(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self, windows=None, span=None):
        """Clocks over the given timed regions (default: every region
        recorded)."""
        windows = self.windows if windows is None else windows
        rows, in_window = [], []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and parts[1] != self.uuid:
                continue
            rows.append(parts[1:])
            t = self._epoch(parts[0])
            if t is not None and any(a <= t <= b for a, b in windows):
                in_window.append(parts[1:])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        use = in_window if in_window else rows
        num = lambda v: v.replace(".", "").isdigit()
        sm = [float(r[1]) for r in use if num(r[1])]
        smax = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i] == "Active"})
        power = [float(r[3]) for r in use if num(r[3])]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "samples_in_timed_regions": len(in_window),
                "power_w_median": statistics.median(power) if power else None,
                "power_w_max": max(power) if power else None,
                "period_ms": self.PERIOD_MS,
                "span": span or ("the timed regions of the layer phases (per-tensor, "
                                 "delayed, block-scaled, MXFP8, row-wise)")}


# Clock-event reasons that void a number measured while they were active; a
# power cap (sw_power_cap) does not: a dense FP8 GEMM step meets it on this part.
REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clock_rejection(summary: dict, stuck_frac: float = 0.8) -> list:
    """Why a timed region's clock record voids its number: a hardware or
    thermal slowdown reported during it, or a median SM clock below
    stuck_frac of the maximum with no reason reported at all (a clock lock
    left behind).  Empty when the number stands."""
    reasons = summary.get("reasons") or []
    causes = [r for r in reasons if r in REJECTING_REASONS]
    sm, smax = summary.get("sm_mhz"), summary.get("sm_max_mhz")
    if not reasons and sm and smax and sm < stuck_frac * smax:
        causes.append(f"median SM clock {sm:.0f} MHz of {smax:.0f} with no reason reported")
    return causes


# ------------------------------------------------------------- layer buffers

class LayerState:
    """Device (and pinned host) buffers for one layer step, for every recipe."""

    def __init__(self, fq, torch, with_host: bool):
        import workloads
        self.fq, self.torch = fq, torch
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        self.linears = []
        self.flops = workloads.gemm_flops()
        self.h2d_bytes = 0
        self.d2h_bytes = 0
        for i, shape in enumerate(workloads.LAYER):
            x, w, g = workloads.layer_inputs(shape, i)
            M, K, N = x.shape[0], shape.K, shape.N
            L = {"shape": shape, "M": M, "K": K, "N": N}
            if with_host:
                L["x_h"], L["w_h"], L["g_h"] = x.pin_memory(), w.pin_memory(), g.pin_memory()
                self.h2d_bytes += sum(t.numel() * t.element_size() for t in (x, w, g))
            L["x"], L["w"], L["g"] = x.to(dev), w.to(dev), g.to(dev)
            u8, f32, bf16 = torch.uint8, torch.float32, torch.bfloat16
            e = lambda shp, dt: torch.empty(shp, dtype=dt, device=dev)
            # FP8 operands in both orientations, with their scales
            L["qx"], L["qxt"] = e((M, K), u8), e((K, M), u8)
            L["qw"], L["qwt"] = e((N, K), u8), e((K, N), u8)
            L["qg"], L["qgt"] = e((M, N), u8), e((N, M), u8)
            L["sx"], L["sxt"] = e(((K + 127) // 128, M), f32), e(((M + 127) // 128, K), f32)
            L["sw"] = e(((N + 127) // 128, (K + 127) // 128), f32)
            L["sg"], L["sgt"] = e(((N + 127) // 128, M), f32), e(((M + 127) // 128, N), f32)
            # row-wise recipe: one scale per row of each K-major operand
            L["rx"], L["rxt"] = e((M,), f32), e((K,), f32)
            L["rw"], L["rwt"] = e((N,), f32), e((K,), f32)
            L["rg"], L["rgt"] = e((M,), f32), e((N,), f32)
            # per-tensor recipe scalars
            for nm in ("ax", "aw", "ag", "tx", "tw", "tg"):
                L[nm] = e((1,), f32)
            # MXFP8 recipe: E8M0 scale atoms of each operand, both orientations
            nb = fq.mx_scale_bytes
            L["mxx"], L["mxxt"] = e((nb(M, K),), u8), e((nb(K, M),), u8)
            L["mxw"], L["mxwt"] = e((nb(N, K),), u8), e((nb(K, N),), u8)
            L["mxg"], L["mxgt"] = e((nb(M, N),), u8), e((nb(N, M),), u8)
            # outputs
            L["y"], L["dx"], L["dw"] = e((M, N), bf16), e((M, K), bf16), e((N, K), bf16)
            if with_host:
                L["y_h"] = torch.empty((M, N), dtype=bf16).pin_memory()
                L["dx_h"] = torch.empty((M, K), dtype=bf16).pin_memory()
                L["dw_h"] = torch.empty((N, K), dtype=bf16).pin_memory()
                self.d2h_bytes += 2 * (M * N + M * K + N * K)
                L["ws_h"] = e((fq.linear_train_host_workspace_size(
                    fq.RECIPE_TENSOR_CURRENT, bf16, bf16, M, N, K),), u8)
            self.linears.append(L)
        self.hist_g = []
        for i, L in enumerate(self.linears):
            draws = workloads.history_draws((L["M"], L["N"]))
            amax = [fq.fp8_amax(d.to(dev)).item() for d in draws]
            self.hist_g.append(fq.History(initial=amax))
        self.operands = None

    # --- operand structs (built once: pointers are stable)
    def block_operands(self):
        fq = self.fq
        T, B, BT = fq.GemmOperand.tile, fq.GemmOperand.block, fq.GemmOperand.block_transposed
        ops = []
        for L in self.linears:
            ops.append({
                "fprop": (T(L["qx"], fq.E4M3, L["sx"]), B(L["qw"], fq.E4M3, L["sw"]), L["y"]),
                "dgrad": (T(L["qg"], fq.E5M2, L["sg"]), BT(L["qwt"], fq.E4M3, L["sw"]), L["dx"]),
                "wgrad": (T(L["qgt"], fq.E5M2, L["sgt"]), T(L["qxt"], fq.E4M3, L["sxt"]),
                          L["dw"]),
            })
        return ops

    def tensor_operands(self):
        fq = self.fq
        T = fq.GemmOperand.tensor
        ops = []
        for L in self.linears:
            ops.append({
                "fprop": (T(L["qx"], fq.E4M3, L["tx"]), T(L["qw"], fq.E4M3, L["tw"]), L["y"]),
                "dgrad": (T(L["qg"], fq.E5M2, L["tg"]), T(L["qwt"], fq.E4M3, L["tw"]), L["dx"]),
                "wgrad": (T(L["qgt"], fq.E5M2, L["tg"]), T(L["qxt"], fq.E4M3, L["tx"]),
                          L["dw"]),
            })
        return ops


    def mx_operands(self):
        fq = self.fq
        X = fq.GemmOperand.mx
        ops = []
        for L in self.linears:
            ops.append({
                "fprop": (X(L["qx"], fq.E4M3, L["mxx"]), X(L["qw"], fq.E4M3, L["mxw"]), L["y"]),
                "dgrad": (X(L["qg"], fq.E5M2, L["mxg"]), X(L["qwt"], fq.E4M3, L["mxwt"]),
                          L["dx"]),
                "wgrad": (X(L["qgt"], fq.E5M2, L["mxgt"]), X(L["qxt"], fq.E4M3, L["mxxt"]),
                          L["dw"]),
            })
        return ops

    def row_operands(self):
        fq = self.fq
        R = fq.GemmOperand.row
        ops = []
        for L in self.linears:
            ops.append({
                "fprop": (R(L["qx"], fq.E4M3, L["rx"]), R(L["qw"], fq.E4M3, L["rw"]), L["y"]),
                "dgrad": (R(L["qg"], fq.E5M2, L["rg"]), R(L["qwt"], fq.E4M3, L["rwt"]), L["dx"]),
                "wgrad": (R(L["qgt"], fq.E5M2, L["rgt"]), R(L["qxt"], fq.E4M3, L["rxt"]),
                          L["dw"]),
            })
        return ops


class Runner:
    """Issues the steps; optionally brackets each GEMM with CUDA events."""

    def __init__(self, state: LayerState, stream):
        self.s, self.stream = state, stream
        self.fq, self.torch = state.fq, state.torch
        self.bops = state.block_operands()
        self.tops = state.tensor_operands()
        self.rops = state.row_operands()
        self.mops = state.mx_operands()
        self.gemm_events = None   # list of (start, end, flops, (linear, role)) when recording
        self._cin, self._cout = self.torch.cuda.Stream(), self.torch.cuda.Stream()
        self._lin_streams = [self.torch.cuda.Stream() for _ in state.linears]

    def _gemm(self, role, A, B, C, linear=0):
        fq, torch = self.fq, self.torch
        rec = self.gemm_events is not None
        if rec:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
        fn = {"fprop": fq.fp8_gemm_fprop, "dgrad": fq.fp8_gemm_dgrad,
              "wgrad": fq.fp8_gemm_wgrad}[role]
        fn(A, B, out=C, stream=self.stream)
        if rec:
            e1.record(self.stream)
            M, N = C.shape
            self.gemm_events.append((e0, e1, 2.0 * M * N * A.K, (linear, role)))

    def _group(self, o, linear=0):
        """One linear's Fprop, Dgrad and Wgrad as one fp8_gemm_grouped call."""
        fq, torch = self.fq, self.torch
        rec = self.gemm_events is not None
        if rec:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
        roles = ("fprop", "dgrad", "wgrad")
        fq.fp8_gemm_grouped([o[r][:2] for r in roles], outs=[o[r][2] for r in roles],
                            stream=self.stream)
        if rec:
            e1.record(self.stream)
            fl = sum(2.0 * o[r][2].shape[0] * o[r][2].shape[1] * o[r][0].K for r in roles)
            self.gemm_events.append((e0, e1, fl, (linear, "group")))

    def gemms_grouped(self, ops):
        for i, o in enumerate(ops):
            self._group(o, i)

    # block recipe ------------------------------------------------------
    def quantize_block(self):
        fq, st = self.fq, self.stream
        for L in self.s.linears:
            fq.fp8_quantize_tile1x128(L["x"], fq.E4M3, rows=True, cols=True, q=L["qx"],
                                      q_scales=L["sx"], q_t=L["qxt"], qt_scales=L["sxt"],
                                      stream=st)
            fq.fp8_quantize_block128x128(L["w"], fq.E4M3, want_q=True, want_qt=True, q=L["qw"],
                                         q_t=L["qwt"], scales=L["sw"], stream=st)
            fq.fp8_quantize_tile1x128(L["g"], fq.E5M2, rows=True, cols=True, q=L["qg"],
                                      q_scales=L["sg"], q_t=L["qgt"], qt_scales=L["sgt"],
                                      stream=st)

    def gemms(self, ops):
        for i, o in enumerate(ops):
            for role in ("fprop", "dgrad", "wgrad"):
                A, B, C = o[role]
                self._gemm(role, A, B, C, i)

    def block_autocast(self):
        # per linear: quantise, then its three GEMMs (as autocast does)
        fq, st = self.fq, self.stream
        for i, (L, o) in enumerate(zip(self.s.linears, self.bops)):
            fq.fp8_quantize_tile1x128(L["x"], fq.E4M3, rows=True, cols=True, q=L["qx"],
                                      q_scales=L["sx"], q_t=L["qxt"], qt_scales=L["sxt"],
                                      stream=st)
            fq.fp8_quantize_block128x128(L["w"], fq.E4M3, want_q=True, want_qt=True, q=L["qw"],
                                         q_t=L["qwt"], scales=L["sw"], stream=st)
            fq.fp8_quantize_tile1x128(L["g"], fq.E5M2, rows=True, cols=True, q=L["qg"],
                                      q_scales=L["sg"], q_t=L["qgt"], qt_scales=L["sgt"],
                                      stream=st)
            for role in ("fprop", "dgrad", "wgrad"):
                self._gemm(role, *o[role], i)

    block_autocast.launches = 4 * 6

    # MXFP8 recipe ------------------------------------------------------
    def mx_autocast(self):
        # per linear: x, w and grad_out each quantised once into both
        # orientations (1x32 row blocks and 32x1 column blocks), then the
        # three block-scaled GEMMs
        fq, st = self.fq, self.stream
        for i, (L, o) in enumerate(zip(self.s.linears, self.mops)):
            for nm, fmt in (("x", fq.E4M3), ("w", fq.E4M3), ("g", fq.E5M2)):
                fq.fp8_quantize_mxfp8(L[nm], fmt, rows=True, cols=True, q=L["q" + nm],
                                      q_scales=L["mx" + nm], q_t=L["q" + nm + "t"],
                                      qt_scales=L["mx" + nm + "t"], stream=st)
            for role in ("fprop", "dgrad", "wgrad"):
                self._gemm(role, *o[role], i)

    mx_autocast.launches = 4 * 6

    def mx_prequant(self):
        self.gemms(self.mops)

    def block_prequant(self):
        self.gemms(self.bops)

    block_prequant.launches = 12

    # per-tensor recipes -------------------------------------------------
    def tensor_autocast(self, delayed=False):
        # per linear: amax of x and w, their casts, then grad_out's, then the
        # three GEMMs (measured a little faster for the whole step than casting
        # each tensor right after its own amax, although that order makes the
        # quantisation alone faster)
        fq, st = self.fq, self.stream
        for i, (L, o) in enumerate(zip(self.s.linears, self.tops)):
            fq.fp8_amax(L["x"], out=L["ax"], stream=st)
            fq.fp8_amax(L["w"], out=L["aw"], stream=st)
            fq.fp8_quantize_tensor(L["x"], fq.E4M3, L["ax"], want_q=True, want_qt=True, q=L["qx"],
                                   q_t=L["qxt"], scale=L["tx"], stream=st)
            fq.fp8_quantize_tensor(L["w"], fq.E4M3, L["aw"], want_q=True, want_qt=True, q=L["qw"],
                                   q_t=L["qwt"], scale=L["tw"], stream=st)
            if delayed:
                fq.fp8_quantize_delayed(L["g"], fq.E5M2, self.s.hist_g[i], want_q=True,
                                        want_qt=True, q=L["qg"], q_t=L["qgt"], scale=L["tg"],
                                        stream=st)
            else:
                fq.fp8_amax(L["g"], out=L["ag"], stream=st)
                fq.fp8_quantize_tensor(L["g"], fq.E5M2, L["ag"], want_q=True, want_qt=True,
                                       q=L["qg"], q_t=L["qgt"], scale=L["tg"], stream=st)
            for role in ("fprop", "dgrad", "wgrad"):
                self._gemm(role, *o[role], i)

    tensor_autocast.launches = 4 * 9   # per linear: 3 amax, 3 casts, 3 GEMMs

    def tensor_prequant(self):
        self.gemms(self.tops)

    def tensor_prequant_grouped(self):
        # each linear's three GEMMs as one fp8_gemm_grouped launch
        self.gemms_grouped(self.tops)

    # row-wise recipe ----------------------------------------------------
    def row_autocast(self):
        fq, st = self.fq, self.stream
        for i, (L, o) in enumerate(zip(self.s.linears, self.rops)):
            for nm, fmt in (("x", fq.E4M3), ("w", fq.E4M3), ("g", fq.E5M2)):
                fq.fp8_quantize_rowwise(L[nm], fmt, rows=True, cols=True, q=L["q" + nm],
                                        q_scales=L["r" + nm], q_t=L["q" + nm + "t"],
                                        qt_scales=L["r" + nm + "t"], stream=st)
            for role in ("fprop", "dgrad", "wgrad"):
                self._gemm(role, *o[role], i)

    row_autocast.launches = 4 * 15   # per linear: 3 x (2 quantize passes + 2 finalizes), 3 GEMMs

    def row_prequant(self):
        self.gemms(self.rops)

    # end to end: host inputs in, host outputs out --------------------------
    def e2e_host(self):
        """One step through the C-ABI's host-buffer entry point: for each
        linear one fp8_linear_train_host call (per-tensor current scaling)
        from its pinned x, w and grad_out to its pinned y, dx and dw.  The
        library copies in and out on its own two streams; each call is issued
        on a stream of its own (all forked from the step's start on the
        compute stream and joined at its end), with a workspace of its own,
        so a linear's copies in queue right behind the previous linear's
        instead of waiting for its GEMMs."""
        torch, fq, st = self.torch, self.fq, self.stream
        start = torch.cuda.Event()
        start.record(st)
        for L, s in zip(self.s.linears, self._lin_streams):
            s.wait_event(start)
            fq.fp8_linear_train_host(L["x_h"], L["w_h"], L["g_h"], L["y_h"], L["dx_h"],
                                     L["dw_h"], L["ws_h"], recipe=fq.RECIPE_TENSOR_CURRENT,
                                     stream=s)
        for s in self._lin_streams:
            st.wait_stream(s)

    def link_rates(self, reps: int = 3):
        """Host<->device copy rates over this step's own pinned buffers: the
        inputs in alone, the outputs out alone, and both at once (GB/s, median
        of `reps`, wall clock between device synchronisations).  The
        both-at-once time is the floor of an end-to-end step."""
        torch = self.torch
        ins = [(L[k], L[k + "_h"]) for L in self.s.linears for k in "xwg"]
        outs = [(L[o + "_h"], L[o]) for L in self.s.linears for o in ("y", "dx", "dw")]

        def issue(pairs, stream):
            with torch.cuda.stream(stream):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)

        def timed(fn):
            ts = []
            for _ in range(reps):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
            return statistics.median(ts)

        t_in = timed(lambda: issue(ins, self._cin))
        t_out = timed(lambda: issue(outs, self._cout))
        t_both = timed(lambda: (issue(ins, self._cin), issue(outs, self._cout)))
        hb, db = self.s.h2d_bytes, self.s.d2h_bytes
        return {"h2d_gbs": hb / t_in / 1e9, "d2h_gbs": db / t_out / 1e9,
                "both_gbs": (hb + db) / t_both / 1e9, "floor_ms": t_both * 1e3}


def time_steps(torch, dist, stream, fn, steps, warmup, flush=None, record=None, clk=None):
    """W untimed steps, then exactly K timed steps between barriers and
    device synchronisations; returns the max-over-ranks ms per step."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t_start = time.time()
    if flush is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if record is not None:
            record.gemm_events = []
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
    else:
        # L2 flushed before each step, outside the event pair
        ms = 0.0
        for _ in range(steps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
    if clk is not None:
        clk.windows.append((t_start, time.time()))
    dist.barrier()
    torch.cuda.synchronize()
    return dist.max(ms / steps)


# ------------------------------------------------------------- CPU baseline

class OracleLayerSample:
    """The oracle on a bounded sample of the headline step (per-tensor current
    scaling, E4M3 x and w, E5M2 grad_out): every run() takes, for each of the
    four linears, the amax of ALL of x, w and grad_out (the recipe's scale
    needs the whole tensor; the oracle's amax runs over row chunks on the
    host threads, and a max is exact in any order), their scales, then for
    each of the 12 GEMMs casts `rows` rows of A and one 128-row block of B with
    those scales and forms that rows x 128 block of the output in double.
    ctypes releases the GIL, so the plain-C oracle runs on `threads` host
    threads.  run() returns (GEMM flops of the sample, seconds)."""

    ROWS = 64     # one sample size for the reference arm and cpu_baseline
    BROWS = 64

    def __init__(self, threads: int, rows: int = ROWS, brows: int = BROWS):
        import numpy as np
        import torch

        import workloads

        def bits(t):
            return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))

        self.rows, self.brows, self.threads = rows, brows, threads
        self.linears = []
        for i, shape in enumerate(workloads.LAYER):
            x, w, g = workloads.layer_inputs(shape, i)
            xb, wb, gb = bits(x), bits(w), bits(g)
            self.linears.append({
                "full": (xb, wb, gb),
                # (A rows, A format, A scale source, B rows, B format, B scale source)
                "jobs": [
                    (xb[:rows], 0, 0, wb[:brows], 0, 1),                             # fprop
                    (gb[:rows], 1, 2, np.ascontiguousarray(wb[:, :brows].T), 0, 1),   # dgrad
                    (np.ascontiguousarray(gb[:, :rows].T), 1, 2,
                     np.ascontiguousarray(xb[:, :brows].T), 0, 0),                  # wgrad
                ]})

    def description(self) -> str:
        return (f"per-tensor current scaling of the 15872-token layer: amax of all of x, w and "
                f"grad_out of the four linears, then for each of the 12 GEMMs the cast of "
                f"{self.rows} rows of A and {self.brows} rows of B and their {self.rows} x "
                f"{self.brows} output block in double, per step")

    def run(self):
        import concurrent.futures as cf

        import numpy as np

        import oracle

        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=self.threads) as pool:
            def amax_all(arr):
                step = max(1, arr.shape[0] // self.threads)
                parts = [arr[r:r + step] for r in range(0, arr.shape[0], step)]
                return max(pool.map(lambda a: float(oracle.amax(a)), parts))

            flops = 0.0
            for L in self.linears:
                xb, wb, gb = L["full"]
                amx = [amax_all(xb), amax_all(wb), amax_all(gb)]
                fmts = [0, 0, 1]
                sc = [oracle.scale_from_amax(a, f) for a, f in zip(amx, fmts)]
                for a, fa, ia, b, fb, ib in L["jobs"]:
                    qa, _, _ = oracle.quantize_tensor(a, fa, sc[ia])
                    qb, _, _ = oracle.quantize_tensor(b, fb, sc[ib])
                    A = oracle.GemmOperand.tensor(qa, fa, sc[ia])
                    B = oracle.GemmOperand.tensor(qb, fb, sc[ib])
                    step = max(1, a.shape[0] // self.threads)
                    parts = [(m0, min(a.shape[0], m0 + step)) for m0 in range(0, a.shape[0], step)]
                    list(pool.map(lambda pr: oracle.gemm_rows(A, B, pr[0], pr[1]), parts))
                    flops += 2.0 * a.shape[0] * b.shape[0] * a.shape[1]
        return flops, time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference

def run_reference(args, dist):
    """The oracle as the reference arm: each step is the bounded sample of
    the headline step above, timed on the host cores."""
    if dist.rank != 0:
        return
    import oracle
    oracle.build()
    threads = cpu_cores()
    sample_run = OracleLayerSample(threads)
    for _ in range(args.warmup):
        sample_run.run()
    flops = secs = 0.0
    for _ in range(args.steps):
        f, s = sample_run.run()
        flops += f
        secs += s
    tflops = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8->f64", "data": "synthetic",
        "config": layer_config(),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample_run.description()},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def layer_config():
    import workloads
    return {
        "workload": ("transformer layer, 12 FP8 GEMMs (fprop/dgrad/wgrad x qkv/attn_out/mlp_up/"
                     "mlp_down), per-tensor current scaling (amax -> scale -> cast of x, w and "
                     "grad_out each step), E4M3 forward / E5M2 gradients, autocast (quantize "
                     "included)"),
        "M": workloads.TOKENS, "hidden": workloads.HIDDEN, "ffn": workloads.FFN,
        "inputs": "bf16 x~N(0,1), w~N(0,0.02), grad_out~N(0,1e-3) + 40.0 spikes per 1e6",
        "out_dtype": "bf16",
        "l2": "inputs larger than L2 (each step streams ~5 GB of operands)",
    }


def tiny_linear_latency(fq, torch, stream, reps: int = 200):
    """The fp8_parity page's linear (x 512x32, w 64x32, grad_out 512x64, fp32,
    per-tensor current scaling, fp32 outputs): microseconds per call of each
    GEMM (operands quantised beforehand) and of the whole autocast forward +
    backward (amax and cast with the transposed copy of x, w and grad_out,
    then the three GEMMs), as `reps` back-to-back calls on one stream timed
    with CUDA events, and as a replayed CUDA graph of the same calls.  At
    2 MFLOP per GEMM this is launch latency, not a roofline."""
    import workloads
    x, w, g = (t.cuda() for t in workloads.tiny_linear())
    f32 = torch.float32
    e = lambda shp, dt: torch.empty(shp, dtype=dt, device=x.device)
    q = {k: (e(t.shape, torch.uint8), e(t.shape[::-1], torch.uint8), e((1,), f32), e((1,), f32))
         for k, t in (("x", x), ("w", w), ("g", g))}
    src = {"x": x, "w": w, "g": g}
    fmt = {"x": fq.E4M3, "w": fq.E4M3, "g": fq.E5M2}
    y, dx, dw = e((512, 64), f32), e((512, 32), f32), e((64, 32), f32)

    def quantize():
        # amax, then the cast (two launches per tensor: at these sizes the
        # one-call form, a memset and a cooperative launch, is no faster
        # eagerly and slower inside a graph)
        for k in "xwg":
            qq, qt, am, sc = q[k]
            fq.fp8_amax(src[k], out=am, stream=stream)
            fq.fp8_quantize_tensor(src[k], fmt[k], am, want_q=True, want_qt=True, q=qq, q_t=qt,
                                   scale=sc, stream=stream)

    T = fq.GemmOperand.tensor
    gemm = {
        "fprop_512x64x32": lambda: fq.fp8_gemm_fprop(T(q["x"][0], 0, q["x"][3]),
                                                     T(q["w"][0], 0, q["w"][3]), out=y,
                                                     stream=stream),
        "dgrad_512x32x64": lambda: fq.fp8_gemm_dgrad(T(q["g"][0], 1, q["g"][3]),
                                                     T(q["w"][1], 0, q["w"][3]), out=dx,
                                                     stream=stream),
        "wgrad_64x32x512": lambda: fq.fp8_gemm_wgrad(T(q["g"][1], 1, q["g"][3]),
                                                     T(q["x"][1], 0, q["x"][3]), out=dw,
                                                     stream=stream),
    }

    def per_call_us(fn):
        for _ in range(20):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    def step():
        quantize()
        for fn in gemm.values():
            fn()

    quantize()
    out = {k: round(per_call_us(fn), 2) for k, fn in gemm.items()}
    out["quantize_x_w_g_us"] = round(per_call_us(quantize), 2)
    out["autocast_fwd_bwd_us"] = round(per_call_us(step), 2)
    # the same nine launches captured once into a CUDA graph and replayed
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        out["autocast_fwd_bwd_graph_us"] = round(per_call_us(graph.replay), 2)
    out["note"] = ("us per call, back-to-back on one stream (CUDA events over "
                   f"{reps} calls); the autocast step is 3 amax + 3 casts + 3 GEMMs = 9 launches, "
                   "issued call by call or replayed as one CUDA graph")
    return out


# --------------------------------------------------------------------- main

def main():
    args = parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
        dist.close()
        return

    import torch
    import scaled_quantize_fp8_warp_gb300 as fq
    from scaled_quantize_fp8_warp_gb300 import build_lib
    import workloads

    if dist.rank == 0:
        build_lib.build()
    dist.barrier()
    fq.load_library()
    torch.cuda.set_device(dist.local)
    if not fq.device_supported():
        raise SystemExit("bench: the current device is not compute capability 10.3 (GB300)")
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dist.local).uuid)
    except Exception:
        pass

    state = LayerState(fq, torch, with_host=True)
    run = Runner(state, stream)
    K, W = args.steps, args.warmup
    # One untimed pass of the host-buffer step right after the pinned buffers
    # are allocated: when the first host<->device round trip came only after
    # the device-resident phases, the timed step ran 29-40 ms instead of
    # ~20 ms, on the same box and build.
    run.e2e_host()
    torch.cuda.synchronize()
    flops = state.flops
    # ---- end to end through host buffers (headline recipe), with the host
    # link's own rates over the same buffers just before, since they bound it
    link = run.link_rates()
    ms_e2e = time_steps(torch, dist, stream, run.e2e_host, max(2, K // 2), W)

    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fp8_peak_sust = FP8_PER_BF16 * float(peaks.get("bf16_tflops_sustained",
                                                   FALLBACK_PEAKS["bf16_tflops_sustained"]))
    fp8_peak_burst = FP8_PER_BF16 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    def gemm_summary(events):
        ms = sum(a.elapsed_time(b) for a, b, _, _ in events)
        fl = sum(f for _, _, f, _ in events)
        return ms, fl, len(events)

    def gemm_table(events):
        """Per GEMM of the layer (linear.role): mean event-timed duration over
        the timed steps, its TFLOP/s and fraction of the burst FP8 peak."""
        agg = {}
        for a, b, fl, key in events:
            t = agg.setdefault(key, [0.0, 0, fl])
            t[0] += a.elapsed_time(b)
            t[1] += 1
        rows = {}
        for (i, role), (ms, n, fl) in sorted(agg.items()):
            us = ms / n * 1e3
            tfl = fl / (us * 1e-6) / 1e12
            nm = workloads.LAYER[i].name
            if role == "group":
                shp = ", ".join(f"{m}x{nn}x{k}" for lname, r, m, nn, k in workloads.gemm_problems()
                                if lname == nm)
                key, label = f"{nm}.fprop+dgrad+wgrad", shp
            else:
                M, N, Kc = [(m, nn, k) for lname, r, m, nn, k in workloads.gemm_problems()
                            if lname == nm and r == role][0]
                key, label = f"{nm}.{role}", f"{M}x{N}x{Kc}"
            rows[key] = {"MxNxK": label, "us": round(us, 2), "TFLOP/s": round(tfl, 1),
                         "frac": round(tfl / fp8_peak_burst, 3)}
        return rows

    per_gemm = {}

    def timed(name, fn, record=True):
        """The phase's ms per step, timed with no event inside the steps (an
        event pair around a launch adds several microseconds to the step);
        then the same K steps again with an event pair around every GEMM,
        whose per-GEMM table goes to per_gemm[name]."""
        ms = time_steps(torch, dist, stream, fn, K, W, clk=clk)
        out = None
        if record:
            time_steps(torch, dist, stream, fn, K, 1, record=run, clk=clk)
            if run.gemm_events:
                per_gemm[name] = gemm_table(run.gemm_events)
                out = gemm_summary(run.gemm_events)
        run.gemm_events = None
        return ms, out

    # ---- headline: the layer with per-tensor current scaling, autocast;
    # clocks are sampled through every timed layer phase
    with ClockSampler(uuid) as clk:
        ms_auto, (t_gemm_ms, t_gemm_fl, t_gemm_n) = timed(
            "tensor_current.autocast", lambda: run.tensor_autocast(False))
        head_windows = list(clk.windows)
        ms_pre, _ = timed("tensor_current.prequant", run.tensor_prequant)
        # the same 12 GEMMs as four grouped launches (one per linear)
        ms_pre_grp, _ = timed("tensor_current.prequant_grouped_launches",
                              run.tensor_prequant_grouped)
        ms_d_auto, _ = timed("tensor_delayed_grad.autocast", lambda: run.tensor_autocast(True))

        # ---- the same layer with 1x128 / 128x128 scaling
        ms_b_auto, _ = timed("block_1x128_128x128.autocast", run.block_autocast)
        ms_b_pre, (b_gemm_ms, b_gemm_fl, b_gemm_n) = timed("block_1x128_128x128.prequant",
                                                           run.block_prequant)

        # ---- the same layer with MXFP8 (1x32 blocks, E8M0 scales)
        ms_m_auto, _ = timed("mxfp8.autocast", run.mx_autocast)
        ms_m_pre, (m_gemm_ms, m_gemm_fl, m_gemm_n) = timed("mxfp8.prequant", run.mx_prequant)

        # ---- the same layer with row-wise scaling
        ms_r_auto, _ = timed("rowwise.autocast", run.row_autocast)
        ms_r_pre, (r_gemm_ms, r_gemm_fl, r_gemm_n) = timed("rowwise.prequant", run.row_prequant)

        # ---- amax fused into the GEMM that produces the next quantize's input:
        # QKV Fprop alone, followed by a separate amax of y, and with the fused amax
        L0, o0 = state.linears[0], run.tops[0]
        xA, wB, y0 = o0["fprop"]
        am_y = torch.empty(1, dtype=torch.float32, device=y0.device)
        ms_f_gemm = time_steps(torch, dist, stream, lambda: fq.fp8_gemm(
            xA, wB, out=y0, stream=stream), K, W, clk=clk)
        ms_f_sep = time_steps(torch, dist, stream, lambda: (
            fq.fp8_gemm(xA, wB, out=y0, stream=stream),
            fq.fp8_amax(y0, out=am_y, stream=stream)), K, W, clk=clk)
        ms_f_fused = time_steps(torch, dist, stream, lambda: fq.fp8_gemm_amax(
            xA, wB, out=y0, amax=am_y, stream=stream), K, W, clk=clk)

    # ---- the headline's own clock record; a slowdown during it (or a clock
    # lock) voids the number, and the phase is measured once more
    head_span = "the timed regions of the headline phase (per-tensor autocast)"
    clk_all = clk
    clk_head = clk.summary(windows=head_windows, span=head_span)
    remeasured = None
    causes = clock_rejection(clk_head)
    if causes:
        first = {"ms_per_step": ms_auto, "causes": causes, "clocks": clk_head}
        with ClockSampler(uuid) as clk:
            ms_auto, (t_gemm_ms, t_gemm_fl, t_gemm_n) = timed(
                "tensor_current.autocast", lambda: run.tensor_autocast(False))
        clk_head = clk.summary(span=head_span)
        remeasured = {"first": first, "second_causes": clock_rejection(clk_head)}

    # ---- the same end-to-end step again after the device-resident phases:
    # on several boxes the device->host rate over these buffers had dropped by
    # then (21-39 GB/s against 192), so both measurements are reported
    link_late = run.link_rates()
    ms_e2e_late = time_steps(torch, dist, stream, run.e2e_host, max(2, K // 2), W)

    # ---- quantize bandwidth on the 8192x4096 activation (L2 flushed)
    xq, out_rows = workloads.quantize_activation()
    xq = xq.cuda()
    R, C = xq.shape
    n = R * C
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=xq.device)
    flush_sink = torch.empty(1, dtype=torch.float32, device=xq.device)

    def flush():
        # write a buffer twice the size of L2, then read it back so the lines
        # left in L2 are clean (no write-backs charged to the timed kernel);
        # on the timed stream, so it completes before the start event
        # (no host sync here: while the GPU runs the ~100 us flush, the host
        # queues the start event and the timed call, so the events do not
        # time host launch latency)
        with torch.cuda.stream(stream):
            flush_buf.fill_(1.0)
            flush_sink.copy_(flush_buf.sum())
            torch.cuda._sleep(400_000)   # ~0.2 ms more queue ahead of the start event

    qt = torch.empty((R, C), dtype=torch.uint8, device=xq.device)
    st = torch.empty(((C + 127) // 128, R), dtype=torch.float32, device=xq.device)
    am = torch.empty(1, dtype=torch.float32, device=xq.device)
    sc = torch.empty(1, dtype=torch.float32, device=xq.device)
    QK = max(K, 10)
    ms_tile = time_steps(torch, dist, stream, lambda: fq.fp8_quantize_tile1x128(
        xq, fq.E4M3, rows=True, q=qt, q_scales=st, stream=stream), QK, W, flush=flush)
    ms_amax = time_steps(torch, dist, stream, lambda: fq.fp8_amax(xq, out=am, stream=stream),
                         QK, W, flush=flush)
    ms_tensor = time_steps(torch, dist, stream, lambda: fq.fp8_quantize_tensor_current(
        xq, fq.E4M3, q=qt, amax=am, scale=sc, stream=stream), QK, W, flush=flush)
    ms_tensor_2k = time_steps(torch, dist, stream, lambda: (
        fq.fp8_amax(xq, out=am, stream=stream),
        fq.fp8_quantize_tensor(xq, fq.E4M3, am, q=qt, scale=sc, stream=stream)), QK, W,
        flush=flush)
    tile_bytes = n * 2 + n * 1 + 4 * n // 128
    # both orientations (q and the transposed copy q_t), as the layer uses them
    qtt = torch.empty((C, R), dtype=torch.uint8, device=xq.device)
    stt = torch.empty(((R + 127) // 128, C), dtype=torch.float32, device=xq.device)
    rs_r = torch.empty((R,), dtype=torch.float32, device=xq.device)
    rs_c = torch.empty((C,), dtype=torch.float32, device=xq.device)
    ms_tile2 = time_steps(torch, dist, stream, lambda: fq.fp8_quantize_tile1x128(
        xq, fq.E4M3, rows=True, cols=True, q=qt, q_scales=st, q_t=qtt, qt_scales=stt,
        stream=stream), QK, W, flush=flush)
    ms_row2 = time_steps(torch, dist, stream, lambda: fq.fp8_quantize_rowwise(
        xq, fq.E4M3, rows=True, cols=True, q=qt, q_scales=rs_r, q_t=qtt, qt_scales=rs_c,
        stream=stream), QK, W, flush=flush)
    ms_tensor2 = time_steps(torch, dist, stream, lambda: fq.fp8_quantize_tensor_current(
        xq, fq.E4M3, want_q=True, want_qt=True, q=qt, q_t=qtt, amax=am, scale=sc,
        stream=stream), QK, W, flush=flush)
    dual_bytes = n * 2 + 2 * n     # read x once, write q and q_t (scales are < 0.1%)

    # ---- the same calls back to back on the stream, as a training step
    # issues them: NROT distinct copies of the activation (each with its own
    # outputs; 4 x 64 MiB, more than L2, so every call reads its input from
    # DRAM), K rounds timed with one event pair, time per call.  A single
    # call, as timed above, also pays the launch floor (an empty kernel
    # measures about 3.6 us between two events); here that overlaps the
    # previous kernel.
    NROT = 4
    xs = [xq] + [xq.clone() for _ in range(NROT - 1)]
    rot = [{"q": torch.empty_like(qt), "s": torch.empty_like(st), "qt": torch.empty_like(qtt),
            "st": torch.empty_like(stt), "a": torch.empty_like(am), "c": torch.empty_like(sc)}
           for _ in range(NROT)]

    def streamed(call):
        def step():
            for j in range(NROT):
                call(xs[j], rot[j])
        return time_steps(torch, dist, stream, step, QK, W) / NROT

    sms_tile = streamed(lambda xj, o: fq.fp8_quantize_tile1x128(
        xj, fq.E4M3, rows=True, q=o["q"], q_scales=o["s"], stream=stream))
    sms_amax = streamed(lambda xj, o: fq.fp8_amax(xj, out=o["a"], stream=stream))
    sms_tensor = streamed(lambda xj, o: fq.fp8_quantize_tensor_current(
        xj, fq.E4M3, q=o["q"], amax=o["a"], scale=o["c"], stream=stream))
    sms_tile2 = streamed(lambda xj, o: fq.fp8_quantize_tile1x128(
        xj, fq.E4M3, rows=True, cols=True, q=o["q"], q_scales=o["s"], q_t=o["qt"],
        qt_scales=o["st"], stream=stream))
    del xs, rot

    # ---- accuracy on the same activation: MSE of the dequantised values on
    # the rows without outliers, 1x128 tiles against one scale per tensor
    # (analysis of the kernels' outputs, outside every timed region)
    keep = torch.ones(R, dtype=torch.bool, device=xq.device)
    keep[out_rows.to(xq.device)] = False
    xf = xq.float()
    fq.fp8_quantize_tile1x128(xq, fq.E4M3, rows=True, q=qt, q_scales=st, stream=stream)
    fq.fp8_amax(xq, out=am, stream=stream)
    qtt2 = torch.empty_like(qt)
    fq.fp8_quantize_tensor(xq, fq.E4M3, am, q=qtt2, scale=sc, stream=stream)
    torch.cuda.synchronize()
    deq_tile = (qt.view(torch.float8_e4m3fn).float().view(R, C // 128, 128)
                * st.t().reshape(R, C // 128, 1)).view(R, C)
    deq_tensor = qtt2.view(torch.float8_e4m3fn).float() * sc
    mse_tile = ((deq_tile - xf)[keep] ** 2).mean().item()
    mse_tensor = ((deq_tensor - xf)[keep] ** 2).mean().item()
    del xf, deq_tile, deq_tensor, qtt2
    gbps = lambda b, ms: b / (ms * 1e-3) / 1e9

    # ---- CPU baseline (oracle on the host cores, rank 0, N = 1 only)
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = cpu_cores()
        sample_run = OracleLayerSample(threads)
        f = s = 0.0
        reps = 0
        while s < 10.0 and reps < 20:     # about ten seconds of host work
            df, ds = sample_run.run()
            f, s, reps = f + df, s + ds, reps + 1
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": (f"{sample_run.description()}; {reps} steps, {f / 1e9:.2f} GFLOP "
                          f"in {s:.1f} s")}

    t_gemm_tflops = t_gemm_fl / (t_gemm_ms * 1e-3) / 1e12
    b_gemm_tflops = b_gemm_fl / (b_gemm_ms * 1e-3) / 1e12
    m_gemm_tflops = m_gemm_fl / (m_gemm_ms * 1e-3) / 1e12
    r_gemm_tflops = r_gemm_fl / (r_gemm_ms * 1e-3) / 1e12
    tile_gbps = gbps(tile_bytes, ms_tile)
    tf = lambda ms: flops / (ms * 1e-3) / 1e12
    peak_src = (f"{peak_src}: bf16_tflops (burst: the layer step is {ms_auto:.1f} ms, not a "
                f"seconds-long loop) x {FP8_PER_BF16} (dense FP8/BF16 nominal ratio)")
    tiny = tiny_linear_latency(fq, torch, stream)

    line = {
        "metric": METRIC,
        "value": tf(ms_auto),
        "unit": "TFLOP/s",
        "n_gpus": dist.world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_auto,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8->f32",
        "data": "synthetic",
        "config": layer_config(),
        "prequant": {"value": tf(ms_pre), "unit": "TFLOP/s", "ms_per_step": ms_pre,
                     "grouped_launches_ms_per_step": ms_pre_grp},
        "quantize_ms_per_step": ms_auto - t_gemm_ms / K,
        "delayed_grad": {
            "autocast": {"value": tf(ms_d_auto), "ms_per_step": ms_d_auto}, "unit": "TFLOP/s",
            "note": "grad_out cast with its amax history (delayed scaling), x and w current"},
        "block_scaled": {
            "workload": ("the same 12 GEMMs with 1x128 tiles on activations and gradients and "
                         "128x128 blocks on weights"),
            "autocast": {"value": tf(ms_b_auto), "ms_per_step": ms_b_auto},
            "prequant": {"value": tf(ms_b_pre), "ms_per_step": ms_b_pre},
            "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": b_gemm_tflops, "peak": fp8_peak_burst,
                         "unit": "TFLOP/s", "frac": b_gemm_tflops / fp8_peak_burst,
                         "traffic": recorded_traffic("gemm_blockscaled_kernel"),
                         "kernel": "gemm_blockscaled_kernel (prequant step)",
                         "launches": b_gemm_n}},
        "mxfp8": {
            "workload": ("the same 12 GEMMs with MXFP8 (OCP MX v1.0: 1x32 blocks, E8M0 scales) "
                         "on x, w and grad_out, each quantised into both orientations"),
            "autocast": {"value": tf(ms_m_auto), "ms_per_step": ms_m_auto},
            "prequant": {"value": tf(ms_m_pre), "ms_per_step": ms_m_pre},
            "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": m_gemm_tflops, "peak": fp8_peak_burst,
                         "unit": "TFLOP/s", "frac": m_gemm_tflops / fp8_peak_burst,
                         "traffic": recorded_traffic("gemm_mx_kernel"),
                         "kernel": ("gemm_mx_kernel, tcgen05.mma kind::mxf8f6f4 block_scale "
                                    "(prequant step)"),
                         "launches": m_gemm_n}},
        "rowwise": {
            "workload": ("the same 12 GEMMs with one scale per row of each K-major operand "
                         "(x, w and grad_out quantised along both orientations)"),
            "autocast": {"value": tf(ms_r_auto), "ms_per_step": ms_r_auto},
            "prequant": {"value": tf(ms_r_pre), "ms_per_step": ms_r_pre},
            "unit": "TFLOP/s",
            "gemm": {"achieved": r_gemm_tflops, "frac": r_gemm_tflops / fp8_peak_burst,
                     "kernel": "gemm_tensor_pair_kernel (cta_group::2), row-scale epilogue",
                     "launches": r_gemm_n}},
        "fused_amax": {
            "workload": ("QKV Fprop 15872x12288x4096, per-tensor E4M3, bf16 y (390 MB): "
                         "amax(y) for the next per-tensor quantize"),
            "gemm_ms": ms_f_gemm, "gemm_then_amax_ms": ms_f_sep,
            "gemm_with_fused_amax_ms": ms_f_fused,
            "saved_ms": ms_f_sep - ms_f_fused},
        "context_pages_B300_ms_per_layer": {
            "fp8_current_autocast": 9.15, "fp8_current_prequant": 6.81,
            "fp8_delayed_autocast": 7.80, "mxfp8_autocast": 8.98,
            "fp8_delayed_prequant_reported": 8.12,
            "note": ("the blog repost's CodonFM-5B layer on B300 with Transformer Engine; "
                     "context, not the target")},
        "quantize": {
            "workload": "8192x4096 bf16 activation (1% rows x 1e4), E4M3, L2 flushed per call",
            "tile1x128": {"GB/s": tile_gbps, "us": ms_tile * 1e3,
                          "bytes": tile_bytes, "frac": tile_gbps / hbm_peak},
            "amax": {"GB/s": gbps(2 * n, ms_amax), "us": ms_amax * 1e3,
                     "frac": gbps(2 * n, ms_amax) / hbm_peak},
            "streamed": {
                "note": ("per call, 4 distinct 64 MiB activations back to back on the "
                         "stream (each read from DRAM), K rounds under one event pair; the "
                         "single-call figures above also include the ~3.6 us launch floor "
                         "between two events"),
                "tile1x128": {"us": sms_tile * 1e3, "GB/s": gbps(tile_bytes, sms_tile),
                              "frac": gbps(tile_bytes, sms_tile) / hbm_peak},
                "amax": {"us": sms_amax * 1e3, "GB/s": gbps(2 * n, sms_amax),
                         "frac": gbps(2 * n, sms_amax) / hbm_peak},
                "tensor_current_over_3B": {"us": sms_tensor * 1e3,
                                           "GB/s": gbps(3 * n, sms_tensor),
                                           "frac": gbps(3 * n, sms_tensor) / hbm_peak},
                "tile1x128_rows_and_cols": {"us": sms_tile2 * 1e3,
                                            "GB/s": gbps(dual_bytes, sms_tile2),
                                            "frac": gbps(dual_bytes, sms_tile2) / hbm_peak}},
            "tensor_current": {"GB/s (over 3 B/elem)": gbps(3 * n, ms_tensor),
                               "us": ms_tensor * 1e3,
                               "frac": gbps(3 * n, ms_tensor) / hbm_peak,
                               "how": ("fp8_quantize_tensor_current: at this size the amax and "
                                       "cast kernels (one cooperative launch only up to 8 MiB, "
                                       "where it is the faster)"),
                               "two_kernels_us": ms_tensor_2k * 1e3},
            "both_orientations": {
                "note": ("q and q_t from one call; GB/s over the unique bytes (2 B read + "
                         "2 B written per element); row-wise and per-tensor read x twice "
                         "(amax pass, then cast), the second read mostly from L2"),
                "tile1x128_rows_and_cols": {"GB/s": gbps(dual_bytes, ms_tile2),
                                            "us": ms_tile2 * 1e3,
                                            "frac": gbps(dual_bytes, ms_tile2) / hbm_peak},
                "rowwise": {"GB/s": gbps(dual_bytes, ms_row2), "us": ms_row2 * 1e3,
                            "frac": gbps(dual_bytes, ms_row2) / hbm_peak},
                "tensor_current": {"GB/s": gbps(dual_bytes, ms_tensor2), "us": ms_tensor2 * 1e3,
                                   "frac": gbps(dual_bytes, ms_tensor2) / hbm_peak}},
            "accuracy": {"mse_rows_without_outliers": {"tile1x128": mse_tile,
                                                       "tensor": mse_tensor},
                         "rows": int(keep.sum().item()),
                         "note": "dequantised E4M3 vs the bf16 input; 1x128 tiles should be lower"},
            "unit": "GB/s", "peak": hbm_peak,
        },
        "roofline": {"bound": "tensor", "achieved": t_gemm_tflops, "peak": fp8_peak_burst,
                     "unit": "TFLOP/s", "frac": t_gemm_tflops / fp8_peak_burst,
                     "traffic": recorded_traffic("gemm_tensor_pair_kernel"),
                     "kernel": "gemm_tensor_pair_kernel, cta_group::2 (12 GEMMs of the autocast step)",
                     "launches": t_gemm_n, "peak_source": peak_src,
                     "frac_of_sustained": t_gemm_tflops / fp8_peak_sust},
        "per_gemm": dict(per_gemm, unit=("us per launch (CUDA events around each GEMM, in a "
                                           "repeat of the phase's timed steps)"),
                         peak_tflops=fp8_peak_burst),
        "tiny_linear": tiny,
        "roofline_quantize": {"bound": "hbm", "achieved": tile_gbps, "peak": hbm_peak,
                              "unit": "GB/s", "frac": tile_gbps / hbm_peak,
                              "traffic": recorded_traffic("quant2d_tile_rows"),
                              "kernel": "quant2d_kernel (1x128 row tiles)",
                              "peak_source": "measured: hbm_gbs"},
        "cpu_baseline": cpu,
        "e2e": {"value": tf(ms_e2e), "unit": "TFLOP/s",
                "ms_per_step": ms_e2e, "h2d_bytes_per_step": state.h2d_bytes,
                "d2h_bytes_per_step": state.d2h_bytes, "host_link": link,
                "measured": "first, right after the buffers are set up",
                "after_layer_phases": {"value": tf(ms_e2e_late), "ms_per_step": ms_e2e_late,
                                       "host_link": link_late},
                "how": ("4 fp8_linear_train_host C-ABI calls per step (per-tensor current "
                        "scaling), pinned host x, w, grad_out in and y, dx, dw out")},
        "gpu_launches": Runner.tensor_autocast.launches * K,
        "clocks": clk_head,
        "clocks_all_layer_phases": clk_all.summary(),
    }
    if remeasured is not None:
        line["remeasured"] = remeasured
    if fq.device_status() != 0:
        line["error"] = "a kernel reported a barrier timeout"
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
