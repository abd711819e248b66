"""Benchmark of one MoE layer step (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dsv3_fp8]
                    [--impl ours|reference]

A step is one pass of the whole layer over one batch of synthetic tokens:
route, permute, grouped SwiGLU FFN, unpermute, and the backward of all of it
(dx, dW_r, dW13, dW2). The default workload is the largest of the five layer
shapes, the FP8 DeepSeek-V3-shaped layer (T=16384, H=7168, E=256, top-8
group-limited sigmoid routing, d_ff=2048, E4M3 operands with power-of-two
block scales, capacity factor 1.25). Prints one JSON line.

  value      tokens/s of fwd+bwd with inputs resident in HBM (CUDA events)
  e2e        the same through the public layer calls with host buffers: each
             step copies x and dY from pinned host memory and reads out and dx
             back inside the timed region
  roofline   the grouped-GEMM kernel family (the dominant kernel) against the
             measured dense tensor peak of its operand type (FP8: twice the
             measured bf16 burst figure, the nominal FP8:bf16 rate ratio)
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload

--impl reference times the CPU oracle instead (the reference arm of this
build: there is no runnable upstream implementation).
Multi-GPU: the layer is not sharded, so N GPUs run N independent replicas
(weak scaling, no collective on the data path); value sums the replicas.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dsv3_fp8",
                    choices=sorted(W.SHAPES) + sorted(W.PROFILE_SHAPES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--weights-in-expert", action="store_true",
                    help="the layer with the routing weight applied inside the expert (bf16)")
    ap.add_argument("--recompute-h", action="store_true",
                    help="the backward rewrites h from GU (fine-grained recompute): h need not "
                         "survive from the forward to the backward")
    ap.add_argument("--paged-stash", action="store_true",
                    help="the end-to-end leg keeps x_perm, GU, h and y_perm in a stash pool of "
                         "128-row pages sized to the layer's live rows (paged stashing) instead "
                         "of worst-case buffers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="reference arm: seconds of oracle work for all timed steps together")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thr = threading.Thread(target=self._read, daemon=True)
            self.thr.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# the sources of the launches in profiles/gemm_traffic.json (the GEMMs and the
# weight-gradient stage's quantisers)
GEMM_SOURCES = ("grouped_gemm.cu", "grouped_gemm_fp8.cu", "gemm_common.cuh", "ptx.cuh",
                "fp8_layout.cuh", "quant.cu")


def gemm_sources_sha256() -> str:
    """Hash of the GEMM sources' code: comments (// to the end of a line) and
    whitespace are left out, so only a change to the code itself retires a
    committed capture of the kernels' DRAM traffic."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        path = os.path.join(ROOT, "routing_dispatch_expert_router_gb300", "csrc", name)
        if os.path.exists(path):
            with open(path, encoding="utf-8") as f:
                text = f.read()
            code = re.sub(r"//[^\n]*", "", text)
            h.update(re.sub(r"\s+", "", code).encode())
    return h.hexdigest()


def gemm_traffic(workload: str, key: str = "dram_bytes_per_step"):
    """DRAM bytes per step of the grouped-GEMM launches from a committed ncu
    capture (`key`: the roofline kernel's launches, or the FP8 weight-gradient
    stage's), or None when a GEMM source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("gemm_sources_sha256") != gemm_sources_sha256() or d.get("workload") != workload:
        return None
    return d.get(key)


def gemm_flops(shape, counts) -> float:
    """Algorithmic flops of one pass of the grouped GEMMs (kept rows only): the
    forward (FC1 + FC2), the data gradients and the weight gradients each do
    this much."""
    rows = float(sum(counts))        # routed kept rows + shared rows (T each)
    return 2.0 * rows * shape.H * 2 * shape.F + 2.0 * rows * shape.F * shape.H


def stash_bytes(shape, bufs) -> dict:
    """Device bytes of the forward state the backward reads (caller-owned
    buffers kept from the forward to the backward): with the routing weight
    inside the expert the permuted expert outputs y_perm are read only by the
    combine, so their buffer need not survive until the backward; with the
    fine-grained recompute the backward rewrites h from GU, so neither does h's."""
    f = bufs.fwd
    kept = ["logits", "idx", "w", "counts", "offsets", "row_of", "token_of", "sel_offsets",
            "sel_tokens", "x_perm", "GU"]
    if not shape.weights_in_expert:
        kept.append("y_perm")
    if not shape.recompute_h:
        kept.append("h")
    n = sum(f[k].numel() * f[k].element_size() for k in kept)
    return {"forward_state_kept": n, "y_perm": f["y_perm"].numel() * f["y_perm"].element_size(),
            "y_perm_kept": not shape.weights_in_expert,
            "h": f["h"].numel() * f["h"].element_size(), "h_kept": not shape.recompute_h}


STAGES = ("route", "permute", "quantize_weights", "grouped_ffn_fwd", "unpermute",
          "unpermute_bwd", "route_bwd", "grouped_ffn_dgrad", "grouped_ffn_wgrad", "permute_bwd",
          "router_wgrad")


def wgrad_bytes(shape, f) -> int:
    """Bytes the FP8 weight-gradient stage must move: per live row of the
    permuted buffers, dO, h and x_perm read in bf16 (2 B), written as E4M3
    (1 B) and read back by the GEMMs (1 B), and dGU's E4M3 column form (which
    the data-gradient stage writes) read by the GEMM (1 B); dW2 and dW13
    written in bf16."""
    H, F, G = shape.H, shape.F, shape.E + shape.n_shared
    counts = f["counts"].cpu().tolist()
    live = sum(-(-c // 128) * 128 for c in counts)
    return live * ((H + F + H) * 4 + 2 * F) + G * 3 * H * F * 2


def stage_table(shape, f, stage_ms, hbm_gbs, fl, tc_peak, bf16_peak):
    """Per-stage device time, algorithmic bytes (or flops) and roofline fraction.

    Bytes count each tensor a stage must read or write once (bf16 rows 2 B per
    element, fp32 4 B, int32 maps 4 B, E4M3 1 B plus 1/32 B of scale atoms): A
    kept routed assignments, S*T shared rows, P zero padding rows of the
    permuted buffers. GEMM stages count flops against the tensor peak of their
    operand type. The FP8 weight-gradient stage also gets its bytes: its four
    128x1 quantisers read the bf16 operands' live rows and write their E4M3
    codes, the two GEMMs read those codes and write dW2 and dW13 in bf16."""
    T, H, E, k, S, F = shape.T, shape.H, shape.E, shape.k, shape.n_shared, shape.F
    counts = f["counts"].cpu().tolist()
    offsets = f["offsets"].cpu().tolist()
    G = E + S
    A = sum(counts[:E])
    rows = A + S * T                     # filled rows of the permuted buffers
    P = offsets[G] - sum(counts)         # padding rows
    bf = 2
    maps = T * k * 4 * 3                 # idx / row_of / w sized reads or writes
    fp8 = shape.dtype in W.FP8_DTYPES
    mx = shape.dtype == W.DT_MXFP8
    wbytes = G * 3 * H * F
    blk = 32 if mx else 128
    work = [
        ("route", T * H * bf + E * H * 4 + T * E * 4 + 2 * T * k * 4, "router logits + top-k"),
        ("permute", T * H * bf + (rows + P) * H * bf + maps, "hist + rank + row scatter"),
        # bf16 read, E4M3 written (twice for MX: forward and data-gradient
        # forms); scale bytes: 128 per 128x128 tile for each of the two atom
        # arrays, or one per 32 elements for each form (MX)
        ("quantize_weights", (wbytes * bf + (2 * wbytes + wbytes // 16 if mx else
                                             wbytes + wbytes // 64)) if fp8 else 0,
         "E4M3 weights + UE8M0 scale atoms (FP8 only)"),
        ("grouped_ffn_fwd", fl, "FC1+SwiGLU, FC2 (tcgen05" + (" kind::mxf8f6f4)" if fp8 else ")")),
        ("unpermute", rows * H * bf + T * H * bf + maps, "gather-scale-reduce"),
        ("unpermute_bwd", T * H * bf + A * H * bf + (rows + P) * H * bf + maps,
         "dO scatter + dw dot products"),
        ("route_bwd", T * E * 4 * 2 + maps, "dlogits"),
        ("grouped_ffn_dgrad", fl, "FC2 dgrad+SwiGLU bwd, FC1 dgrad (tcgen05"
         + (" kind::mxf8f6f4)" if fp8 else ")")),
        ("grouped_ffn_wgrad", fl, "dW2, dW13 (tcgen05"
         + (f" kind::mxf8f6f4, with their three {blk}x1 quantisers)" if fp8 else " bf16)")),
        ("permute_bwd", rows * H * bf + T * H * bf + maps, "dx gather-reduce"),
        ("router_wgrad", T * H * bf + E * H * 4 + T * E * 4, "dW_r (each x row once)"),
    ]
    out = []
    for (name, w, what), ms in zip(work, stage_ms):
        if name.startswith("grouped_ffn"):
            ach = w / (ms * 1e-3) / 1e12
            row = {"stage": name, "what": what, "ms": ms, "tflop": w / 1e12,
                   "tflops": ach, "frac_tensor": ach / tc_peak}
            if fp8 and name == "grouped_ffn_wgrad":
                wb = wgrad_bytes(shape, f)
                row.update({"mb": wb / 1e6, "gbs": wb / (ms * 1e-3) / 1e9,
                            "frac_hbm": wb / (ms * 1e-3) / 1e9 / hbm_gbs})
            out.append(row)
        elif w > 0:
            ach = w / (ms * 1e-3) / 1e9
            out.append({"stage": name, "what": what, "ms": ms, "mb": w / 1e6,
                        "gbs": ach, "frac_hbm": ach / hbm_gbs})
    return out


# ---------------------------------------------------------------------------- ours
def run_ours(args, rank, world, local):
    import routing_dispatch_expert_router_gb300.binding as B
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = {**W.SHAPES, **W.PROFILE_SHAPES}[args.workload]
    if args.weights_in_expert:
        shape = shape.with_(weights_in_expert=1)
    if args.recompute_h:
        shape = shape.with_(recompute_h=1)
    cfg = B.config(shape)
    inp = W.make_inputs(shape, seed=args.seed + rank, device=str(dev))
    bufs = B.alloc_buffers(cfg, dev)
    T, H, E, F, S = shape.T, shape.H, shape.E, shape.F, shape.n_shared
    G = E + S
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    dx = torch.empty_like(out)
    dW_r = torch.empty(E, H, dtype=torch.float32, device=dev)
    dW13 = torch.empty(G, 2 * F, H, dtype=torch.bfloat16, device=dev)
    dW2 = torch.empty(G, H, F, dtype=torch.bfloat16, device=dev)
    P = B.params(inp["W_r"], inp["bias"], inp["W13"], inp["W2"])
    f, b = bufs.fwd, bufs.bwd
    x, dY = inp["x"], inp["dY"]
    stream = torch.cuda.current_stream(dev)
    sc = bufs.scratch

    fp8 = shape.dtype in W.FP8_DTYPES
    mx = shape.dtype == W.DT_MXFP8
    reord = bool(shape.weights_in_expert)
    # fine-grained recompute: the data gradient rewrites h from GU
    h_re = f["h"] if shape.recompute_h else None

    def step(ev=None):
        # the layer step through the per-stage entry points (the same launches
        # as moe_layer_fwd + moe_layer_bwd); ev[i] is recorded after stage i
        # (ev[0] before the first), so every stage gets its own device time
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        B.moe_route(cfg, x, inp["W_r"], inp["bias"], f["logits"], f["idx"], f["w"], sc)
        rec(1)
        B.moe_permute(cfg, x, f["idx"], f["counts"], f["offsets"], f["row_of"], f["token_of"],
                      f["sel_offsets"], f["sel_tokens"], f["x_perm"], sc)
        rec(2)
        B.moe_quantize_weights(cfg, inp["W13"], inp["W2"], sc)
        rec(3)
        if reord:
            # the routing weight inside the expert: no y_perm read in the
            # backward; dw and dlogits come out of the data-gradient stage
            B.moe_grouped_ffn_fwd_reordered(cfg, f["x_perm"], f["counts"], f["offsets"],
                                            f["token_of"], f["row_of"], f["w"], inp["W13"],
                                            inp["W2"], f["GU"], f["h"], f["y_perm"], sc)
            rec(4)
            B.moe_unpermute(cfg, f["y_perm"], f["row_of"], None, f["offsets"], out)
            rec(5)
            B.moe_unpermute_bwd_reordered(cfg, dY, f["row_of"], f["counts"], f["offsets"],
                                          b["dO_perm"])
            rec(6)
            rec(7)
            B.moe_grouped_ffn_dgrad_reordered(cfg, b["dO_perm"], f["GU"], h_re, f["counts"],
                                              f["offsets"], f["token_of"], f["row_of"],
                                              f["logits"], f["idx"], f["w"], inp["W_r"],
                                              inp["W13"], inp["W2"], b["dGU"], b["dX_perm"],
                                              b["dw"], b["dlogits"], sc)
        else:
            B.moe_grouped_ffn_fwd(cfg, f["x_perm"], f["counts"], f["offsets"], inp["W13"],
                                  inp["W2"], f["GU"], f["h"], f["y_perm"], sc)
            rec(4)
            B.moe_unpermute(cfg, f["y_perm"], f["row_of"], f["w"], f["offsets"], out)
            rec(5)
            B.moe_unpermute_bwd(cfg, dY, f["y_perm"], f["row_of"], f["w"], f["counts"],
                                f["offsets"], b["dO_perm"], b["dw"], sc)
            rec(6)
            B.moe_route_bwd(cfg, f["logits"], f["idx"], f["w"], b["dw"], b["dlogits"])
            rec(7)
            B.moe_grouped_ffn_dgrad(cfg, b["dO_perm"], f["GU"], h_re, f["counts"], f["offsets"],
                                    f["token_of"], b["dlogits"], inp["W_r"], inp["W13"],
                                    inp["W2"], b["dGU"], b["dX_perm"], sc)
        rec(8)
        B.moe_grouped_ffn_wgrad(cfg, b["dO_perm"], f["x_perm"], f["h"], b["dGU"], f["counts"],
                                f["offsets"], dW13, dW2, sc)
        rec(9)
        B.moe_permute_bwd(cfg, b["dX_perm"], f["row_of"], f["offsets"], f["idx"], b["dlogits"],
                          inp["W_r"], dx)
        rec(10)
        B.moe_router_wgrad(cfg, x, f["sel_offsets"], f["sel_tokens"], b["dlogits"], dW_r, sc)
        rec(11)

    # kernels launched by one step: route (logits [+ W_r split on the tensor-core
    # path] + selection), dispatch (hist, rank, scatter), FC1 and FC2, combine,
    # combine bwd, route bwd, the four backward GEMMs, dispatch bwd, router wgrad
    # (on the tensor-core path: dlogits split, GEMM, chunk sum); the FP8 mode adds
    # the two weight quantisers, dGU's row-and-column quantiser in the data
    # gradients and three column quantisers in the weight gradients (x_perm's, h's and dO's
    # row forms come out of the scatter, the FC1 epilogue and the combine
    # backward, in either recipe)
    tc_router = shape.E >= 128 and shape.E % 128 == 0
    launches_per_step = ((3 if tc_router else 2) + 3 + 2 + 1 + 1 + 1 + 4 + 1
                         + (3 if tc_router else 1))
    if fp8:
        launches_per_step += 2 + 1 + 3
    if reord:
        launches_per_step += 2          # row weights, dw reduction
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    status = B.moe_last_device_status(sc)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    counts = f["counts"].cpu().tolist()
    fl = gemm_flops(shape, counts)
    nst = len(STAGES)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
           for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1)
    stage_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i in range(nst)]
    sm = dict(zip(STAGES, stage_ms))

    # end to end through the public layer calls, host buffers: every step copies
    # its x and dY from pinned host memory and reads out and dx back. Uploads and
    # downloads run on two more streams (one per direction, so the two copy
    # directions proceed at once), double-buffered and ordered by events, so
    # step i+1's uploads and step i's downloads overlap the neighbouring compute.
    # paged stash: the end-to-end leg runs on a pool of exactly the pages the
    # layer's kept rows need (its own page table, scratch and backward buffers);
    # the device-resident step above keeps the worst-case buffers
    cfg_e, bufs_e, stash = cfg, bufs, None
    if args.paged_stash:
        pages = sum(-(-int(c) // 128) for c in counts)
        cfg_e = B.config(shape)
        cfg_e.stash_pool_pages = pages
        pool = B.alloc_stash_pool(cfg_e, pages, dev)
        bufs_e = B.alloc_buffers(cfg_e, dev, pool=pool)
        row_bytes = 2 * H + 4 * F + 2 * F + 2 * H        # x_perm, GU, h, y_perm (bf16)
        R = int(bufs.sizes.rows_max)
        stash = {"pool_pages": pages, "pool_rows": (pages + 1) * 128,
                 "pool_bytes": (pages + 1) * 128 * row_bytes,
                 "worst_case_rows": R, "worst_case_bytes": R * row_bytes,
                 "what": "x_perm, GU, h, y_perm of the end-to-end leg in a pool of 128-row pages "
                         "taken on the device (one spill page more), against rows_max rows"}
    cs = torch.cuda.Stream(dev)                       # uploads
    cd = torch.cuda.Stream(dev)                       # downloads
    xh = [x.cpu().pin_memory() for _ in range(2)]
    dYh = [dY.cpu().pin_memory() for _ in range(2)]
    outh = [torch.empty_like(xh[0]).pin_memory() for _ in range(2)]
    dxh = [torch.empty_like(xh[0]).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    dYd = [torch.empty_like(dY) for _ in range(2)]
    outd = [torch.empty_like(out) for _ in range(2)]
    dxd = [torch.empty_like(dx) for _ in range(2)]
    up = [torch.cuda.Event() for _ in range(2)]       # inputs of buffer b uploaded
    done = [torch.cuda.Event() for _ in range(2)]     # compute on buffer b finished
    down = [torch.cuda.Event() for _ in range(2)]     # results of buffer b downloaded

    def upload(b):
        with torch.cuda.stream(cs):
            cs.wait_event(done[b])                    # previous compute on b is finished
            xd[b].copy_(xh[b], non_blocking=True)
            dYd[b].copy_(dYh[b], non_blocking=True)
            up[b].record(cs)

    def e2e_run(n):
        for b in range(2):
            done[b].record(stream)
            down[b].record(stream)
        upload(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                upload(1 - b)
            stream.wait_event(up[b])
            stream.wait_event(down[b])                # results of step i-2 are out
            B.moe_layer_fwd(cfg_e, P, xd[b], outd[b], bufs_e.fwd_struct, bufs_e.scratch)
            B.moe_layer_bwd(cfg_e, P, xd[b], dYd[b], bufs_e.fwd_struct, bufs_e.bwd_struct,
                            dxd[b], dW_r, dW13, dW2, bufs_e.scratch)
            done[b].record(stream)
            with torch.cuda.stream(cd):
                cd.wait_event(done[b])
                outh[b].copy_(outd[b], non_blocking=True)
                dxh[b].copy_(dxd[b], non_blocking=True)
                down[b].record(cd)
        stream.wait_stream(cs)
        stream.wait_stream(cd)

    e2e_run(3)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    status = B.moe_last_device_status(sc) or B.moe_last_device_status(bufs_e.scratch)
    if status != 0:
        raise RuntimeError(f"device status {status} after timed steps")
    if not torch.equal(outh[(args.steps - 1) & 1], out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident run")

    times = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(times, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms = times.tolist()
    pk, src = peaks()
    bf16_peak = pk["bf16_tflops"]                  # burst: the kernels are timed in a short loop
    tc_peak = 2.0 * bf16_peak if fp8 else bf16_peak
    if fp8:
        gemm_ms = sm["grouped_ffn_fwd"] + sm["grouped_ffn_dgrad"]
        gemm_fl = 2 * fl
        kern = (f"grouped_gemm_fp8_kernel (tcgen05 kind::mxf8f6f4, E4M3 x UE8M0 "
                f"{32 if mx else 128}-blocks: FC1+SwiGLU, FC2, FC2 dgrad+SwiGLU bwd, FC1 dgrad)")
        peak_src = (f"{src}: 2 x bf16_tflops (the nominal FP8:bf16 dense rate ratio; no FP8 "
                    "figure is measured)")
        gemm_note = ("time of the grouped_ffn_fwd and grouped_ffn_dgrad stages, which also hold "
                     "the activation quantisers (h's in the FC1 epilogue, dGU's pass)")
    else:
        gemm_ms = sm["grouped_ffn_fwd"] + sm["grouped_ffn_dgrad"] + sm["grouped_ffn_wgrad"]
        gemm_fl = 3 * fl
        kern = "grouped_gemm_kernel (tcgen05 kind::f16; FC1+SwiGLU, FC2, 2 dgrad, 2 wgrad)"
        peak_src = f"{src}: bf16_tflops"
        gemm_note = "time of the three grouped-FFN stages"
    achieved = gemm_fl / (gemm_ms * 1e-3) / 1e12
    tokens = T * args.steps * world
    cf = shape.capacity_factor
    dt_name = ("mxfp8_e4m3_32" if mx else "fp8_e4m3_block") if fp8 else "bf16"
    res = {
        "metric": "MoE-layer tokens/s fwd+bwd on 1 GB300",
        "value": tokens / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dt_name,
        "dtype_detail": (("E4M3 operands with one UE8M0 power-of-two scale per 32 elements (MX): "
                          "1x32 along K for activations, each weight in two forms (1x32 along K "
                          "for the forward, 32x1 for the data gradients), 32x1 along the tokens "
                          "for the weight gradients" if mx else
                          "E4M3 operands with UE8M0 power-of-two scales per 128x128 weight tile, "
                          "1x128 activation slice along K (forward and data gradients) and "
                          "128x1 slice along the tokens (weight gradients)")
                         + "; all six expert GEMMs on the block-scaled FP8 tensor cores with "
                         "fp32 accumulation; router fp32; activations and outputs bf16"
                         if fp8 else "bf16 operands, fp32 accumulation, fp32 router"),
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02^2) weights; no dataset)",
        "config": {"workload": f"{shape.name}: T={T} H={H} E={E}(+{S} shared) top-{shape.k} "
                               f"F={F} capacity_factor={cf if cf > 0 else 'dropless'} "
                               f"dtype={dt_name}"
                               + (" weights_in_expert" if reord else "")
                               + (" recompute_h" if shape.recompute_h else "")
                               + (" paged_stash(e2e)" if args.paged_stash else "") + " fwd+bwd",
                   "l2": "inputs larger than L2 (expert weights "
                         f"{2 * G * 3 * H * F / 1e9:.2f} GB in bf16, streamed every step)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * T * H * 2, "d2h_bytes_per_step": 2 * T * H * 2},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": kern, "bound": "tensor", "achieved": achieved, "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": achieved / tc_peak, "peak_source": peak_src,
                     "traffic": gemm_traffic(shape.name),
                     "traffic_note": "DRAM bytes of this kernel's launches in one step "
                                     "(ncu dram__bytes_read+write, profiles/gemm_traffic.json); "
                                     "achieved is per step too",
                     "gemm_ms_per_step": gemm_ms, "gemm_time_note": gemm_note,
                     "gemm_tflop_per_step": gemm_fl / 1e12,
                     "frac_of_sustained": achieved / (2.0 * pk.get("bf16_tflops_sustained",
                                                                   bf16_peak) if fp8 else
                                                      pk.get("bf16_tflops_sustained",
                                                             bf16_peak))},
        "stages": stage_table(shape, f, stage_ms, pk["hbm_gbs"], fl, tc_peak, bf16_peak),
        "stash_bytes": stash_bytes(shape, bufs),
        "paged_stash": stash,
        "clocks": clk,
    }
    if fp8:
        # the weight gradients write both expert weights in bf16 every step:
        # bound by HBM, not by the FP8 tensor rate
        wb = wgrad_bytes(shape, f)
        wms = sm["grouped_ffn_wgrad"]
        res["roofline_wgrad"] = {
            "kernel": ("grouped_gemm_fp8_kernel<kEpiWgrad> (tcgen05 kind::mxf8f6f4, K = each "
                       "expert's rows) with the column quantisers of dO, h and x_perm"),
            "bound": "hbm", "achieved": wb / (wms * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": wb / (wms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "bytes_per_step": wb, "ms_per_step": wms,
            "traffic": gemm_traffic(shape.name, "wgrad_stage_dram_bytes_per_step"),
            "tflops": fl / (wms * 1e-3) / 1e12,
            "note": "of measured copy bandwidth; the stage writes the weight gradients "
                    f"({G * 3 * H * F * 2 / 1e9:.2f} GB bf16)"}
    return res, shape, inp


# ---------------------------------------------------------------------- the oracle
def oracle_subproblem(shape, inp: dict, max_tokens: int, max_experts: int):
    """A bounded sample of the workload for the CPU oracle: the first n tokens
    (n <= max_tokens) that together select at most max(max_experts, k)
    experts, with the layer restricted to those experts.

    The oracle's own router scores the sampled tokens against all E experts
    (timed); the layer functions then run on a problem of the selected
    experts only, so no other expert's weights are converted to fp64 and no
    other expert's weight gradient is allocated. Each sampled token keeps its
    experts and routing weights: the restricted logits hold the token's
    scores (softmax: logit + bias) at its selected experts and -700 elsewhere,
    which the restricted top-k (no groups, no bias) passes over. The first
    tokens are never dropped by the capacity limit (it keeps an expert's first
    C tokens, C >= 128), so the restricted problem is dropless."""
    from oracle import moe_oracle as O
    h = lambda t: t.detach().to("cpu").double().numpy()  # noqa: E731
    Wr = h(inp["W_r"])
    bias = None if inp["bias"] is None else h(inp["bias"])
    n_try = min(shape.T, max_tokens)
    x_all = h(inp["x"][:n_try])
    idx, _ = O.route(O.router_logits(x_all, Wr), shape, bias)
    cap = max(max_experts, shape.k)
    used = set(int(e) for e in idx[0])
    n = 1
    while n < n_try and len(used | set(int(e) for e in idx[n])) <= cap:
        used |= set(int(e) for e in idx[n])
        n += 1
    U = sorted(used)
    pos = {e: i for i, e in enumerate(U)}
    sub = shape.with_(T=n, E=len(U), n_groups=1, topk_groups=1, capacity_factor=0.0,
                      bias_kind="none")
    sel = torch.as_tensor(U, device=inp["W13"].device)
    return {"shape": shape, "sub": sub, "n": n, "experts": U, "pos": pos, "x": x_all[:n],
            "dY": h(inp["dY"][:n]), "W_r": Wr, "bias": bias, "W_r_sub": Wr[U],
            "W13": h(inp["W13"][sel]), "W2": h(inp["W2"][sel])}


def oracle_sample(o: dict) -> float:
    """Seconds the CPU oracle takes for fwd+bwd of the sampled tokens: the
    router logits over all experts, the selection, then the layer on the
    selected experts (FP8 layer functions for the FP8 configuration)."""
    from oracle import moe_oracle as O
    shape, sub = o["shape"], o["sub"]
    t0 = time.perf_counter()
    lg = O.router_logits(o["x"], o["W_r"])
    idx, _ = O.route(lg, shape, o["bias"])
    score = lg + (o["bias"] if (o["bias"] is not None and shape.score_fn == O.SOFTMAX) else 0.0)
    lg_sub = np.full((sub.T, sub.E), -700.0)
    for t in range(sub.T):
        for e in idx[t]:
            lg_sub[t, o["pos"][int(e)]] = score[t, int(e)]
    if shape.dtype in W.FP8_DTYPES:
        fwd = O.layer_forward_fp8(sub, o["x"], o["W_r_sub"], None, o["W13"], o["W2"], logits=lg_sub)
        O.layer_backward_fp8(sub, o["x"], o["W_r_sub"], o["W13"], o["W2"], fwd, o["dY"])
    else:
        fwd = O.layer_forward(sub, o["x"], o["W_r_sub"], None, o["W13"], o["W2"], logits=lg_sub)
        O.layer_backward(sub, o["x"], o["W_r_sub"], o["W13"], o["W2"], fwd, o["dY"])
    return time.perf_counter() - t0


def sample_text(o: dict, steps: int = 1) -> str:
    sh = o["shape"]
    return (f"first {o['n']} tokens of {sh.name} ({len(o['experts'])} of {sh.E} experts "
            f"selected), {steps} pass(es): router logits over all experts, selection, then "
            "fwd+bwd of the selected experts incl. their weight gradients"
            + (" (FP8 layer functions)" if sh.dtype in W.FP8_DTYPES else "") + ", fp64 numpy")


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    """The oracle as the reference arm: each step runs the oracle's fwd+bwd on
    the bounded sample of the workload that cpu_baseline uses, on the host
    cores. The inputs are drawn with the same seeded recipe (on the GPU when
    there is one, which only draws the random numbers); a step takes tens of
    seconds on the large shapes, so fewer steps than requested run when they
    would not fit in about --ref-budget-s seconds ("steps", with
    "steps_requested")."""
    shape = {**W.SHAPES, **W.PROFILE_SHAPES}[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_inputs(shape, seed=args.seed, device=dev)
    o = oracle_subproblem(shape, inp, args.cpu_sample_tokens or 64, 8)
    del inp
    t1 = oracle_sample(o)                                         # warm-up and probe
    want = max(args.steps, 1)
    steps = int(min(want, max(1, args.ref_budget_s / max(t1, 1e-6))))
    secs = [oracle_sample(o) for _ in range(steps)]
    tot = sum(secs)
    val = o["n"] * steps / tot
    cb = {"value": val, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
          "sample": sample_text(o, steps)}
    return {"impl": "reference", "metric": "MoE-layer tokens/s fwd+bwd on 1 GB300", "value": val,
            "unit": "tokens/s", "n_gpus": 1, "steps": steps, "steps_requested": args.steps,
            "warmup": 1, "ms_per_step": 1e3 * tot / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": shape.name}, "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    res, shape, inp = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            n_tok = args.cpu_sample_tokens or (shape.T if shape.name == "tiny" else 64)
            o = oracle_subproblem(shape, inp, n_tok, 8)
            del inp
            secs = oracle_sample(o)
            res["cpu_baseline"] = {"value": o["n"] / secs, "unit": "tokens/s",
                                   "cores": cpu_cores(), "kind": "oracle",
                                   "sample": sample_text(o)}
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
