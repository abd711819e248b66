"""Benchmark of one MoE layer step (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixtral]
                    [--impl ours|reference]

A step is one pass of the whole layer over one batch of synthetic tokens:
route, permute, grouped SwiGLU FFN, unpermute, and the backward of all of it
(dx, dW_r, dW13, dW2). The default workload is the Mixtral-style layer
(T=4096, H=4096, E=8, top-2 softmax, d_ff=14336, bf16). Prints one JSON line.

  value      tokens/s of fwd+bwd with inputs resident in HBM (CUDA events)
  e2e        the same through the public layer calls with host buffers: each
             step copies x and dY from pinned host memory and reads out and dx
             back inside the timed region
  roofline   the grouped-GEMM kernel family (the dominant kernel) against the
             measured dense bf16 tensor peak
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
    ap.add_argument("--workload", default="mixtral",
                    choices=sorted(W.SHAPES) + sorted(W.PROFILE_SHAPES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
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
                 "--format=csv,noheader,nounits", "-lms", "200"],
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


def gemm_traffic(workload: str):
    """DRAM bytes per step of the grouped-GEMM launches from a committed ncu
    capture, or None when the GEMM source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    src = os.path.join(ROOT, "routing_dispatch_expert_router_gb300", "csrc", "grouped_gemm.cu")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    if d.get("grouped_gemm_cu_sha256") != h or d.get("workload") != workload:
        return None
    return d.get("dram_bytes_per_step")


def gemm_flops(shape, counts) -> tuple:
    """Algorithmic flops of the grouped GEMMs of one step (kept rows only)."""
    rows = float(sum(counts))        # routed kept rows + shared rows (T each)
    fwd = 2.0 * rows * shape.H * 2 * shape.F + 2.0 * rows * shape.F * shape.H
    bwd = 2.0 * fwd
    return fwd, bwd


def stage_table(shape, cfg, f, stage_ms, hbm_gbs, fl_fwd, fl_bwd, tc_peak):
    """Per-stage device time, algorithmic bytes (or flops) and roofline fraction.

    Bytes count each tensor a stage must read or write once (bf16 rows 2 B per
    element, fp32 4 B, int32 maps 4 B): A kept routed assignments, S*T shared
    rows, P zero padding rows of the permuted buffers."""
    T, H, E, k, S = shape.T, shape.H, shape.E, shape.k, shape.n_shared
    counts = f["counts"].cpu().tolist()
    offsets = f["offsets"].cpu().tolist()
    G = E + S
    A = sum(counts[:E])
    rows = A + S * T                     # filled rows of the permuted buffers
    P = offsets[G] - sum(counts)         # padding rows
    bf = 2
    maps = T * k * 4 * 3                 # idx / row_of / w sized reads or writes
    work = [
        ("route", T * H * bf + E * H * 4 + T * E * 4 + 2 * T * k * 4, "router logits + top-k"),
        ("permute", T * H * bf + (rows + P) * H * bf + maps, "hist + rank + row scatter"),
        ("grouped_ffn_fwd", fl_fwd, "FC1+SwiGLU, FC2 (tcgen05)"),
        ("unpermute", rows * H * bf + T * H * bf + maps, "gather-scale-reduce"),
        ("unpermute_bwd", T * H * bf + A * H * bf + (rows + P) * H * bf + maps,
         "dO scatter + dw dot products"),
        ("route_bwd", T * E * 4 * 2 + maps, "dlogits"),
        ("grouped_ffn_bwd", fl_bwd, "FC2 dgrad+SwiGLU bwd, FC1 dgrad, dW2, dW13 (tcgen05)"),
        ("permute_bwd", rows * H * bf + T * H * bf + maps, "dx gather-reduce"),
        ("router_wgrad", T * H * bf + E * H * 4 + T * E * 4, "dW_r (each x row once)"),
    ]
    out = []
    for (name, w, what), ms in zip(work, stage_ms):
        if name.startswith("grouped_ffn"):
            ach = w / (ms * 1e-3) / 1e12
            out.append({"stage": name, "what": what, "ms": ms, "tflop": w / 1e12,
                        "tflops": ach, "frac_tensor": ach / tc_peak})
        else:
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
        B.moe_grouped_ffn_fwd(cfg, f["x_perm"], f["counts"], f["offsets"], inp["W13"], inp["W2"],
                              f["GU"], f["h"], f["y_perm"], sc)
        rec(3)
        B.moe_unpermute(cfg, f["y_perm"], f["row_of"], f["w"], f["offsets"], out)
        rec(4)
        B.moe_unpermute_bwd(cfg, dY, f["y_perm"], f["row_of"], f["w"], f["counts"], f["offsets"],
                            b["dO_perm"], b["dw"])
        rec(5)
        B.moe_route_bwd(cfg, f["logits"], f["idx"], f["w"], b["dw"], b["dlogits"])
        rec(6)
        B.moe_grouped_ffn_bwd(cfg, b["dO_perm"], f["x_perm"], f["GU"], f["h"], f["counts"],
                              f["offsets"], f["token_of"], b["dlogits"], inp["W_r"], inp["W13"],
                              inp["W2"], b["dGU"], b["dX_perm"], dW13, dW2, sc)
        rec(7)
        B.moe_permute_bwd(cfg, b["dX_perm"], f["row_of"], f["offsets"], f["idx"], b["dlogits"],
                          inp["W_r"], dx)
        rec(8)
        B.moe_router_wgrad(cfg, x, f["sel_offsets"], f["sel_tokens"], b["dlogits"], dW_r, sc)
        rec(9)

    # kernels launched by one step: route (logits [+ W_r split on the tensor-core
    # path] + selection), dispatch (hist, rank, scatter), FC1 and FC2, combine,
    # combine bwd, route bwd, the four backward GEMMs, dispatch bwd, router wgrad
    # (on the tensor-core path: dlogits split, GEMM, chunk sum); the FP8 mode adds
    # 4 quantisation launches forward and 6 backward
    tc_router = shape.E >= 128 and shape.E % 128 == 0
    launches_per_step = ((3 if tc_router else 2) + 3 + 2 + 1 + 1 + 1 + 4 + 1
                         + (3 if tc_router else 1))
    if shape.dtype == W.DT_FP8:
        launches_per_step += 4 + 6
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    status = B.moe_last_device_status(sc)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    counts = f["counts"].cpu().tolist()
    fl_fwd, fl_bwd = gemm_flops(shape, counts)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(args.steps)]
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
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    stage_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i in range(9)]
    fwd_gemm_ms, bwd_gemm_ms = stage_ms[2], stage_ms[6]
    gemm_ms = fwd_gemm_ms + bwd_gemm_ms

    # end to end through the public layer calls, host buffers: every step copies
    # its x and dY from pinned host memory and reads out and dx back. Copies run
    # on a second stream, double-buffered and ordered by events, so step i+1's
    # uploads and step i's downloads overlap the neighbouring compute.
    cs = torch.cuda.Stream(dev)
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
            B.moe_layer_fwd(cfg, P, xd[b], outd[b], bufs.fwd_struct, sc)
            B.moe_layer_bwd(cfg, P, xd[b], dYd[b], bufs.fwd_struct, bufs.bwd_struct, dxd[b], dW_r,
                            dW13, dW2, sc)
            done[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(done[b])
                outh[b].copy_(outd[b], non_blocking=True)
                dxh[b].copy_(dxd[b], non_blocking=True)
                down[b].record(cs)
        stream.wait_stream(cs)

    e2e_run(3)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    status = B.moe_last_device_status(sc)
    if status != 0:
        raise RuntimeError(f"device status {status} after timed steps")
    if not torch.equal(outh[(args.steps - 1) & 1], out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident run")

    times = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(times, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms = times.tolist()
    pk, src = peaks()
    peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    achieved = (fl_fwd + fl_bwd) / (gemm_ms * 1e-3) / 1e12
    tokens = T * args.steps * world
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
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02^2) weights; no dataset)",
        "config": {"workload": f"{shape.name}: T={T} H={H} E={E}(+{S} shared) top-{shape.k} "
                               f"F={F} fwd+bwd", "l2": "inputs larger than L2 (weights "
                               f"{2 * G * 3 * H * F / 1e9:.2f} GB streamed per step)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * T * H * 2, "d2h_bytes_per_step": 2 * T * H * 2},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": "grouped_gemm_kernel (tcgen05; FC1+SwiGLU, FC2, 2 dgrad, 2 wgrad)",
                     "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{src} bf16_tflops_sustained",
                     "traffic": gemm_traffic(shape.name),
                     "traffic_note": "DRAM bytes of the six grouped-GEMM launches of one step "
                                     "(ncu dram__bytes_read+write); achieved is per step too",
                     "gemm_ms_per_step": gemm_ms,
                     "fwd_gemm_ms": fwd_gemm_ms, "bwd_gemm_ms": bwd_gemm_ms,
                     "gemm_tflop_per_step": (fl_fwd + fl_bwd) / 1e12},
        "stages": stage_table(shape, cfg, f, stage_ms, pk["hbm_gbs"], fl_fwd, fl_bwd, peak),
        "clocks": clk,
    }
    return res, shape, inp


# ---------------------------------------------------------------------- the oracle
def oracle_inputs(inp: dict, n_tok: int) -> dict:
    """Host fp64 copies of the first n_tok tokens and all weights (not timed)."""
    h = lambda t: None if t is None else t.detach().to("cpu").double().numpy()  # noqa: E731
    return {"x": h(inp["x"][:n_tok]), "dY": h(inp["dY"][:n_tok]), "W_r": h(inp["W_r"]),
            "bias": h(inp["bias"]), "W13": h(inp["W13"]), "W2": h(inp["W2"])}


def oracle_sample(shape, o: dict) -> float:
    """Seconds the CPU oracle takes for fwd+bwd of the sampled tokens."""
    from oracle import moe_oracle as O
    sub = shape.with_(T=o["x"].shape[0])
    t0 = time.perf_counter()
    fwd = O.layer_forward(sub, o["x"], o["W_r"], o["bias"], o["W13"], o["W2"])
    O.layer_backward(sub, o["x"], o["W_r"], o["W13"], o["W2"], fwd, o["dY"])
    return time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    """The oracle as the reference arm: every step runs its fwd+bwd (weight
    gradients included) on a sample of the workload's tokens, on the host cores.

    A step of the oracle has a floor that does not shrink with the sample (it
    builds every expert's full-size fp64 weight gradient), so the run is held
    to about --ref-budget-s seconds: a timed 1-token step (also the warm-up)
    sizes the sample (1 token at least, the whole batch at most) and, when even
    1-token steps do not fit, fewer steps than requested run; the JSON line says
    how many ("steps", with "steps_requested")."""
    shape = {**W.SHAPES, **W.PROFILE_SHAPES}[args.workload]
    want = max(args.steps, 1)
    o_all = oracle_inputs(W.make_inputs(shape, seed=args.seed, device="cpu"), shape.T)
    t1 = oracle_sample(shape, oracle_inputs_slice(o_all, 1))            # warm-up and probe
    if args.cpu_sample_tokens:
        n_tok = min(args.cpu_sample_tokens, shape.T)
        steps = want
    else:
        n_tok = int(min(shape.T, max(1, args.ref_budget_s / (want * max(t1, 1e-6)))))
        steps = int(min(want, max(1, args.ref_budget_s / (n_tok * max(t1, 1e-6)))))
    o = oracle_inputs_slice(o_all, n_tok)
    secs = [oracle_sample(shape, o) for _ in range(steps)]
    tot = sum(secs)
    val = n_tok * steps / tot
    cb = {"value": val, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
          "sample": f"first {n_tok} tokens of {shape.name} per step, {steps} steps (routing, "
                    "experts, combine, full backward incl. every expert's weight gradient), "
                    "fp64 numpy"}
    return {"impl": "reference", "metric": "MoE-layer tokens/s fwd+bwd on 1 GB300", "value": val,
            "unit": "tokens/s", "n_gpus": 1, "steps": steps, "steps_requested": args.steps,
            "warmup": 1, "ms_per_step": 1e3 * tot / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": shape.name}, "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def oracle_inputs_slice(o: dict, n: int) -> dict:
    d = dict(o)
    d["x"] = o["x"][:n]
    d["dY"] = o["dY"][:n]
    return d


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
            o = oracle_inputs(inp, n_tok)
            del inp
            secs = oracle_sample(shape, o)
            res["cpu_baseline"] = {
                "value": n_tok / secs, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                "sample": f"first {n_tok} tokens of {shape.name}: oracle fwd+bwd incl. weight "
                          "gradients of those tokens, fp64 numpy, one pass"}
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
