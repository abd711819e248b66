"""Time each stage of the layer alone, on its own buffers, with a cold L2.

    python -m routing_dispatch_expert_router_gb300.stages [workload ...] [--reps N] [--no-flush]

For every workload (default: mixtral) the route, dispatch, combine, combine
backward, route backward, dispatch backward and router weight-gradient entry
points, and the load-balancing loss (forward and backward), run once as warm-up and then N times (default 20), each timed with CUDA
events after a 512 MB write that evicts L2. Prints the median time, the
stage's algorithmic bytes (every tensor read or written once) and the rate
against the measured copy bandwidth. The grouped GEMMs are timed by bench.py.
Inputs come from workloads.make_inputs (the routing inputs) and seeded
normal rows for the permuted buffers.
"""
from __future__ import annotations

import json
import os
import sys

import torch

from . import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _peak_gbs() -> float:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"])
    return 6800.0


def run(name: str, reps: int, flush: bool, peak: float, fl: torch.Tensor) -> None:
    sys.path.insert(0, ROOT)
    import workloads as W
    dev = torch.device("cuda")
    shape = {**W.SHAPES, **W.PROFILE_SHAPES}[name]
    cfg = B.config(shape)
    sz = B.moe_query_sizes(cfg)
    T, H, E, k, S = shape.T, shape.H, shape.E, shape.k, shape.n_shared
    G, R = E + S, sz.rows_max
    inp = W.make_inputs(shape, seed=0, device="cuda", weights=False)
    x, Wr, bias, dY = inp["x"], inp["W_r"], inp["bias"], inp["dY"]
    g = torch.Generator(device=dev).manual_seed(0)
    sc = torch.zeros(sz.scratch_bytes, dtype=torch.uint8, device=dev)

    def i32(n):
        return torch.empty(n, dtype=torch.int32, device=dev)

    logits = torch.empty(T, E, device=dev)
    idx, w = i32(T * k), torch.empty(T * k, device=dev)
    counts, offsets = i32(G), i32(G + 1)
    row_of, token_of = i32(T * k), i32(R)
    sel_off, sel_tok = i32(E + 1), i32(T * k)
    x_perm = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    y_perm = torch.randn(R, H, device=dev, generator=g).to(torch.bfloat16)
    out, dx = torch.empty_like(dY), torch.empty_like(dY)
    dO = torch.empty_like(y_perm)
    dw = torch.empty(T * k, device=dev)
    dl = torch.empty(T, E, device=dev)
    dX_perm = torch.randn(R, H, device=dev, generator=g).to(torch.bfloat16)
    dWr = torch.empty(E, H, device=dev)
    sel_cnt, p_mean, loss = i32(E), torch.empty(E, device=dev), torch.empty(1, device=dev)
    bias_out = torch.empty(E, device=dev)
    dl_aux = torch.empty(T, E, device=dev)
    stages = {
        "route": lambda: B.moe_route(cfg, x, Wr, bias, logits, idx, w, sc),
        "permute": lambda: B.moe_permute(cfg, x, idx, counts, offsets, row_of, token_of, sel_off,
                                         sel_tok, x_perm, sc),
        "unpermute": lambda: B.moe_unpermute(cfg, y_perm, row_of, w, offsets, out),
        "unpermute_bwd": lambda: B.moe_unpermute_bwd(cfg, dY, y_perm, row_of, w, counts, offsets,
                                                     dO, dw, sc),
        "route_bwd": lambda: B.moe_route_bwd(cfg, logits, idx, w, dw, dl),
        "permute_bwd": lambda: B.moe_permute_bwd(cfg, dX_perm, row_of, offsets, idx, dl, Wr, dx),
        "router_wgrad": lambda: B.moe_router_wgrad(cfg, x, sel_off, sel_tok, dl, dWr, sc),
        "route_aux": lambda: B.moe_route_aux(cfg, logits, bias, idx, 0.01, 1e-3, sel_cnt, p_mean,
                                             loss, bias_out, sc),
        "route_aux_bwd": lambda: B.moe_route_aux_bwd(cfg, x, logits, bias, Wr, sel_cnt, 0.01, 1.0,
                                                     dl_aux, dx, dWr, sc),
    }
    for f in stages.values():
        f()
    torch.cuda.synchronize()
    cnt = counts.cpu().tolist()
    A = sum(cnt[:E])
    rows = A + S * T
    P = int(offsets[G].item()) - sum(cnt)
    bf, maps = 2, T * k * 12
    nbytes = {
        "route": T * H * bf + E * H * 4 + T * E * 4 + 2 * T * k * 4,
        "permute": T * H * bf + (rows + P) * H * bf + maps,
        "unpermute": rows * H * bf + T * H * bf + maps,
        "unpermute_bwd": T * H * bf + A * H * bf + (rows + P) * H * bf + maps,
        "route_bwd": T * E * 8 + maps,
        "permute_bwd": rows * H * bf + T * H * bf + maps,
        "router_wgrad": T * H * bf + E * H * 4 + T * E * 4,
        "route_aux": T * E * 4 + T * k * 4,
        "route_aux_bwd": 2 * T * E * 4 + 3 * T * H * bf + 3 * E * H * 4,
    }
    print(f"== {name} T={T} H={H} E={E} k={k} S={S} A={A} P={P} "
          f"status={B.moe_last_device_status(sc)} cold_l2={flush}")
    for s, f in stages.items():
        ts = []
        for _ in range(reps):
            if flush:
                fl.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ts.sort()
        ms = ts[len(ts) // 2]
        gbs = nbytes[s] / (ms * 1e-3) / 1e9
        print(f"  {s:14s} {ms * 1e3:9.1f} us  {nbytes[s] / 1e6:9.1f} MB  {gbs:8.0f} GB/s  "
              f"{gbs / peak:5.2f}")


def main(argv=None) -> None:
    argv = list(sys.argv[1:] if argv is None else argv)
    reps = 20
    if "--reps" in argv:
        i = argv.index("--reps")
        reps = int(argv[i + 1])
        del argv[i:i + 2]
    flush = "--no-flush" not in argv
    names = [a for a in argv if not a.startswith("--")] or ["mixtral"]
    fl = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    peak = _peak_gbs()
    for n in names:
        run(n, reps, flush, peak, fl)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
