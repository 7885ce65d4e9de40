"""Run the whole path (predictor, forward, and optionally backward) on one workload.

    python profile_step.py --workload fwd_61k [--heads 10] [--backward] [--steps 1]
    python profile_step.py --workload merge_131k --merge [--heads 4]
    python profile_step.py --workload dsa3d_524k --dsa3d [--heads 1] [--backward]

With --merge it runs the state merge and its gradient instead: the workload's
partition count of random (O, LSE) states of its shapes, then sda_merge_states
and sda_merge_states_bwd once per step.  With --dsa3d it runs 3D deformable
sliding attention on a workload of DSA3D_WORKLOADS: sda_dsa3d_offsets from the
seeded offset-network weights, then sda_dsa3d_fwd on those offsets (Q, K, V
drawn N(0,1) on the device); with --backward also sda_dsa3d_bwd (dO drawn
N(0,1)) and sda_dsa3d_offsets_bwd on the offsets' gradient it returns.  With
--distill it runs sda_predictor_grad (the predictor's training signal) on the
workload's seeded Q, K, Wq, Wk.

A small driver for inspecting the kernels (e.g. under a profiler) on a chosen
workload: inputs come from the seeded generator, every step runs all the
calls of the path on the current stream (with a backward, the training pair:
sda_attn_fwd_train and the three phases of sda_attn_bwd_train), and the
per-call times (CUDA events) are printed as one JSON line.  The library must
be built.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="fwd_61k")
    ap.add_argument("--heads", type=int, default=0, help="override the workload's head count")
    ap.add_argument("--backward", action="store_true", help="also run the backward (always on for training workloads)")
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--merge", action="store_true", help="run the state merge and its gradient instead")
    ap.add_argument("--dsa3d", action="store_true", help="run 3D deformable sliding attention instead")
    ap.add_argument("--distill", action="store_true", help="run the predictor's training signal instead")
    args = ap.parse_args()

    import torch

    from dynamic_block_sparse_rank_gb300 import inputs, sda

    if args.dsa3d:
        return dsa3d_steps(args)
    wl = inputs.WORKLOADS[args.workload]
    if args.heads:
        wl = wl.with_(heads=args.heads)
    if args.merge:
        return merge_steps(wl, args)
    if args.distill:
        return distill_steps(wl, args)
    backward = args.backward or wl.backward
    names = ("Q", "K", "V", "Wq", "Wk") + (("dO",) if backward else ())
    x = inputs.generate(wl, names=names)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    d = {n: torch.from_numpy(a).to(tdt).cuda() for n, a in x.items()}
    p = sda.problem_from_workload(wl)
    nb, k = sda.sda_num_blocks(p)
    idx = torch.empty((wl.B, wl.heads, nb, k), dtype=torch.int32, device="cuda")
    O = torch.empty_like(d["Q"])
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    ws_p = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICT), dtype=torch.uint8, device="cuda")
    if backward:  # the training pair, as bench.py runs it
        grads = [torch.empty(d["Q"].shape, dtype=torch.float32, device="cuda") for _ in range(3)]
        ws_t = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_TRAIN), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    names_t = ["predict", "fwd"] + (["bwd_prepare", "bwd_dq", "bwd_dkdv"] if backward else [])

    def step(ev):
        ev[0].record(st)
        sda.sda_predict_blocks(p, d["Q"], d["K"], d["Wq"], d["Wk"], idx, None, ws_p, st)
        ev[1].record(st)
        if backward:
            sda.sda_attn_fwd_train(p, d["Q"], d["K"], d["V"], idx, O, LSE, ws_t, stream=st)
            ev[2].record(st)
            for i, ph in enumerate((1, 2, 4)):
                sda.sda_attn_bwd_train(p, LSE, d["dO"], idx, *grads, "f32", ws_t, phases=ph, stream=st)
                ev[3 + i].record(st)
        else:
            sda.sda_attn_fwd(p, d["Q"], d["K"], d["V"], idx, O, LSE, stream=st)
            ev[2].record(st)

    times = {n: [] for n in names_t}
    for s in range(args.warmup + args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        step(ev)
        torch.cuda.synchronize()
        if s >= args.warmup:
            for i, n in enumerate(names_t):
                times[n].append(ev[i].elapsed_time(ev[i + 1]))
    status = sda.sda_get_device_status()
    print(json.dumps({"workload": wl.name, "heads": wl.heads, "tokens": wl.N, "k": k,
                      "ms": {n: statistics.median(v) for n, v in times.items()},
                      "status": sda.status_string(status)}))
    if status != sda.SDA_OK:
        raise SystemExit(1)


def merge_steps(wl, args):
    import torch

    from dynamic_block_sparse_rank_gb300 import sda

    n = max(wl.partitions, 2)
    g = torch.Generator(device="cuda").manual_seed(0)
    shape, lshape = (wl.B, wl.N, wl.heads, wl.d), (wl.B, wl.heads, wl.N)
    Os = [torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16) for _ in range(n)]
    Ls = [torch.randn(lshape, device="cuda", generator=g) for _ in range(n)]
    dO = torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16)
    dL = torch.randn(lshape, device="cuda", generator=g)
    Oo, Lo = torch.empty_like(Os[0]), torch.empty_like(Ls[0])
    gO = [torch.empty_like(Os[0]) for _ in range(n)]
    gL = [torch.empty_like(Ls[0]) for _ in range(n)]
    st = torch.cuda.current_stream()
    times = {"merge": [], "merge_bwd": []}
    for s in range(args.warmup + args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(st)
        sda.sda_merge_states(Os, Ls, wl.B, wl.N, wl.heads, wl.d, "bf16", Oo, Lo, st)
        ev[1].record(st)
        sda.sda_merge_states_bwd(Os, Ls, dO, dL, wl.B, wl.N, wl.heads, wl.d, "bf16", gO, gL, st)
        ev[2].record(st)
        torch.cuda.synchronize()
        if s >= args.warmup:
            times["merge"].append(ev[0].elapsed_time(ev[1]))
            times["merge_bwd"].append(ev[1].elapsed_time(ev[2]))
    rows = wl.B * wl.N * wl.heads
    status = sda.sda_get_device_status()
    print(json.dumps({"workload": wl.name, "heads": wl.heads, "tokens": wl.N, "states": n,
                      "ms": {k: statistics.median(v) for k, v in times.items()},
                      "bytes": {"merge": (n + 1) * rows * (2 * wl.d + 4), "merge_bwd": (2 * n + 1) * rows * (2 * wl.d + 4)},
                      "status": sda.status_string(status)}))
    if status != sda.SDA_OK:
        raise SystemExit(1)


def distill_steps(wl, args):
    import torch

    from dynamic_block_sparse_rank_gb300 import inputs, sda

    x = inputs.generate(wl, names=("Q", "K", "Wq", "Wk"))
    d = {n: torch.from_numpy(a).to(torch.bfloat16).cuda() for n, a in x.items()}
    p = sda.problem_from_workload(wl)
    gq = torch.empty((wl.heads, wl.d, wl.rank), dtype=torch.float32, device="cuda")
    gk = torch.empty_like(gq)
    loss = torch.empty((1,), dtype=torch.float64, device="cuda")
    ws = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICTOR_GRAD), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    times = []
    for s in range(args.warmup + args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(st)
        sda.sda_predictor_grad(p, d["Q"], d["K"], d["Wq"], d["Wk"], gq, gk, loss, ws, stream=st)
        ev[1].record(st)
        torch.cuda.synchronize()
        if s >= args.warmup:
            times.append(ev[0].elapsed_time(ev[1]))
    status = sda.sda_get_device_status()
    print(json.dumps({"workload": wl.name, "heads": wl.heads, "tokens": wl.N, "ms": statistics.median(times),
                      "status": sda.status_string(status)}))
    if status != sda.SDA_OK:
        raise SystemExit(1)


def dsa3d_steps(args):
    import torch

    from dynamic_block_sparse_rank_gb300 import inputs, sda

    wl = inputs.DSA3D_WORKLOADS[args.workload]
    if args.heads:
        wl = wl.with_(heads=args.heads)
    x = inputs.generate_dsa3d(wl, names=("Wc", "bc", "Wl", "bl"))
    w = {n: torch.from_numpy(a).cuda() for n, a in x.items()}
    g = torch.Generator(device="cuda").manual_seed(0)
    shape = (wl.B, wl.N, wl.heads, wl.d)
    Q, K, V = (torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3))
    off = torch.empty((wl.B, wl.N, wl.heads, wl.S, 3), dtype=torch.float32, device="cuda")
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    p = sda.dsa3d_problem(wl.B, wl.T, wl.H, wl.W, wl.heads, wl.d, wl.kt, wl.kh, wl.kw)
    st = torch.cuda.current_stream()
    times = {"offsets": [], "attention": []}
    if args.backward:
        dO = torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16)
        dQ, dK, dV = (torch.empty(shape, dtype=torch.float32, device="cuda") for _ in range(3))
        doff = torch.empty_like(off)
        gw = [torch.empty_like(w[n]) for n in ("Wc", "bc", "Wl", "bl")]
        ws = torch.empty(sda.sda_dsa3d_offsets_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
        bws = torch.empty(sda.sda_dsa3d_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
        times.update(attention_bwd=[], offsets_bwd=[])
    for s in range(args.warmup + args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record(st)
        sda.sda_dsa3d_offsets(p, Q, w["Wc"], w["bc"], w["Wl"], w["bl"], off, st)
        ev[1].record(st)
        sda.sda_dsa3d_fwd(p, Q, K, V, off, O, LSE, st)
        ev[2].record(st)
        if args.backward:
            sda.sda_dsa3d_bwd(p, Q, K, V, off, LSE, dO, dQ, dK, dV, doff, bws, st)
            ev[3].record(st)
            sda.sda_dsa3d_offsets_bwd(p, Q, w["Wc"], w["bc"], w["Wl"], doff, dQ, *gw, ws, st)
            ev[4].record(st)
        torch.cuda.synchronize()
        if s >= args.warmup:
            times["offsets"].append(ev[0].elapsed_time(ev[1]))
            times["attention"].append(ev[1].elapsed_time(ev[2]))
            if args.backward:
                times["attention_bwd"].append(ev[2].elapsed_time(ev[3]))
                times["offsets_bwd"].append(ev[3].elapsed_time(ev[4]))
    status = sda.sda_get_device_status()
    print(json.dumps({"workload": wl.name, "heads": wl.heads, "tokens": wl.N, "window": [wl.kt, wl.kh, wl.kw],
                      "ms": {k: statistics.median(v) for k, v in times.items()},
                      "status": sda.status_string(status)}))
    if status != sda.SDA_OK:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
