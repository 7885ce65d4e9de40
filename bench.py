#!/usr/bin/env python3
"""Benchmark of one training step of dynamic block-sparse attention on GB300.

A step is the whole path on the 524,288-token workload (batch 1, 8 heads,
grid 32 x 128 x 128, d = 128, bf16, 2x8x8 tiles, rank 32, keep 0.05 = 204 of
4,096 key blocks per query block): low-rank predictor + top-k, block-sparse
forward, backward (prepare, dQ, dK/dV; fp32 gradients).  Inputs are the
seeded synthetic generator's arrays, resident in HBM before timing; each
input tensor (1.07 GB) is larger than L2, so no flush is needed.

The reported metric is sparse-attention TFLOP/s: the algorithmic forward +
backward FLOPs of the kept blocks (4 d and 10 d per kept (query, key) token
pair) divided by the step time, which also contains the predictor.  The same
line carries tokens/s, per-phase times, the roofline of the dominant kernel,
the end-to-end figure through host buffers, clocks, and the CPU oracle timed
on a bounded sample (rank 0, one GPU only).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

With N > 1 (torchrun), every rank runs an independent replica of the step
(the path has no exchange step: query blocks, heads and batches are independent): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from dynamic_block_sparse_rank_gb300 import inputs  # noqa: E402

WORKLOAD = "train_524k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}



# Per-launch counters of the kernels that can be the dominant one, each from its own ncu capture of ONE
# kernel on a small case of the same workload (one head of the 524,288-token step, so every tensor is
# 134 MB, larger than L2), scaled to the eight-head launch by the units processed (DRAM bytes grow in
# proportion to the heads), and the tensor pipe's active fraction as ncu reports it:
#   python profile_step.py --workload train_524k --heads 1 --steps 1 --warmup 1 &&
#   ncu --set full --clock-control none -k regex:<kernel> -s 1 -c 1 -o prof_<kernel> \
#       python profile_step.py --workload train_524k --heads 1 --steps 1 --warmup 1
# (dram__bytes_read.sum + dram__bytes_write.sum; sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active);
# the three attention kernels' entries come from those metrics alone, on the same command:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active
#       --clock-control none -k "regex:fwd_tc_kernel|dqx_kernel|dkdv_kernel" -s 3 -c 3 python profile_step.py ...
# An entry goes back to None whenever its kernel changes, until it is captured again.
NCU_COUNTERS = {
    "score_kernel": {"dram_bytes": 8 * (0.0686e9 + 0.0051e9), "tensor_active": 0.586},
    "fwd_tc_kernel": {"dram_bytes": 8 * (8.507e9 + 0.574e9), "tensor_active": 0.628},
    "dqx_kernel": {"dram_bytes": 8 * (6.909e9 + 0.260e9), "tensor_active": 0.774},
    "dkdv_kernel": {"dram_bytes": 8 * (15.402e9 + 0.517e9), "tensor_active": 0.678},
}

GAP_REL = 1e-3  # selection rows whose k-th / (k+1)-th score gap is below this (relative) are near-ties


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU oracle sample")
    return ap.parse_args()


def dsa3d_fractions(dsa, hbm_peak, sm_mhz):
    """Fractions for the 3D-DSA kernels: of the measured HBM peak, and of the FP32 peak derived from the unit
    counts (152 SMs x 128 FP32 lanes x 2 FLOP per FMA) at the clock sampled during the run."""
    fp32_peak = 152 * 128 * 2 * (sm_mhz or 1900.0) * 1e6 / 1e12
    for k in ("offsets", "attention", "attention_bwd", "offsets_bwd"):
        dsa[k]["frac_of_hbm_peak"] = dsa[k]["gbs"] / hbm_peak
        dsa[k]["frac_of_fp32_peak"] = dsa[k]["tflops"] / fp32_peak
    dsa["fp32_peak_tflops"] = fp32_peak
    return dsa


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- work counting
def block_sizes(wl) -> np.ndarray:
    nT, nH, nW = wl.grid
    it, ih, iw = np.meshgrid(np.arange(nT), np.arange(nH), np.arange(nW), indexing="ij")
    st = np.minimum(wl.bt, wl.T - it * wl.bt)
    sh = np.minimum(wl.bh, wl.H - ih * wl.bh)
    sw = np.minimum(wl.bw, wl.W - iw * wl.bw)
    return (st * sh * sw).reshape(-1).astype(np.int64)


def kept_pairs(wl, idx: np.ndarray) -> int:
    """Sum over (b, h, I) of |I| * sum_{J kept} |J|: the (query, key) token pairs attended."""
    sz = block_sizes(wl)
    per_row = sz[idx.astype(np.int64)].sum(axis=-1)  # [B, Hh, nb]
    return int((per_row * sz[None, None, :]).sum())


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest value of x over all ranks (the slowest replica sets the step time)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_replica: float, ms: float) -> float:
    """Aggregate throughput of `world` replicas that each do `flops_per_replica` in `ms`."""
    return world * flops_per_replica / (ms / 1e3) / 1e12


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        loaded = [s for s in sm if s > 0.5 * (max(mx) if mx else 1)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


# ----------------------------------------------------------------------------- CPU oracle sample
_HEAD0 = {}


def _head0_inputs(wl):
    """Head 0 of the workload's inputs, generated once per process (not timed)."""
    if wl.name not in _HEAD0:
        _HEAD0[wl.name] = inputs.generate(wl, names=("Q", "K", "V", "dO", "Wq", "Wk"), heads=[0])
    return _HEAD0[wl.name]


def selection_outcome(gpu_row, scores, k) -> str:
    """The gap rule for one query block: 'exact' when the GPU's kept blocks equal the oracle's top k and the
    oracle's k-th / (k+1)-th score gap exceeds GAP_REL (relative); 'near_tie' / 'near_tie_differs' when the
    gap is smaller and every GPU-kept block scores within GAP_REL of the (k+1)-th; otherwise 'fail'."""
    nb = scores.shape[0]
    order = np.lexsort((np.arange(nb), -scores))
    want = np.sort(order[:k])
    got = np.asarray(gpu_row)
    if k == nb:
        return "exact" if np.array_equal(got, want) else "fail"
    sk, sk1 = scores[order[k - 1]], scores[order[k]]
    big = max(abs(sk), abs(sk1), 1e-30)
    if (sk - sk1) / big > GAP_REL:
        return "exact" if np.array_equal(got, want) else "fail"
    ok = (len(set(got.tolist())) == k and np.all(got >= 0) and np.all(got < nb)
          and np.all(scores[got] >= sk1 - GAP_REL * big))
    if not ok:
        return "fail"
    return "near_tie" if np.array_equal(got, want) else "near_tie_differs"


def cpu_oracle_sample(wl, seconds: float, gpu_idx_head0=None) -> dict:
    """Time the oracle (as it stands) on query blocks of head 0 until `seconds` of work are done.  With the
    GPU's block map of head 0 ([n_b, k]), the oracle's predictor rows of the sampled query blocks also grade
    the GPU's selection of those rows (near-ties counted)."""
    import oracle as orc

    cores = len(os.sched_getaffinity(0))
    x = _head0_inputs(wl)
    geom = orc.Geometry(wl.T, wl.H, wl.W, wl.bt, wl.bh, wl.bw)
    sz = block_sizes(wl)
    rng = np.random.default_rng(0)
    order = rng.permutation(geom.n_blocks)
    t0 = time.perf_counter()
    flops = 0.0
    done = []
    outcomes = {"rows": 0, "exact": 0, "near_tie": 0, "near_tie_differs": 0, "fail": 0}
    for I in order:
        I = int(I)
        idx, sc = orc.predict_blocks(x["Q"], x["K"], x["Wq"], x["Wk"], geom, wl.keep, wl.dtype, query_blocks=[I])
        if gpu_idx_head0 is not None:
            outcomes["rows"] += 1
            outcomes[selection_outcome(gpu_idx_head0[I], sc[0, 0, 0], idx.shape[-1])] += 1
        orc.attn_fwd(x["Q"], x["K"], x["V"], idx, geom, query_blocks=[I])
        orc.attn_bwd(x["Q"], x["K"], x["V"], x["dO"], idx, geom, query_blocks=[I])
        flops += 14.0 * wl.d * sz[I] * sz[idx[0, 0, 0]].sum()
        done.append(I)
        if time.perf_counter() - t0 > seconds and len(done) >= 2:
            break
    dt = time.perf_counter() - t0
    return {"tflops": flops / dt / 1e12, "seconds": dt, "cores": cores, "cpu_count": os.cpu_count(),
            "query_blocks": len(done), "selection": outcomes if gpu_idx_head0 is not None else None,
            "sample": f"{len(done)} random query blocks of head 0 of {wl.name}: oracle predictor row "
                      f"(scores against all {geom.n_blocks} key blocks) + forward + backward of their kept "
                      f"blocks, fp64 NumPy"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, wl):
    """The oracle on the host cores, each step a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = max(1.0, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, per_step)
    res = [cpu_oracle_sample(wl, per_step) for _ in range(args.steps)]
    tfl = statistics.median(r["tflops"] for r in res)
    tokens = wl.B * wl.N
    line = {"impl": "reference", "metric": "sparse attn fwd+bwd TFLOP/s (step incl. predictor), 524,288 tokens",
            "value": tfl, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Fourier-field Q/K + Gaussian V, dO)",
            "config": {"workload": wl.name, "tokens": tokens, "grid": [wl.T, wl.H, wl.W], "heads": wl.heads,
                       "head_dim": wl.d, "tile": [wl.bt, wl.bh, wl.bw], "rank": wl.rank, "keep": wl.keep,
                       "k": wl.k, "sample": res[0]["sample"]},
            "cpu_baseline": {"value": tfl, "unit": "TFLOP/s", "cores": res[0]["cores"], "kind": "oracle",
                             "sample": res[0]["sample"]},
            "e2e": {"value": tfl, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- native arm
def main():
    args = parse()
    wl = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
        return

    import torch

    from dynamic_block_sparse_rank_gb300 import build, sda

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if not os.path.exists(sda.LIB_PATH):
        build.build()
    sda.lib()

    # ---- inputs (host generation, then resident in HBM)
    t_gen = time.perf_counter()
    x = inputs.generate(wl, names=("Q", "K", "V", "dO", "Wq", "Wk"))
    t_gen = time.perf_counter() - t_gen
    dev = torch.device("cuda", local)
    host_bf16 = {n: torch.from_numpy(x[n]).to(torch.bfloat16) for n in ("Q", "K", "V", "dO", "Wq", "Wk")}
    del x
    d_in = {n: t.to(dev) for n, t in host_bf16.items()}
    Q, K, V, dO, Wq, Wk = (d_in[n] for n in ("Q", "K", "V", "dO", "Wq", "Wk"))
    p = sda.problem_from_workload(wl)
    nb, k = sda.sda_num_blocks(p)
    idx = torch.empty((wl.B, wl.heads, nb, k), dtype=torch.int32, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device=dev)
    dQ, dK, dV = (torch.empty(Q.shape, dtype=torch.float32, device=dev) for _ in range(3))
    ws_p = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICT), dtype=torch.uint8, device=dev)
    ws_t = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_TRAIN), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    main_set = dict(Q=Q, K=K, V=V, dO=dO, Wq=Wq, Wk=Wk, dQ=dQ, dK=dK, dV=dV)

    def step(ev=None, b=None, gate=None):
        # gate(name), when given, runs before the predictor ("predict"), the forward ("fwd") and the
        # backward ("bwd"), and once dQ is final ("dq"): the end-to-end loop waits there for that
        # phase's inputs and starts dQ's copy to the host under the dK/dV phase.
        b = main_set if b is None else b
        if ev is not None:
            ev[0].record(stream)
        if gate:
            gate("predict")
        sda.sda_predict_blocks(p, b["Q"], b["K"], b["Wq"], b["Wk"], idx, None, ws_p, stream)
        if ev is not None:
            ev[1].record(stream)
        if gate:
            gate("fwd")
        sda.sda_attn_fwd_train(p, b["Q"], b["K"], b["V"], idx, O, LSE, ws_t, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        if gate:
            gate("bwd")
        for i, ph in enumerate((1, 2, 4)):  # prepare, dQ, dK/dV: one call each so every phase is timed
            sda.sda_attn_bwd_train(p, LSE, b["dO"], idx, b["dQ"], b["dK"], b["dV"], "f32", ws_t, phases=ph,
                                   stream=stream)
            if ev is not None:
                ev[3 + i].record(stream)
            if gate and ph == 2:
                gate("dq")

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if sda.sda_get_device_status(stream.cuda_stream) != sda.SDA_OK:
        raise RuntimeError("device status not OK after warm-up")
    idx_host = idx.cpu().numpy()
    pairs = kept_pairs(wl, idx_host)
    f_fwd = 4.0 * wl.d * pairs
    f_bwd = 10.0 * wl.d * pairs
    f_dkdv = 8.0 * wl.d * pairs
    f_dq = 2.0 * wl.d * pairs

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = sda.sda_kernel_launch_count()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for s in range(args.steps):
            step(evs[s])
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = sda.sda_kernel_launch_count() - launches0
    ms = max_over_ranks(start.elapsed_time(end) / args.steps, dist, dev)
    phase_names = ["predict", "fwd", "bwd_prepare", "bwd_dq", "bwd_dkdv"]
    phase_ms = {n: statistics.median(e[i].elapsed_time(e[i + 1]) for e in evs) for i, n in enumerate(phase_names)}
    status = sda.sda_get_device_status(stream.cuda_stream)

    # ---- end to end through host buffers (pinned), copies inside the timed region.
    # Every step copies its inputs host->device and its gradients device->host.  The
    # copies run on two copy streams against two sets of device buffers, so step i+1's
    # inputs arrive and step i-1's gradients leave while step i computes.  Each phase waits
    # only for its own inputs (the predictor for Q, K, Wq, Wk; the forward for V; the
    # backward for dO), and dQ leaves while dK, dV are computed, so the first step's wait
    # and the last step's tail are one part of the copies, not all of them.
    e2e = None
    if not args.no_e2e:
        pin = {n: t.pin_memory() for n, t in host_bf16.items()}
        out_host = [torch.empty(dQ.shape, dtype=torch.float32).pin_memory() for _ in range(3)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in out_host)
        sets = [dict(d_in, dQ=dQ, dK=dK, dV=dV),
                dict({n: torch.empty_like(t) for n, t in d_in.items()},
                     **{g: torch.empty_like(dQ) for g in ("dQ", "dK", "dV")})]
        s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

        groups = {"predict": ("Q", "K", "Wq", "Wk"), "fwd": ("V",), "bwd": ("dO",)}

        def run_e2e(nsteps):
            h2d_done = [{g: ev() for g in groups} for _ in range(nsteps)]
            dq_done = [ev() for _ in range(nsteps)]
            comp_done = [ev() for _ in range(nsteps)]
            d2h_done = [ev() for _ in range(nsteps)]

            def issue_h2d(i):
                b = sets[i % 2]
                if i >= 2:
                    s_h2d.wait_event(comp_done[i - 2])  # step i-2 no longer reads this set's inputs
                with torch.cuda.stream(s_h2d):
                    for g, names in groups.items():
                        for n in names:
                            b[n].copy_(pin[n], non_blocking=True)
                        h2d_done[i][g].record(s_h2d)

            t0 = ev()
            t0.record(s_h2d)
            issue_h2d(0)
            for i in range(nsteps):
                b = sets[i % 2]
                if i + 1 < nsteps:
                    issue_h2d(i + 1)
                if i >= 2:
                    stream.wait_event(d2h_done[i - 2])  # step i-2's gradients have left this set

                def gate(name, i=i, b=b):
                    if name in groups:
                        stream.wait_event(h2d_done[i][name])
                        return
                    dq_done[i].record(stream)  # dQ is final: it leaves while dK, dV are computed
                    s_d2h.wait_event(dq_done[i])
                    with torch.cuda.stream(s_d2h):
                        out_host[0].copy_(b["dQ"], non_blocking=True)

                step(None, b, gate)
                comp_done[i].record(stream)
                s_d2h.wait_event(comp_done[i])
                with torch.cuda.stream(s_d2h):
                    for h, g in zip(out_host[1:], (b["dK"], b["dV"])):
                        h.copy_(g, non_blocking=True)
                d2h_done[i].record(s_d2h)
            stream.wait_event(d2h_done[nsteps - 1])
            t1 = ev()
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)

        run_e2e(2)
        # one instrumented pass: the copies alone
        c = [ev() for _ in range(4)]
        c[0].record(stream)
        for n, t in pin.items():
            d_in[n].copy_(t, non_blocking=True)
        c[1].record(stream)
        c[2].record(stream)
        for h, g in zip(out_host, (dQ, dK, dV)):
            h.copy_(g, non_blocking=True)
        c[3].record(stream)
        torch.cuda.synchronize()
        h2d_ms, d2h_ms = c[0].elapsed_time(c[1]), c[2].elapsed_time(c[3])
        barrier()
        ms_e2e = run_e2e(args.steps) / args.steps
        barrier()
        ms_e2e = max_over_ranks(ms_e2e, dist, dev)
        e2e = {"value": whole_job_tflops(world, f_fwd + f_bwd, ms_e2e), "unit": "TFLOP/s",
               "ms_per_step": ms_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "h2d_ms": h2d_ms, "d2h_ms": d2h_ms, "copies": "two copy streams, double-buffered device sets, each phase gated on its own inputs",
               "tokens_per_s": world * wl.B * wl.N / (ms_e2e / 1e3)}
        del sets

    # ---- merge of partial states on the 4-partition workload's shapes (HBM-bound kernel)
    merge = None
    if rank == 0:
        mw = inputs.WORKLOADS["merge_131k"]
        n_st = mw.partitions
        g = torch.Generator(device=dev).manual_seed(0)
        Os = [torch.randn((1, mw.N, mw.heads, mw.d), device=dev, generator=g).to(torch.bfloat16) for _ in range(n_st)]
        Ls = [torch.randn((1, mw.heads, mw.N), device=dev, generator=g) for _ in range(n_st)]
        Oo, Lo = torch.empty_like(Os[0]), torch.empty_like(Ls[0])
        for _ in range(3):
            sda.sda_merge_states(Os, Ls, 1, mw.N, mw.heads, mw.d, "bf16", Oo, Lo, stream)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        m0.record(stream)
        for _ in range(reps):
            sda.sda_merge_states(Os, Ls, 1, mw.N, mw.heads, mw.d, "bf16", Oo, Lo, stream)
        m1.record(stream)
        torch.cuda.synchronize()
        mms = m0.elapsed_time(m1) / reps
        rows = mw.N * mw.heads
        mbytes = (n_st + 1) * rows * (2 * mw.d + 4)
        merge = {"workload": mw.name, "states": n_st, "ms": mms, "bytes": mbytes, "gbs": mbytes / (mms / 1e3) / 1e9}
        del Oo, Lo
        # its gradient: reads the states, dO and dLSE, writes dO_p and dLSE_p for every state
        dO = torch.randn((1, mw.N, mw.heads, mw.d), device=dev, generator=g).to(torch.bfloat16)
        dL = torch.randn((1, mw.heads, mw.N), device=dev, generator=g)
        gO = [torch.empty_like(Os[0]) for _ in range(n_st)]
        gL = [torch.empty_like(Ls[0]) for _ in range(n_st)]
        for _ in range(3):
            sda.sda_merge_states_bwd(Os, Ls, dO, dL, 1, mw.N, mw.heads, mw.d, "bf16", gO, gL, stream)
        m0.record(stream)
        for _ in range(reps):
            sda.sda_merge_states_bwd(Os, Ls, dO, dL, 1, mw.N, mw.heads, mw.d, "bf16", gO, gL, stream)
        m1.record(stream)
        torch.cuda.synchronize()
        bms = m0.elapsed_time(m1) / reps
        bbytes = (2 * n_st + 1) * rows * (2 * mw.d + 4)
        merge["bwd"] = {"ms": bms, "bytes": bbytes, "gbs": bbytes / (bms / 1e3) / 1e9}
        del Os, Ls, dO, dL, gO, gL

    # ---- the predictor's training signal on the 61K-token shapes (distillation gradient of Wq, Wk)
    pgrad = None
    if rank == 0:
        pw = inputs.WORKLOADS["fwd_61k"]
        xp = inputs.generate(pw, names=("Q", "K", "Wq", "Wk"))
        tp = {n: torch.from_numpy(xp[n]).to(torch.bfloat16).to(dev) for n in ("Q", "K", "Wq", "Wk")}
        del xp
        pp = sda.problem_from_workload(pw)
        gq = torch.empty((pw.heads, pw.d, pw.rank), dtype=torch.float32, device=dev)
        gk = torch.empty_like(gq)
        gl = torch.empty((1,), dtype=torch.float64, device=dev)
        gws = torch.empty(sda.sda_workspace_size(pp, sda.SDA_OP_PREDICTOR_GRAD), dtype=torch.uint8, device=dev)
        for _ in range(2):
            sda.sda_predictor_grad(pp, tp["Q"], tp["K"], tp["Wq"], tp["Wk"], gq, gk, gl, gws, stream=stream)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        g0.record(stream)
        for _ in range(reps):
            sda.sda_predictor_grad(pp, tp["Q"], tp["K"], tp["Wq"], tp["Wk"], gq, gk, gl, gws, stream=stream)
        g1.record(stream)
        torch.cuda.synchronize()
        gms = g0.elapsed_time(g1) / reps
        gflops = 2.0 * (pw.rank + pw.d) * pw.B * pw.heads * float(pw.N) ** 2  # both products, every token pair
        pgrad = {"workload": pw.name, "ms": gms, "flops": gflops, "tflops": gflops / (gms / 1e3) / 1e12}
        del tp, gws

    # ---- 3D deformable sliding attention on the same 524K-token grid: offsets, then the window attention
    dsa = None
    if rank == 0:
        dw = inputs.DSA3D_WORKLOADS["dsa3d_524k"]
        xd = inputs.generate_dsa3d(dw, names=("Wc", "bc", "Wl", "bl"))
        td = {n: torch.from_numpy(xd[n]).to(dev) for n in xd}
        g = torch.Generator(device=dev).manual_seed(1)
        dshape = (dw.B, dw.N, dw.heads, dw.d)
        # seeded device draws of the activations (N(0,1), bf16): the offsets come from the network
        aQ, aK, aV = (torch.randn(dshape, device=dev, generator=g).to(torch.bfloat16) for _ in range(3))
        doff = torch.empty((dw.B, dw.N, dw.heads, dw.S, 3), dtype=torch.float32, device=dev)
        aO = torch.empty_like(aQ)
        aL = torch.empty((dw.B, dw.heads, dw.N), dtype=torch.float32, device=dev)
        dp = sda.dsa3d_problem(dw.B, dw.T, dw.H, dw.W, dw.heads, dw.d, dw.kt, dw.kh, dw.kw)
        for _ in range(2):
            sda.sda_dsa3d_offsets(dp, aQ, td["Wc"], td["bc"], td["Wl"], td["bl"], doff, stream=stream)
            sda.sda_dsa3d_fwd(dp, aQ, aK, aV, doff, aO, aL, stream=stream)
        de = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        reps = 3
        t_off = t_att = 0.0
        for _ in range(reps):
            de[0].record(stream)
            sda.sda_dsa3d_offsets(dp, aQ, td["Wc"], td["bc"], td["Wl"], td["bl"], doff, stream=stream)
            de[1].record(stream)
            sda.sda_dsa3d_fwd(dp, aQ, aK, aV, doff, aO, aL, stream=stream)
            de[2].record(stream)
            torch.cuda.synchronize()
            t_off += de[0].elapsed_time(de[1]) / reps
            t_att += de[1].elapsed_time(de[2]) / reps
        # the backward of both: attention (dQ, dK, dV, d_offsets), then the offset network (dQ added to, the
        # weight gradients)
        adO = torch.randn(dshape, device=dev, generator=g).to(torch.bfloat16)
        gQ, gK, gV = (torch.empty(dshape, dtype=torch.float32, device=dev) for _ in range(3))
        goff = torch.empty_like(doff)
        gw = [torch.empty_like(td[n]) for n in ("Wc", "bc", "Wl", "bl")]
        gws = torch.empty(sda.sda_dsa3d_offsets_bwd_workspace_size(dp), dtype=torch.uint8, device=dev)
        bws = torch.empty(sda.sda_dsa3d_bwd_workspace_size(dp), dtype=torch.uint8, device=dev)
        for _ in range(2):
            sda.sda_dsa3d_bwd(dp, aQ, aK, aV, doff, aL, adO, gQ, gK, gV, goff, bws, stream=stream)
            sda.sda_dsa3d_offsets_bwd(dp, aQ, td["Wc"], td["bc"], td["Wl"], goff, gQ, *gw, gws, stream=stream)
        t_abwd = t_obwd = 0.0
        for _ in range(reps):
            de[0].record(stream)
            sda.sda_dsa3d_bwd(dp, aQ, aK, aV, doff, aL, adO, gQ, gK, gV, goff, bws, stream=stream)
            de[1].record(stream)
            sda.sda_dsa3d_offsets_bwd(dp, aQ, td["Wc"], td["bc"], td["Wl"], goff, gQ, *gw, gws, stream=stream)
            de[2].record(stream)
            torch.cuda.synchronize()
            t_abwd += de[0].elapsed_time(de[1]) / reps
            t_obwd += de[1].elapsed_time(de[2]) / reps
        th = float(dw.B * dw.N * dw.heads)  # (token, head) units
        row = 2.0 * dw.d  # bytes of one bf16 row
        # algorithmic work per (token, head): offsets 2 * 27 d + 2 d 3S FLOP, reading the Q row and writing
        # 3S fp32; attention 8 corners x (q.k and the weighted v) = 32 d FLOP per window point, reading the
        # Q, K, V rows once (ideal reuse) and the offsets, writing the O row and the LSE
        f_off, b_off = th * (2.0 * 27 * dw.d + 2.0 * dw.d * 3 * dw.S), th * (row + 12.0 * dw.S)
        f_att, b_att = th * 32.0 * dw.d * dw.S, th * (3 * row + 12.0 * dw.S + row + 4.0)
        # attention backward per window point: 8 corners x (q.K[m], dO.V[m], the dq term, the dK and dV rows)
        # = 80 d FLOP, reading the Q, K, V, dO rows, the offsets and LSE, writing dQ, dK, dV (fp32) and the
        # offsets' gradient; offset network backward: the convolution twice forward-sized (Y recomputed, the
        # transposed one) plus dWc, and the two d x 3S products (dY, dWl), reading the Q row and the offsets'
        # gradient, updating the fp32 dQ row
        f_abwd = th * 80.0 * dw.d * dw.S
        b_abwd = th * (4 * row + 24.0 * dw.S + 4.0 + 12.0 * dw.d)
        f_obwd = th * (3 * 2.0 * 27 * dw.d + 2 * 2.0 * dw.d * 3 * dw.S)
        b_obwd = th * (row + 12.0 * dw.S + 8.0 * dw.d)
        t_all = t_off + t_att + t_abwd + t_obwd
        dsa = {"workload": dw.name, "tokens": dw.N, "heads": dw.heads, "window": [dw.kt, dw.kh, dw.kw],
               "ms": {"offsets": t_off, "attention": t_att, "total": t_off + t_att, "attention_bwd": t_abwd,
                      "offsets_bwd": t_obwd, "fwd_bwd_total": t_all},
               "tokens_per_s": dw.B * dw.N / ((t_off + t_att) / 1e3),
               "tokens_per_s_fwd_bwd": dw.B * dw.N / (t_all / 1e3),
               "offsets": {"tflops": f_off / (t_off / 1e3) / 1e12, "gbs": b_off / (t_off / 1e3) / 1e9},
               "attention": {"tflops": f_att / (t_att / 1e3) / 1e12, "gbs": b_att / (t_att / 1e3) / 1e9},
               "attention_bwd": {"tflops": f_abwd / (t_abwd / 1e3) / 1e12, "gbs": b_abwd / (t_abwd / 1e3) / 1e9},
               "offsets_bwd": {"tflops": f_obwd / (t_obwd / 1e3) / 1e12, "gbs": b_obwd / (t_obwd / 1e3) / 1e9},
               "status": sda.status_string(sda.sda_get_device_status(stream))}
        del aQ, aK, aV, doff, aO, aL, td, adO, gQ, gK, gV, goff, gw, gws, bws

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    pk, pk_src = peaks()
    tc_peak = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm_peak = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # algorithmic FLOPs per launch: predictor 2 r per token pair (all pairs of a head), forward 4 d and
    # dK/dV 8 d per kept pair, dQ 2 d per kept pair (its S and dP products are recomputation)
    f_pred = 2.0 * wl.rank * wl.B * wl.heads * float(wl.N) ** 2
    kern = {"predict (score_kernel; phase incl. 2 proj_kernel)": (phase_ms["predict"], f_pred),
            "attn_fwd_train (fwd_tc_kernel; phase incl. 3 fp16 copies)": (phase_ms["fwd"], f_fwd),
            "attn_bwd_train dK/dV (dkdv_kernel)": (phase_ms["bwd_dkdv"], f_dkdv),
            "attn_bwd_train dQ (dqx_kernel)": (phase_ms["bwd_dq"], f_dq)}
    dom = max(kern, key=lambda n: kern[n][0])
    dom_ms, dom_flops = kern[dom]
    counters = next((v for key, v in NCU_COUNTERS.items() if key in dom and v), None)
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    burst_peak = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    clocks = clk.summary()
    # the sustained peak was taken at the clock its own loop ran at (power-capped); this step's kernels ran at
    # the median clock sampled above, so the fraction is also given against that peak scaled to this clock
    peak_mhz = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    run_mhz = clocks.get("sm_mhz")
    scaled = tc_peak * run_mhz / peak_mhz if peak_mhz and run_mhz else None
    if merge:
        merge["frac_of_hbm_peak"] = merge["gbs"] / hbm_peak
        merge["bwd"]["frac_of_hbm_peak"] = merge["bwd"]["gbs"] / hbm_peak
    attn_ms = phase_ms["fwd"] + phase_ms["bwd_prepare"] + phase_ms["bwd_dq"] + phase_ms["bwd_dkdv"]
    cpu = None
    selection = None
    if not args.no_cpu_baseline and world == 1:
        c = cpu_oracle_sample(wl, args.cpu_seconds, gpu_idx_head0=idx_host[0, 0])
        cpu = {"value": c["tflops"], "unit": "TFLOP/s", "cores": c["cores"], "kind": "oracle", "sample": c["sample"],
               "seconds": c["seconds"]}
        selection = dict(c["selection"], rule=f"gap rule, {GAP_REL:g} relative; rows = the oracle sample's "
                                              f"query blocks (head 0)")
    line = {
        "metric": "sparse attn fwd+bwd TFLOP/s (step incl. predictor), 524,288 tokens",
        "value": whole_job_tflops(world, f_fwd + f_bwd, ms),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Fourier-field Q/K + Gaussian V, dO; random-init Wq, Wk)",
        "config": {"workload": wl.name, "tokens": wl.B * wl.N, "grid": [wl.T, wl.H, wl.W], "heads": wl.heads,
                   "head_dim": wl.d, "tile": [wl.bt, wl.bh, wl.bw], "rank": wl.rank, "keep": wl.keep, "k": k,
                   "grad_dtype": "f32", "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (1.07 GB per tensor), no flush"},
        "tokens_per_s": world * wl.B * wl.N / (ms / 1e3),
        "attn_only": {"ms": attn_ms, "tflops": (f_fwd + f_bwd) / (attn_ms / 1e3) / 1e12,
                      "frac_of_peak": (f_fwd + f_bwd) / (attn_ms / 1e3) / 1e12 / tc_peak},
        "phase_ms": phase_ms,
        "flops": {"fwd": f_fwd, "bwd": f_bwd, "kept_pairs": pairs},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak,
                     "traffic": counters["dram_bytes"] if counters else None,
                     "traffic_unit": "DRAM bytes per launch (ncu, one head scaled to eight)",
                     "peak_source": f"{pk_src} bf16_tflops_sustained (fp16 and bf16 share the dense rate)",
                     "peak_burst": burst_peak, "frac_vs_burst": achieved / burst_peak,
                     "peak_sm_mhz": peak_mhz, "run_sm_mhz": run_mhz,
                     "frac_vs_sustained_at_run_clock": achieved / scaled if scaled else None,
                     "ncu_tensor_pipe_active": counters["tensor_active"] if counters else None},
        "selection": selection,
        "kernels": {n: {"ms": t, "tflops": f / (t / 1e3) / 1e12, "frac": f / (t / 1e3) / 1e12 / tc_peak}
                    for n, (t, f) in kern.items()},
        "merge": merge,
        "predictor_grad": dict(pgrad, frac_of_peak=pgrad["tflops"] / tc_peak) if pgrad else None,
        "dsa3d": dsa3d_fractions(dsa, hbm_peak, clocks.get("sm_mhz")) if dsa else None,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": launches,
        "device_status": sda.status_string(status),
        "input_generation_s": t_gen,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
