"""GPU vs oracle parity at the five workloads' full sizes, in the launch configuration bench.py times.

The CUDA path runs the whole problem; the fp64 oracle recomputes sampled outputs, a batch of query blocks
(or key blocks) at a time.  Where a GPU call needs a full block map but the oracle only computes some
rows, the sampled rows come from the oracle's own predictor: for the forward the GPU map's sampled rows
are replaced by them before the call; for the backward at 524K tokens (whose key-block sums need every
row of the map) the other rows come from the seeded scattered map generator, whose rows are spread over
the grid with heavy-tailed key-block popularity like the predictor's.  So every compared GPU output
derives from oracle-selected (or seeded) blocks and no oracle input comes from the GPU.

Each test adds its figures (rows compared, selection outcome including near-ties, max-abs and relative
Frobenius error per output, oracle seconds and the sampled fraction) to the session's parity report.
"""
import time

import numpy as np
import pytest

import oracle as orc
from dynamic_block_sparse_rank_gb300 import inputs
from tests.parity_util import assert_close, check_scores, check_selection, dev, errors, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_rank_gb300 import sda as s

    s.lib()
    return s


_INPUTS = {}


def _inputs(wl, names):
    """The workload's inputs, generated once per module for every name asked so far."""
    have = _INPUTS.setdefault(wl.name, {})
    missing = tuple(n for n in names if n not in have)
    if missing:
        have.update(inputs.generate(wl, names=missing))
    return {n: have[n] for n in names}


def _geom(wl):
    return orc.Geometry(wl.T, wl.H, wl.W, wl.bt, wl.bh, wl.bw)


def _samples(wl, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    nb = wl.n_blocks
    picks = {0, nb - 1, nb // 2} | set(int(x) for x in rng.choice(nb, n, replace=False)) | set(extra)
    return sorted(picks)


def _head(x, h):
    return {k: (v[:, :, h:h + 1] if v.ndim == 4 and k not in ("Wq", "Wk") else v[h:h + 1]) for k, v in x.items()}


class _Record:
    """One workload's entry of the parity report."""

    def __init__(self, report, name, fraction_note):
        self.e = report.setdefault(name, {"outputs": {}, "selection": {}, "oracle_seconds": 0.0,
                                          "sampled": fraction_note})
        self.t = 0.0

    def oracle(self, fn, *a, **kw):
        t0 = time.perf_counter()
        out = fn(*a, **kw)
        self.e["oracle_seconds"] += time.perf_counter() - t0
        return out

    def selection(self, st):
        for k, v in st.items():
            self.e["selection"][k] = self.e["selection"].get(k, 0) + int(v)

    def close(self, got, ref, dtype, what, key):
        mx, rel = assert_close(got, ref, dtype, what)
        o = self.e["outputs"].setdefault(key, {"max_abs": 0.0, "rel_frob_max": 0.0, "values": 0})
        o["max_abs"] = max(o["max_abs"], float(mx))
        o["rel_frob_max"] = max(o["rel_frob_max"], float(rel))
        o["values"] += int(np.size(ref))


def _gpu_predict(sda, wl, Q, K, Wq, Wk, with_score=True):
    p = sda.problem_from_workload(wl)
    nb, k = sda.sda_num_blocks(p)
    idx = torch.empty((wl.B, wl.heads, nb, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.B, wl.heads, nb, nb), dtype=torch.float32, device="cuda") if with_score else None
    ws = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICT), dtype=torch.uint8, device="cuda")
    sda.sda_predict_blocks(p, Q, K, Wq, Wk, idx, sc, ws)
    torch.cuda.synchronize()
    return idx, sc


def _check_predictor_and_forward(sda, rec, wl, heads, qb):
    """Predictor rows (gap rule) and forward rows of query blocks qb on every head in `heads`."""
    x = _inputs(wl, ("Q", "K", "V", "Wq", "Wk"))
    geom = _geom(wl)
    Q, K, V, Wq, Wk = (dev(x[n], wl.dtype) for n in ("Q", "K", "V", "Wq", "Wk"))
    idx, sc = _gpu_predict(sda, wl, Q, K, Wq, Wk)
    ref_rows = {}
    for h in heads:
        xh = _head(x, h)
        ridx, rsc = rec.oracle(orc.predict_blocks, xh["Q"], xh["K"], xh["Wq"], xh["Wk"], geom, wl.keep, wl.dtype,
                               query_blocks=qb)
        st = check_selection(idx[0, h, qb].cpu().numpy(), rsc, wl.k)
        rec.selection(st)
        assert st["fail"] == 0, (h, st)
        check_scores(sc[0, h, qb].cpu().numpy().astype(np.float64), rsc)
        ref_rows[h] = ridx
        idx[0, h, qb] = torch.from_numpy(ridx[0, 0]).cuda()  # compared rows use the oracle's selection
    del sc
    p = sda.problem_from_workload(wl)
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_attn_fwd(p, Q, K, V, idx, O, LSE)
    torch.cuda.synchronize()
    rows = np.concatenate([geom.tokens(I) for I in qb])
    for h in heads:
        xh = _head(x, h)
        Or, Lr = rec.oracle(orc.attn_fwd, xh["Q"], xh["K"], xh["V"], ref_rows[h], geom, query_blocks=qb)
        rec.close(host(O[0, rows, h]), Or[0, rows, 0], wl.dtype, f"O head {h}", "O")
        rec.close(host(LSE[0, h, rows]), Lr[0, 0, rows], wl.dtype, f"LSE head {h}", "LSE")
    assert sda.sda_get_device_status() == sda.SDA_OK


def test_fwd_8k_full_oracle(sda, parity_report):
    """The 8,192-token workload in full: every head, every query block."""
    wl = inputs.WORKLOADS["fwd_8k"]
    rec = _Record(parity_report, wl.name, "all 12 heads x all 64 query blocks (fraction 1.0)")
    x = _inputs(wl, ("Q", "K", "V", "Wq", "Wk"))
    geom = _geom(wl)
    Q, K, V, Wq, Wk = (dev(x[n], wl.dtype) for n in ("Q", "K", "V", "Wq", "Wk"))
    idx, sc = _gpu_predict(sda, wl, Q, K, Wq, Wk)
    ridx, rsc = rec.oracle(orc.predict_blocks, x["Q"], x["K"], x["Wq"], x["Wk"], geom, wl.keep, wl.dtype)
    st = check_selection(idx.cpu().numpy(), rsc, wl.k)
    rec.selection(st)
    assert st["fail"] == 0, st
    check_scores(host(sc), rsc)
    p = sda.problem_from_workload(wl)
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_attn_fwd(p, Q, K, V, torch.from_numpy(ridx).cuda(), O, LSE)
    torch.cuda.synchronize()
    Or, Lr = rec.oracle(orc.attn_fwd, x["Q"], x["K"], x["V"], ridx, geom)
    rec.close(host(O), Or, "bf16", "O", "O")
    rec.close(host(LSE), Lr, "bf16", "LSE", "LSE")


def test_fwd_61k_every_head_sampled(sda, parity_report):
    """61,440 tokens: all 24 heads, 48 seeded query blocks each plus the first, middle and last."""
    wl = inputs.WORKLOADS["fwd_61k"]
    qb = _samples(wl, 48, 3)
    rec = _Record(parity_report, wl.name, f"all 24 heads x {len(qb)} of 480 query blocks "
                                          f"(fraction {len(qb) / 480:.3f})")
    _check_predictor_and_forward(sda, rec, wl, list(range(wl.heads)), qb)


def test_train_524k_predictor_and_forward_sampled(sda, parity_report):
    """524,288 tokens: 3 of 8 heads, 16 seeded query blocks each plus the first, middle and last."""
    wl = inputs.WORKLOADS["train_524k"]
    qb = _samples(wl, 16, 4)
    rec = _Record(parity_report, wl.name + " predictor+forward",
                  f"heads 0, 3, 6 x {len(qb)} of 4096 query blocks (fraction {3 * len(qb) / (8 * 4096):.4f})")
    _check_predictor_and_forward(sda, rec, wl, [0, 3, 6], qb)


def test_train_524k_backward_on_predictor_rows(sda, parity_report):
    """The training pair (forward and backward) at 524,288 tokens, as bench.py runs it (fp32 gradients).  The map: for heads 1 and 6,
    16 seeded query blocks (plus first, middle, last) keep the oracle predictor's own rows; every other
    row comes from the seeded scattered generator.  Checked: dQ of those query blocks; dK and dV of 8 key
    blocks per head, among them the key block with the shortest list of query blocks (both heads) and
    with the longest (head 1); the forward's rows; and, on every row of every head, the exact sums
    sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i."""
    wl = inputs.WORKLOADS["train_524k"]
    x = _inputs(wl, ("Q", "K", "V", "dO", "Wq", "Wk"))
    geom = _geom(wl)
    heads = [1, 6]
    qb = _samples(wl, 16, 6)
    rec = _Record(parity_report, wl.name + " backward",
                  f"heads 1, 6: dQ of {len(qb)} query blocks and dK/dV of 8 key blocks per head, on a map whose "
                  f"sampled rows are the oracle predictor's; all rows of all heads through the exact sums")
    m = inputs.scattered_block_map(wl, seed=1)
    for h in heads:
        xh = _head(x, h)
        ridx, _ = rec.oracle(orc.predict_blocks, xh["Q"], xh["K"], xh["Wq"], xh["Wk"], geom, wl.keep, wl.dtype,
                             query_blocks=qb)
        m[0, h, qb] = ridx[0, 0]
    p = sda.problem_from_workload(wl)
    Q, K, V, dO = (dev(x[n], wl.dtype) for n in ("Q", "K", "V", "dO"))
    idx = torch.from_numpy(m).cuda()
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    dQ, dK, dV = (torch.empty(Q.shape, dtype=torch.float32, device="cuda") for _ in range(3))
    ws = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_TRAIN), dtype=torch.uint8, device="cuda")
    sda.sda_attn_fwd_train(p, Q, K, V, idx, O, LSE, ws)  # the training pair, as bench.py runs it
    sda.sda_attn_bwd_train(p, LSE, dO, idx, dQ, dK, dV, "f32", ws)
    torch.cuda.synchronize()
    del ws
    assert sda.sda_get_device_status() == sda.SDA_OK
    # exact invariants over every row of every head: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    sk = dK.double().sum(dim=1)
    sv = dV.double().sum(dim=1) - dO.double().sum(dim=1)
    assert float((sk.abs() / dK.double().abs().sum(dim=1)).max()) < 1e-4
    assert float((sv.abs() / dV.double().abs().sum(dim=1)).max()) < 1e-4
    rng = np.random.default_rng(7)
    rows = np.concatenate([geom.tokens(I) for I in qb])
    lengths = {}
    for h in heads:
        xh = _head(x, h)
        mh = m[:, h:h + 1]
        fan_in = np.bincount(m[0, h].ravel(), minlength=geom.n_blocks)
        order = np.argsort(fan_in, kind="stable")
        picks = [int(order[0])]  # the shortest list
        if h == heads[0]:
            picks.append(int(order[-1]))  # the longest list
        in_oracle_rows = sorted(set(int(J) for J in m[0, h, qb].ravel()) - set(picks))
        picks += [int(J) for J in rng.choice(in_oracle_rows, 2, replace=False)]
        short_half = [int(J) for J in order[1:geom.n_blocks // 2] if int(J) not in picks]
        picks += [int(J) for J in rng.choice(short_half, 8 - len(picks), replace=False)]
        lengths[h] = sorted(int(fan_in[J]) for J in picks)
        dq_ref, dkv_ref = rec.oracle(orc.attn_bwd_blocks, xh["Q"], xh["K"], xh["V"], xh["dO"], mh, geom,
                                     query_blocks=qb, key_blocks=picks)
        for (_, _, I), ref in dq_ref.items():
            rec.close(host(dQ[0, geom.tokens(I), h]), ref, "bf16", f"dQ h{h} block {I}", "dQ")
        for (_, _, J), (rk, rv) in dkv_ref.items():
            rec.close(host(dK[0, geom.tokens(J), h]), rk, "bf16", f"dK h{h} block {J}", "dK")
            rec.close(host(dV[0, geom.tokens(J), h]), rv, "bf16", f"dV h{h} block {J}", "dV")
        Or, Lr = rec.oracle(orc.attn_fwd, xh["Q"], xh["K"], xh["V"], mh[:, :, qb], geom, query_blocks=qb)
        rec.close(host(O[0, rows, h]), Or[0, rows, 0], "bf16", f"O h{h}", "O")
        rec.close(host(LSE[0, h, rows]), Lr[0, 0, rows], "bf16", f"LSE h{h}", "LSE")
    rec.e["key_block_list_lengths"] = {str(h): v for h, v in lengths.items()}


def _tile_classes(geom):
    """Query blocks grouped by their clipped extent (t, h, w) on a non-divisible grid."""
    classes = {}
    for I in range(geom.n_blocks):
        it, ih, iw = geom.block_coords(I)
        ext = (min(geom.bt, geom.T - it * geom.bt), min(geom.bh, geom.H - ih * geom.bh),
               min(geom.bw, geom.W - iw * geom.bw))
        classes.setdefault(ext, []).append(I)
    return classes


def test_merge_131k_partition_states_and_reuse_every_head(sda, parity_report):
    """131,040 tokens on a ragged grid, 4 frame partitions, the 2 farthest reused from the previous step, the
    partition states kept in fp32 (so the merged result is rounded once): all 16 heads, each on 8 seeded query blocks plus one block of every clipped-tile class (full 2x8x8,
    1x8x8, 2x4x8, 1x4x8) and the last block of partition 0's reuse set.  Checked per head: the selection
    of both steps (gap rule), every partition state the GPU keeps (reused or fresh), the reuse merge, the
    exact merge of fresh states, and the full-range forward; the reuse merge's deviation from the exact
    merge is reported, not graded."""
    wl = inputs.WORKLOADS["merge_131k"]
    x = _inputs(wl, ("Q", "K", "V", "Qp", "Kp", "Vp", "Wq", "Wk"))
    geom = _geom(wl)
    P = wl.partitions
    bounds = orc.frame_partitions(geom, P)
    reuse = orc.reuse_mask(geom, P, wl.n_reuse)
    classes = _tile_classes(geom)
    assert len(classes) == 4, sorted(classes)
    rng = np.random.default_rng(5)
    extra = [int(rng.choice(v)) for v in classes.values()] + [int(np.flatnonzero(reuse[0])[-1])]
    qb = _samples(wl, 8, 5, extra)
    heads = list(range(wl.heads))
    rec = _Record(parity_report, wl.name, f"all 16 heads x {len(qb)} of 1144 query blocks (every clipped-tile "
                                          f"class) x 4 partition states, both steps (fraction {len(qb) / 1144:.3f})")
    p = sda.problem_from_workload(wl)
    T = {n: dev(x[n], wl.dtype) for n in ("Q", "K", "V", "Qp", "Kp", "Vp", "Wq", "Wk")}

    def gpu_map(Qn, Kn):
        idx, _ = _gpu_predict(sda, wl, T[Qn], T[Kn], T["Wq"], T["Wk"], with_score=False)
        rows = {}
        for h in heads:
            xh = _head(x, h)
            r, sc = rec.oracle(orc.predict_blocks, xh[Qn], xh[Kn], xh["Wq"], xh["Wk"], geom, wl.keep, wl.dtype,
                               query_blocks=qb)
            st = check_selection(idx[0, h, qb].cpu().numpy(), sc, wl.k)
            rec.selection(st)
            assert st["fail"] == 0, (Qn, h, st)
            idx[0, h, qb] = torch.from_numpy(r[0, 0]).cuda()
            rows[h] = r
        return idx, rows

    def new_state():  # partition states are kept in fp32 (sda_attn_fwd's out_dtype), merged in fp32
        return (torch.empty(T["Q"].shape, dtype=torch.float32, device="cuda"),
                torch.empty((1, wl.heads, wl.N), dtype=torch.float32, device="cuda"))

    idx_prev, rows_prev = gpu_map("Qp", "Kp")
    idx_now, rows_now = gpu_map("Q", "K")
    # previous step: every partition state for every query block (the reuse cache)
    states = [new_state() for _ in range(P)]
    for (b0, b1), (Op, Lp) in zip(bounds, states):
        sda.sda_attn_fwd(p, T["Qp"], T["Kp"], T["Vp"], idx_prev, Op, Lp, kb_begin=b0, kb_end=b1, out_dtype="f32")
    # current step: recompute the near partitions only, in place
    for q, ((b0, b1), (Op, Lp)) in enumerate(zip(bounds, states)):
        act = torch.from_numpy((~reuse[q]).astype(np.uint8)).cuda()
        sda.sda_attn_fwd(p, T["Q"], T["K"], T["V"], idx_now, Op, Lp, kb_begin=b0, kb_end=b1, qb_active=act,
                         out_dtype="f32")
    Om, Lm = new_state()
    sda.sda_merge_states([s[0] for s in states], [s[1] for s in states], 1, wl.N, wl.heads, wl.d, "f32", Om, Lm)
    # exact merge of fresh states equals the full-range forward
    fresh = [new_state() for _ in range(P)]
    for (b0, b1), (Op, Lp) in zip(bounds, fresh):
        sda.sda_attn_fwd(p, T["Q"], T["K"], T["V"], idx_now, Op, Lp, kb_begin=b0, kb_end=b1, out_dtype="f32")
    Oe, Le = new_state()
    sda.sda_merge_states([s[0] for s in fresh], [s[1] for s in fresh], 1, wl.N, wl.heads, wl.d, "f32", Oe, Le)
    Of = torch.empty_like(T["Q"])  # the full-range forward in the problem's dtype
    Lf = torch.empty((1, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_attn_fwd(p, T["Q"], T["K"], T["V"], idx_now, Of, Lf)
    torch.cuda.synchronize()
    assert sda.sda_get_device_status() == sda.SDA_OK
    rows = np.concatenate([geom.tokens(I) for I in qb])
    deviation = []
    for h in heads:
        xh = _head(x, h)
        ref_states = []
        for q, (b0, b1) in enumerate(bounds):
            prev = rec.oracle(orc.attn_fwd, xh["Qp"], xh["Kp"], xh["Vp"], rows_prev[h], geom, kb_begin=b0, kb_end=b1,
                              query_blocks=qb)
            now = rec.oracle(orc.attn_fwd, xh["Q"], xh["K"], xh["V"], rows_now[h], geom, kb_begin=b0, kb_end=b1,
                             query_blocks=qb)
            O_q, L_q = now[0].copy(), now[1].copy()
            for I in qb:
                if reuse[q, I]:
                    t = geom.tokens(I)
                    O_q[:, t] = prev[0][:, t]
                    L_q[:, :, t] = prev[1][:, :, t]
            ref_states.append((O_q[0, rows, 0], L_q[0, 0, rows], now[0][0, rows, 0], now[1][0, 0, rows]))
            # each state the GPU keeps equals the oracle's (reused or fresh)
            rec.close(host(states[q][0][0, rows, h]), ref_states[-1][0], "bf16", f"state O p{q} h{h}", "state O")
            rec.close(host(states[q][1][0, h, rows]), ref_states[-1][1], "bf16", f"state LSE p{q} h{h}", "state LSE")
        Ro, Rl = orc.merge_states([s[0] for s in ref_states], [s[1] for s in ref_states])
        rec.close(host(Om[0, rows, h]), Ro, "bf16", f"reuse-merged O h{h}", "reuse-merged O")
        rec.close(host(Lm[0, h, rows]), Rl, "bf16", f"reuse-merged LSE h{h}", "reuse-merged LSE")
        Eo, El = orc.merge_states([s[2] for s in ref_states], [s[3] for s in ref_states])
        rec.close(host(Oe[0, rows, h]), Eo, "bf16", f"exact-merged O h{h}", "exact-merged O")
        rec.close(host(Le[0, h, rows]), El, "bf16", f"exact-merged LSE h{h}", "exact-merged LSE")
        Fo, Fl = rec.oracle(orc.attn_fwd, xh["Q"], xh["K"], xh["V"], rows_now[h], geom, query_blocks=qb)
        rec.close(host(Of[0, rows, h]), Fo[0, rows, 0], "bf16", f"full-range O h{h}", "full-range O")
        assert_close(Eo, Fo[0, rows, 0], "bf16", "oracle: merge of partitions equals the union")
        deviation.append(errors(Ro, Eo))
    # the reuse approximation's deviation from the exact merge is reported, not graded
    rec.e["reuse_vs_exact_merge_max_abs_rel_frob"] = [max(d[0] for d in deviation), max(d[1] for d in deviation)]


def test_fwd_8k_predictor_training_signal_full_oracle(sda, parity_report):
    """The predictor's training signal on the 8,192-token workload in full (all 12 heads, all 4,096 block pairs
    each): per-pair s and t, the loss and dWq, dWk against the oracle's distillation gradient."""
    from tests.test_gpu_parity import _gpu_predictor_grad, check_predictor_grad

    wl = inputs.WORKLOADS["fwd_8k"]
    rec = _Record(parity_report, wl.name + " predictor training signal", "all 12 heads x all 4,096 block pairs")
    x = _inputs(wl, ("Q", "K", "Wq", "Wk"))
    geom = _geom(wl)
    dWq, dWk, L, s, t = _gpu_predictor_grad(sda, wl, x)
    L_ref, dWq_ref, dWk_ref, s_ref, t_ref = rec.oracle(orc.predictor_distill_grad, x["Q"], x["K"], x["Wq"], x["Wk"],
                                                       geom, wl.dtype)
    check_scores(s, s_ref)
    terr = float(np.abs(t - t_ref).max() / np.abs(t_ref).max())
    assert terr < 1e-5, terr
    assert abs(L - L_ref) <= 1e-4 * abs(L_ref), (L, L_ref)
    rq = check_predictor_grad(dWq, dWq_ref, "dWq")
    rk = check_predictor_grad(dWk, dWk_ref, "dWk")
    rec.e["outputs"]["dWq (max-abs / scale, rel-frob)"] = list(rq)
    rec.e["outputs"]["dWk (max-abs / scale, rel-frob)"] = list(rk)
    rec.e["outputs"]["loss (relative error)"] = abs(L - L_ref) / abs(L_ref)
    rec.e["outputs"]["t (max error / max |t|)"] = terr
    assert sda.sda_get_device_status() == sda.SDA_OK


def test_dsa3d_524k_sampled_tokens_every_head(sda, parity_report):
    """3D deformable sliding attention on the 524,288-token grid, 8 heads, d = 128, 3 x 3 x 3 window: the GPU
    runs the whole path (predicted offsets, then the attention) on every token; the oracle recomputes the
    offsets and the attention of 1,024 seeded tokens per head plus the grid's 8 corners ("MegaSlide-DiT",
    section 2 "3D-DSA")."""
    from oracle import dsa3d_oracle as D

    wl = inputs.DSA3D_WORKLOADS["dsa3d_524k"]
    rng = np.random.default_rng(11)
    corners = [((t * wl.H + h) * wl.W + w) for t in (0, wl.T - 1) for h in (0, wl.H - 1) for w in (0, wl.W - 1)]
    toks = np.unique(np.concatenate([rng.choice(wl.N, 1024, replace=False), corners]))
    rec = _Record(parity_report, wl.name, f"all 8 heads x {len(toks)} of {wl.N} tokens (fraction "
                                          f"{len(toks) / wl.N:.4f}), whole path: offsets then attention")
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "Wc", "bc", "Wl", "bl"))
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    p = sda.dsa3d_problem(wl.B, wl.T, wl.H, wl.W, wl.heads, wl.d, wl.kt, wl.kh, wl.kw)
    Q, K, V = (dev(x[n], "bf16") for n in ("Q", "K", "V"))
    off = torch.empty((wl.B, wl.N, wl.heads, wl.S, 3), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_offsets(p, Q, f(x["Wc"]), f(x["bc"]), f(x["Wl"]), f(x["bl"]), off)
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_fwd(p, Q, K, V, off, O, LSE)
    torch.cuda.synchronize()
    assert sda.sda_get_device_status() == sda.SDA_OK
    tt = torch.from_numpy(toks).cuda()
    off_s = host(off[:, tt])
    O_s, L_s = host(O[:, tt]), host(LSE[:, :, tt])
    del off, O, LSE, Q, K, V
    ref_off = rec.oracle(D.dsa3d_offsets, x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], wl.T, wl.H, wl.W, tokens=toks)
    mx, rel = errors(off_s, ref_off)
    scale = float(np.abs(ref_off).max())
    assert mx <= 1e-4 * scale and rel <= 1e-4, (mx, scale, rel)
    # the attention of the sampled tokens from the oracle's own offsets
    Or, Lr = rec.oracle(D.dsa3d_fwd, x["Q"], x["K"], x["V"], ref_off, wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw,
                        tokens=toks, offsets_of_tokens=True)
    rec.close(O_s, Or, "bf16", "O", "O")
    mx, rel = errors(L_s, Lr)
    assert mx <= 1e-4 * max(1.0, float(np.abs(Lr).max())) and rel <= 1e-4, (mx, rel)
    o = rec.e["outputs"].setdefault("offsets", {"max_abs": 0.0, "rel_frob_max": 0.0, "values": 0})
    o.update(max_abs=max(o["max_abs"], float(errors(off_s, ref_off)[0])), values=o["values"] + int(ref_off.size))
    o["rel_frob_max"] = max(o["rel_frob_max"], float(errors(off_s, ref_off)[1]))
    lo = rec.e["outputs"].setdefault("LSE", {"max_abs": 0.0, "rel_frob_max": 0.0, "values": 0})
    lo.update(max_abs=max(lo["max_abs"], mx), rel_frob_max=max(lo["rel_frob_max"], rel), values=lo["values"] + Lr.size)


def _fp32_record(rec, key, got, ref, rel):
    mx, rf = errors(got, ref)
    scale = max(1.0, float(np.abs(ref).max()))
    assert mx <= rel * scale and rf <= rel, f"{key}: max-abs {mx:.3e} (scale {scale:.3e}), rel-frob {rf:.3e}"
    o = rec.e["outputs"].setdefault(key, {"max_abs": 0.0, "rel_frob_max": 0.0, "values": 0})
    o["max_abs"] = max(o["max_abs"], float(mx))
    o["rel_frob_max"] = max(o["rel_frob_max"], float(rf))
    o["values"] += int(np.size(ref))


def test_dsa3d_524k_backward_sampled(sda, parity_report):
    """Both 3D-DSA backward calls on the 524,288-token grid, 8 heads, d = 128, 3 x 3 x 3 window, every token on
    the GPU.  The oracle recomputes: dQ and d_offsets of 512 seeded tokens (plus the grid's corners) on every
    head; dK and dV of 6 seeded rows (plus the first and last) on heads 0 and 7, from every token that can
    reach them; and the offset network's gradients of head 0 in full (dWc, dbc, dWl, dbl sum over all
    524,288 tokens) with its dQ at the sampled tokens.  Tolerance 5e-4 of scale, as at the small sizes."""
    from oracle import dsa3d_oracle as D
    from tests.parity_util import reaching_tokens

    wl = inputs.DSA3D_WORKLOADS["dsa3d_524k"]
    rng = np.random.default_rng(12)
    corners = [((t * wl.H + h) * wl.W + w) for t in (0, wl.T - 1) for h in (0, wl.H - 1) for w in (0, wl.W - 1)]
    toks = np.unique(np.concatenate([rng.choice(wl.N, 512, replace=False), corners]))
    rows = np.unique(np.concatenate([rng.choice(wl.N, 6, replace=False), [0, wl.N - 1]]))
    rec = _Record(parity_report, wl.name + "_backward",
                  f"dQ, d_offsets: 8 heads x {len(toks)} tokens; dK, dV: 2 heads x {len(rows)} rows; offset "
                  f"network: head 0 in full")
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "dO", "offsets", "Wc", "bc", "Wl", "d_offsets"))
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    p = sda.dsa3d_problem(wl.B, wl.T, wl.H, wl.W, wl.heads, wl.d, wl.kt, wl.kh, wl.kw)
    Q, K, V, dO = (dev(x[n], "bf16") for n in ("Q", "K", "V", "dO"))
    off = f(x["offsets"])
    O = torch.empty_like(Q)
    LSE = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_fwd(p, Q, K, V, off, O, LSE)
    shape = (wl.B, wl.N, wl.heads, wl.d)
    dQ, dK, dV = (torch.empty(shape, dtype=torch.float32, device="cuda") for _ in range(3))
    doff = torch.empty_like(off)
    bws = torch.empty(sda.sda_dsa3d_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    sda.sda_dsa3d_bwd(p, Q, K, V, off, LSE, dO, dQ, dK, dV, doff, bws)
    del bws
    dQn = torch.zeros(shape, dtype=torch.float32, device="cuda")
    gW = [torch.empty(x[n].shape, dtype=torch.float32, device="cuda") for n in ("Wc", "bc", "Wl")]
    gW.append(torch.empty((wl.heads, 3 * wl.S), dtype=torch.float32, device="cuda"))
    ws = torch.empty(sda.sda_dsa3d_offsets_bwd_workspace_size(p) // 4, dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_offsets_bwd(p, Q, f(x["Wc"]), f(x["bc"]), f(x["Wl"]), f(x["d_offsets"]), dQn, *gW, ws)
    torch.cuda.synchronize()
    assert sda.sda_get_device_status() == sda.SDA_OK
    tt, rr = torch.from_numpy(toks).cuda(), torch.from_numpy(rows).cuda()
    dQ_s, doff_s = host(dQ[:, tt]), host(doff[:, tt])
    dK_r, dV_r = host(dK[:, rr]), host(dV[:, rr])
    dQn_s = host(dQn[:, tt, :1])
    gW = [host(g[:1]) for g in gW]
    del Q, K, V, dO, off, O, LSE, dQ, dK, dV, doff, dQn, ws
    torch.cuda.empty_cache()
    rel = 5e-4
    ref = rec.oracle(D.dsa3d_bwd, x["Q"], x["K"], x["V"], x["offsets"], x["dO"], wl.T, wl.H, wl.W, wl.kt, wl.kh,
                     wl.kw, tokens=toks)
    _fp32_record(rec, "dQ", dQ_s, ref[0], rel)
    _fp32_record(rec, "d_offsets", doff_s, ref[3], rel)
    for hi, h in enumerate((0, wl.heads - 1)):
        xs = {n: x[n][:, :, h:h + 1] for n in ("Q", "K", "V", "dO", "offsets")}
        near = reaching_tokens(rows, xs["offsets"], wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
        rk = rec.oracle(D.dsa3d_bwd, xs["Q"], xs["K"], xs["V"], xs["offsets"], xs["dO"], wl.T, wl.H, wl.W, wl.kt,
                        wl.kh, wl.kw, tokens=near, rows=rows)
        _fp32_record(rec, "dK", dK_r[:, :, h:h + 1], rk[1], rel)
        _fp32_record(rec, "dV", dV_r[:, :, h:h + 1], rk[2], rel)
    rn = rec.oracle(D.dsa3d_offsets_bwd, x["Q"][:, :, :1], x["Wc"][:1], x["bc"][:1], x["Wl"][:1], None,
                    x["d_offsets"][:, :, :1], wl.T, wl.H, wl.W)
    _fp32_record(rec, "offset network dQ", dQn_s, rn[0][:, toks], rel)
    for name, g, r in zip(("dWc", "dbc", "dWl", "dbl"), gW, rn[1:]):
        _fp32_record(rec, name, g, r, rel)


def test_predictor_with_two_query_blocks_per_cta(sda, parity_report):
    """A grid whose score rows no longer fit four query blocks per CTA in shared memory (7,680 blocks of
    2 x 8 x 8, 983,040 tokens; four fit up to about 7,500 blocks and the API admits 8,192): the score kernel
    runs two query blocks per CTA, its two MMA issuers still splitting the pairs by parity.  One head,
    d = 64, r = 32, 5% kept; the first, middle and last query blocks plus three seeded ones: selection by
    the gap rule, scores, and the forward on those rows."""
    wl = inputs.Workload("fwd_983k_qb2", 1, 1, 32, 128, 240, 64, 2, 8, 8, 32, 0.05, "bf16", 4.0, 32)
    assert wl.n_blocks == 7680
    qb = _samples(wl, 3, 53)
    rec = _Record(parity_report, wl.name, f"1 head x {len(qb)} of {wl.n_blocks} query blocks (two query "
                                          f"blocks per score CTA)")
    _check_predictor_and_forward(sda, rec, wl, [0], qb)
