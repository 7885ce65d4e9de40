"""One small pass of the whole path on cuda:0 through the C ABI, checked against the oracle.

A 2-head bf16 problem on a ragged 3 x 10 x 12 grid (2x8x8 tiles, 8 blocks,
d = 64, r = 16, 4 of 8 key blocks kept): predictor + top-k, forward, backward,
two key-partition states and their merge, the gradient through that merge
(merge backward, then each partition state's backward, summed), the
predictor's training signal (distillation gradient of Wq, Wk), and 3D deformable
sliding attention (predicted offsets, the sampled-window attention, and the
backward of both).
"""
from __future__ import annotations

import numpy as np


def run(device: int = 0) -> dict:
    import torch

    import oracle as orc
    from dynamic_block_sparse_rank_gb300 import inputs, sda
    from tests.parity_util import assert_close, check_selection, dev, host

    torch.cuda.set_device(device)
    wl = inputs.Workload("smoke", 1, 2, 3, 10, 12, 64, 2, 8, 8, 16, 0.5, "bf16", 3.0, 16, backward=True)
    x = inputs.generate(wl, names=("Q", "K", "V", "dO", "Wq", "Wk"))
    geom = orc.Geometry(wl.T, wl.H, wl.W, wl.bt, wl.bh, wl.bw)
    p = sda.problem_from_workload(wl)
    nb, k = sda.sda_num_blocks(p)
    Q, K, V, dO, Wq, Wk = (dev(x[n], "bf16") for n in ("Q", "K", "V", "dO", "Wq", "Wk"))

    # 1. predictor
    idx = torch.empty((1, wl.heads, nb, k), dtype=torch.int32, device="cuda")
    score = torch.empty((1, wl.heads, nb, nb), dtype=torch.float32, device="cuda")
    ws = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICT), dtype=torch.uint8, device="cuda")
    sda.sda_predict_blocks(p, Q, K, Wq, Wk, idx, score, ws)
    ref_idx, ref_scores = orc.predict_blocks(x["Q"], x["K"], x["Wq"], x["Wk"], geom, wl.keep, "bf16")
    sel = check_selection(idx.cpu().numpy(), ref_scores, k)
    assert sel["fail"] == 0, sel
    s_err = np.abs(host(score) - ref_scores).max() / np.abs(ref_scores).max()
    assert s_err < 1e-4, s_err

    # 2. forward on the oracle's map
    idx_t = torch.from_numpy(ref_idx).cuda()
    O = torch.empty_like(Q)
    LSE = torch.empty((1, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_attn_fwd(p, Q, K, V, idx_t, O, LSE)
    O_ref, L_ref = orc.attn_fwd(x["Q"], x["K"], x["V"], ref_idx, geom)
    assert_close(host(O), O_ref, "bf16", "smoke O")
    assert_close(host(LSE), L_ref, "bf16", "smoke LSE")

    # 3. backward
    dQ, dK, dV = (torch.empty(Q.shape, dtype=torch.float32, device="cuda") for _ in range(3))
    wsb = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_BWD), dtype=torch.uint8, device="cuda")
    sda.sda_attn_bwd(p, Q, K, V, O, LSE, dO, idx_t, dQ, dK, dV, "f32", wsb)
    gref = orc.attn_bwd(x["Q"], x["K"], x["V"], x["dO"], ref_idx, geom)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dQ, dK, dV), gref):
        assert_close(host(got), ref, "bf16", "smoke " + name)

    # 4. two key partitions and their merge
    cut = nb // 2
    parts = []
    for b0, b1 in ((0, cut), (cut, nb)):
        Op = torch.empty_like(Q)
        Lp = torch.empty_like(LSE)
        sda.sda_attn_fwd(p, Q, K, V, idx_t, Op, Lp, kb_begin=b0, kb_end=b1)
        parts.append((Op, Lp))
    Om, Lm = torch.empty_like(Q), torch.empty_like(LSE)
    sda.sda_merge_states([q[0] for q in parts], [q[1] for q in parts], 1, wl.N, wl.heads, wl.d, "bf16", Om, Lm)
    assert_close(host(Om), O_ref, "bf16", "smoke merged O")
    assert_close(host(Lm), L_ref, "bf16", "smoke merged LSE")

    # 5. training through the merge: the two partitions are the grid's two frame slabs and cover every key;
    # the oracle's reference is the same composition with the fresh states read as stored (bf16)
    gO = [torch.empty_like(Q) for _ in parts]
    gL = [torch.empty_like(LSE) for _ in parts]
    sda.sda_merge_states_bwd([q[0] for q in parts], [q[1] for q in parts], dO, None, 1, wl.N, wl.heads, wl.d, "bf16",
                             gO, gL)
    total = [torch.zeros(Q.shape, dtype=torch.float32, device="cuda") for _ in range(3)]
    for (b0, b1), (Op, Lp), g_o, g_l in zip(((0, cut), (cut, nb)), parts, gO, gL):
        part = [torch.empty_like(total[0]) for _ in range(3)]
        sda.sda_attn_bwd_partition(p, Q, K, V, Op, Lp, g_o, g_l, idx_t, *part, "f32", wsb, kb_begin=b0, kb_end=b1)
        for acc, v in zip(total, part):
            acc += v
    assert orc.frame_partitions(geom, 2) == [(0, cut), (cut, nb)]
    mref = orc.reuse_bwd(x["Q"], x["K"], x["V"], x["dO"], ref_idx, geom, 2, 0, None, state_dtype="bf16")
    for name, got, ref in zip(("dQ", "dK", "dV"), total, mref):
        assert_close(host(got), ref, "bf16", "smoke merged-partition " + name)
    # 6. the predictor's training signal (distillation gradient of Wq, Wk)
    dWq = torch.empty((wl.heads, wl.d, wl.rank), dtype=torch.float32, device="cuda")
    dWk = torch.empty_like(dWq)
    loss = torch.empty((1,), dtype=torch.float64, device="cuda")
    wsg = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICTOR_GRAD), dtype=torch.uint8, device="cuda")
    sda.sda_predictor_grad(p, Q, K, Wq, Wk, dWq, dWk, loss, wsg)
    loss_ref, dWq_ref, dWk_ref, _, _ = orc.predictor_distill_grad(x["Q"], x["K"], x["Wq"], x["Wk"], geom, "bf16")
    for name, got, ref in (("dWq", dWq, dWq_ref), ("dWk", dWk, dWk_ref)):
        err = np.linalg.norm(host(got) - ref) / np.linalg.norm(ref)
        assert err < 1e-2, (name, err)
    assert abs(float(loss.item()) - loss_ref) <= 1e-4 * abs(loss_ref)
    # 7. 3D deformable sliding attention: predicted offsets, the sampled-window attention, then the backward
    # of both (attention, then the offset network)
    from oracle import dsa3d_oracle as D

    dw = inputs.Dsa3dWorkload("smoke_dsa3d", 1, 2, 3, 8, 10, 64, 3, 3, 3, 1.0)
    xd = inputs.generate_dsa3d(dw, names=("Q", "K", "V", "dO", "Wc", "bc", "Wl", "bl"))
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    dp = sda.dsa3d_problem(dw.B, dw.T, dw.H, dw.W, dw.heads, dw.d, dw.kt, dw.kh, dw.kw)
    dQ, dK, dV = (dev(xd[n], "bf16") for n in ("Q", "K", "V"))
    doff = torch.empty((dw.B, dw.N, dw.heads, dw.S, 3), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_offsets(dp, dQ, f32(xd["Wc"]), f32(xd["bc"]), f32(xd["Wl"]), f32(xd["bl"]), doff)
    dO_ = torch.empty_like(dQ)
    dL = torch.empty((dw.B, dw.heads, dw.N), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_fwd(dp, dQ, dK, dV, doff, dO_, dL)
    roff = D.dsa3d_offsets(xd["Q"], xd["Wc"], xd["bc"], xd["Wl"], xd["bl"], dw.T, dw.H, dw.W)
    assert np.abs(host(doff) - roff).max() <= 1e-4 * max(1.0, np.abs(roff).max())
    rO, rL = D.dsa3d_fwd(xd["Q"], xd["K"], xd["V"], roff, dw.T, dw.H, dw.W, dw.kt, dw.kh, dw.kw)
    assert_close(host(dO_), rO, "bf16", "smoke 3D-DSA O")
    assert np.abs(host(dL) - rL).max() <= 1e-4 * max(1.0, np.abs(rL).max())
    shape = (dw.B, dw.N, dw.heads, dw.d)
    gQ, gK, gV = (torch.empty(shape, dtype=torch.float32, device="cuda") for _ in range(3))
    goff = torch.empty_like(doff)
    ws = torch.empty(sda.sda_dsa3d_bwd_workspace_size(dp), dtype=torch.uint8, device="cuda")
    sda.sda_dsa3d_bwd(dp, dQ, dK, dV, doff, dL, dev(xd["dO"], "bf16"), gQ, gK, gV, goff, ws)
    gw = [torch.empty(xd[n].shape, dtype=torch.float32, device="cuda") for n in ("Wc", "bc", "Wl", "bl")]
    ws2 = torch.empty(sda.sda_dsa3d_offsets_bwd_workspace_size(dp), dtype=torch.uint8, device="cuda")
    sda.sda_dsa3d_offsets_bwd(dp, dQ, f32(xd["Wc"]), f32(xd["bc"]), f32(xd["Wl"]), goff, gQ, *gw, ws2)
    rQ, rK, rV, rdo = D.dsa3d_bwd(xd["Q"], xd["K"], xd["V"], roff, xd["dO"], dw.T, dw.H, dw.W, dw.kt, dw.kh, dw.kw)
    rn = D.dsa3d_offsets_bwd(xd["Q"], xd["Wc"], xd["bc"], xd["Wl"], xd["bl"], rdo, dw.T, dw.H, dw.W)
    for name, got, ref in (("dQ", gQ, rQ + rn[0]), ("dK", gK, rK), ("dV", gV, rV), ("dWc", gw[0], rn[1]),
                           ("dWl", gw[2], rn[3])):
        err = np.abs(host(got) - ref).max()
        assert err <= 5e-4 * max(1.0, np.abs(ref).max()), f"smoke 3D-DSA {name}: {err}"
    st = sda.sda_get_device_status()
    assert st == sda.SDA_OK, sda.status_string(st)
    return {"selection": sel, "score_rel_err": float(s_err)}


if __name__ == "__main__":
    print(run())
