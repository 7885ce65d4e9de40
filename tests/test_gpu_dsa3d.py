"""GPU parity of 3D deformable sliding attention against the fp64 oracle (through the C ABI).

"MegaSlide-DiT" (gist.science explainer), section 2 "3D deformable sliding attention": offsets from a
depthwise 3x3x3 convolution and a linear layer, trilinear sampling of K and V around every token, softmax
over the window.  Tolerances: O is stored in bf16, so the bf16 bound (max-abs 2e-2, rel-Frobenius 1e-2);
LSE and the offsets are fp32 results of exact bf16 inputs, held to 1e-4 of their scale (fp32 accumulation
over at most 27 + d terms).
"""
import math

import numpy as np
import pytest

from dynamic_block_sparse_rank_gb300 import inputs
from oracle import dsa3d_oracle as D
from tests.parity_util import assert_close, dev, errors, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_rank_gb300 import sda as s

    s.lib()
    return s


WLS = inputs.DSA3D_WORKLOADS
SMALL = [WLS["dsa3d_ragged_d64"], WLS["dsa3d_d128_1x5x5"], WLS["dsa3d_far"]]


def _problem(sda, wl, scale=0.0):
    return sda.dsa3d_problem(wl.B, wl.T, wl.H, wl.W, wl.heads, wl.d, wl.kt, wl.kh, wl.kw, scale)


def _gpu_fwd(sda, wl, x, offsets, scale=0.0):
    O = torch.full((wl.B, wl.N, wl.heads, wl.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = torch.full((wl.B, wl.heads, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_fwd(_problem(sda, wl, scale), dev(x["Q"], "bf16"), dev(x["K"], "bf16"), dev(x["V"], "bf16"),
                      torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.float32)).cuda(), O, L)
    torch.cuda.synchronize()
    assert sda.sda_get_device_status() == sda.SDA_OK
    return host(O), host(L)


def _gpu_offsets(sda, wl, x):
    off = torch.full((wl.B, wl.N, wl.heads, wl.S, 3), float("nan"), dtype=torch.float32, device="cuda")
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    sda.sda_dsa3d_offsets(_problem(sda, wl), dev(x["Q"], "bf16"), f(x["Wc"]), f(x["bc"]), f(x["Wl"]), f(x["bl"]),
                          off)
    torch.cuda.synchronize()
    return host(off)


def check_fp32(got, ref, what, rel=1e-4, frob=True):
    """max-abs within rel of max(1, |ref|), and (frob) the relative Frobenius error within rel."""
    mx, rf = errors(got, ref)
    scale = max(1.0, float(np.abs(ref).max()))
    print(f"{what}: max-abs/scale {mx / scale:.2e}, rel-frob {rf:.2e}")
    assert mx <= rel * scale and (rf <= rel or not frob), \
        f"{what}: max-abs {mx:.3e} (scale {scale:.3e}), rel-frob {rf:.3e}"


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_dsa3d_forward_matches_oracle(sda, wl):
    x = inputs.generate_dsa3d(wl)
    O, L = _gpu_fwd(sda, wl, x, x["offsets"])
    Or, Lr = D.dsa3d_fwd(x["Q"], x["K"], x["V"], x["offsets"], wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    assert_close(O, Or, "bf16", "O")
    check_fp32(L, Lr, "LSE")


@pytest.mark.parametrize("wl", SMALL[:2], ids=lambda w: w.name)
def test_dsa3d_offsets_match_oracle(sda, wl):
    x = inputs.generate_dsa3d(wl, names=("Q", "Wc", "bc", "Wl", "bl"))
    got = _gpu_offsets(sda, wl, x)
    ref = D.dsa3d_offsets(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], wl.T, wl.H, wl.W)
    check_fp32(got, ref, "offsets")


def test_dsa3d_predicted_offsets_then_attention(sda):
    """The whole path: the GPU's offsets feed the GPU's attention; the oracle's own offsets feed its own."""
    wl = WLS["dsa3d_ragged_d64"]
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "Wc", "bc", "Wl", "bl"))
    off = _gpu_offsets(sda, wl, x)
    O, L = _gpu_fwd(sda, wl, x, off)
    ref_off = D.dsa3d_offsets(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], wl.T, wl.H, wl.W)
    Or, Lr = D.dsa3d_fwd(x["Q"], x["K"], x["V"], ref_off, wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    assert_close(O, Or, "bf16", "O")
    check_fp32(L, Lr, "LSE")


def test_dsa3d_samples_outside_or_not_finite(sda):
    """Samples wholly outside the raster, and non-finite offsets, give k = v = 0 and logit 0 on both sides;
    with every sample out, O = 0 and LSE = log S exactly."""
    wl = WLS["dsa3d_ragged_d64"]
    x = inputs.generate_dsa3d(wl)
    off = x["offsets"].copy()
    rng = np.random.default_rng(3)
    pick = rng.random(off.shape[:4]) < 0.2
    off[pick, 0] = np.where(rng.random(pick.sum()) < 0.5, np.nan, np.inf)
    O, L = _gpu_fwd(sda, wl, x, off)
    Or, Lr = D.dsa3d_fwd(x["Q"], x["K"], x["V"], off, wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    assert_close(O, Or, "bf16", "O (non-finite offsets)")
    check_fp32(L, Lr, "LSE (non-finite offsets)")
    O2, L2 = _gpu_fwd(sda, wl, x, np.full_like(off, 1.0e6))
    assert np.all(O2 == 0.0)
    np.testing.assert_allclose(L2, math.log(wl.S), rtol=0, atol=2e-6)


def test_dsa3d_one_point_window_returns_v(sda):
    wl = WLS["dsa3d_d128_1x5x5"].with_(kt=1, kh=1, kw=1)
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V"))
    O, L = _gpu_fwd(sda, wl, x, np.zeros((wl.B, wl.N, wl.heads, 1, 3), np.float32), scale=0.25)
    np.testing.assert_array_equal(O, x["V"])  # softmax over one sample, stored exactly
    ref = 0.25 * np.einsum("bnhd,bnhd->bhn", x["Q"].astype(np.float64), x["K"].astype(np.float64))
    check_fp32(L, ref, "LSE")


def test_dsa3d_integer_offsets_gather_rows(sda):
    wl = WLS["dsa3d_far"]
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "offsets"))
    off = np.rint(x["offsets"])
    O, L = _gpu_fwd(sda, wl, x, off)
    Or, Lr = D.dsa3d_fwd(x["Q"], x["K"], x["V"], off, wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    assert_close(O, Or, "bf16", "O (integer offsets)")
    check_fp32(L, Lr, "LSE (integer offsets)")


@pytest.mark.parametrize("wl", [inputs.Dsa3dWorkload("dsa3d_5x5x5_d64", 1, 2, 6, 7, 9, 64, 5, 5, 5, 1.5),
                                inputs.Dsa3dWorkload("dsa3d_one_token_d128", 2, 3, 1, 1, 1, 128, 3, 3, 3, 0.5),
                                inputs.Dsa3dWorkload("dsa3d_line_d128", 1, 1, 1, 1, 37, 128, 1, 1, 7, 2.0)],
                         ids=lambda w: w.name)
def test_dsa3d_edge_shapes(sda, wl):
    """The largest window (5 x 5 x 5 = 125 points: 375 offset outputs, four passes of the offset network's
    output tiles), a single-token grid (every sample but the centre's corners outside), and a 1 x 1 x 37 line
    with a 1 x 1 x 7 window; both steps against the oracle."""
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "offsets", "Wc", "bc", "Wl", "bl"))
    O, L = _gpu_fwd(sda, wl, x, x["offsets"])
    Or, Lr = D.dsa3d_fwd(x["Q"], x["K"], x["V"], x["offsets"], wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    assert_close(O, Or, "bf16", "O")
    check_fp32(L, Lr, "LSE")
    got = _gpu_offsets(sda, wl, x)
    ref = D.dsa3d_offsets(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], wl.T, wl.H, wl.W)
    check_fp32(got, ref, "offsets")


BWD_REL = 5e-4  # backward results, relative to their scale (see test_dsa3d_backward_matches_oracle)
OFFB_REL = 1e-5  # the offset network's backward: fp32 sums of exact inputs (see its test)


def _gpu_bwd(sda, wl, x, offsets):
    O, L = None, None
    p = _problem(sda, wl)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    Q, K, V, dO = (dev(x[n], "bf16") for n in ("Q", "K", "V", "dO"))
    off = f32(offsets)
    Ot = torch.empty_like(Q)
    Lt = torch.empty((wl.B, wl.heads, wl.N), dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_fwd(p, Q, K, V, off, Ot, Lt)
    shape = (wl.B, wl.N, wl.heads, wl.d)
    dQ, dK, dV = (torch.full(shape, float("nan"), dtype=torch.float32, device="cuda") for _ in range(3))
    doff = torch.full(off.shape, float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.full((sda.sda_dsa3d_bwd_workspace_size(p),), 0xA5, dtype=torch.uint8, device="cuda")  # not zeroed
    sda.sda_dsa3d_bwd(p, Q, K, V, off, Lt, dO, dQ, dK, dV, doff, ws)
    torch.cuda.synchronize()
    assert sda.sda_get_device_status() == sda.SDA_OK
    del O, L
    return host(dQ), host(dK), host(dV), host(doff)


@pytest.mark.parametrize("wl", SMALL + [inputs.Dsa3dWorkload("dsa3d_5x5x5_d64", 1, 2, 6, 7, 9, 64, 5, 5, 5, 1.5)],
                         ids=lambda w: w.name)
def test_dsa3d_backward_matches_oracle(sda, wl):
    """dQ (the attention's part), dK, dV and the offsets' gradient against the oracle's reading D5 (pinned by
    torch autograd through grid_sample and by finite differences).  fp32 results of bf16 inputs, held to
    BWD_REL of their scale: with the correlated Q, K of these inputs the logits' dot products reach a few
    hundred, whose fp32 accumulation moves each logit, and so each P, by ~1e-5 relative; dP - D then cancels,
    and dK, dV sum up to 8 S contributions per row by atomics."""
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "dO", "offsets"))
    dQ, dK, dV, doff = _gpu_bwd(sda, wl, x, x["offsets"])
    rQ, rK, rV, roff = D.dsa3d_bwd(x["Q"], x["K"], x["V"], x["offsets"], x["dO"], wl.T, wl.H, wl.W, wl.kt, wl.kh,
                                   wl.kw)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV), ("d_offsets", doff, roff)):
        check_fp32(got, ref, name, rel=BWD_REL)


def test_dsa3d_backward_outside_and_integer_samples(sda):
    """Non-finite offsets give no gradient through their samples; integer offsets take the derivative from
    above (floor's side), as the oracle does."""
    wl = WLS["dsa3d_ragged_d64"]
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "dO", "offsets"))
    off = np.rint(x["offsets"]).astype(np.float32)
    rng = np.random.default_rng(5)
    pick = rng.random(off.shape[:4]) < 0.15
    off[pick, 1] = np.nan
    dQ, dK, dV, doff = _gpu_bwd(sda, wl, x, off)
    rQ, rK, rV, roff = D.dsa3d_bwd(x["Q"], x["K"], x["V"], off, x["dO"], wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV), ("d_offsets", doff, roff)):
        check_fp32(got, ref, name, rel=BWD_REL)


def _gpu_offsets_bwd(sda, wl, x, dQ0):
    p = _problem(sda, wl)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    dQ = f32(dQ0)
    outs = [torch.full(x[n].shape, float("nan"), dtype=torch.float32, device="cuda") for n in ("Wc", "bc", "Wl", "bl")]
    ws = torch.empty(sda.sda_dsa3d_offsets_bwd_workspace_size(p) // 4, dtype=torch.float32, device="cuda")
    sda.sda_dsa3d_offsets_bwd(p, dev(x["Q"], "bf16"), f32(x["Wc"]), f32(x["bc"]), f32(x["Wl"]), f32(x["d_offsets"]),
                              dQ, *outs, ws)
    torch.cuda.synchronize()
    assert sda.sda_get_device_status() == sda.SDA_OK
    return [host(dQ)] + [host(t) for t in outs]


@pytest.mark.parametrize("wl", SMALL + [inputs.Dsa3dWorkload("dsa3d_5x5x5_d64", 1, 2, 6, 7, 9, 64, 5, 5, 5, 1.5),
                                        inputs.Dsa3dWorkload("dsa3d_3x5x5_d128", 2, 1, 5, 6, 70, 128, 3, 5, 5, 1.0)],
                         ids=lambda w: w.name)
def test_dsa3d_offsets_backward_matches_oracle(sda, wl):
    """The offset network's gradients (reading D5: dY = G Wl^T, dWl = Y^T G, dbl, dWc, dbc and the transposed
    convolution added into dQ) against the oracle, which torch autograd through conv3d pins.  dQ starts from a
    given value, so the call's addition is checked too.  The inputs are exact in fp32 and every result is an
    fp32 sum of at most a few thousand products (weight gradients over every token, by atomics), whose
    rounding stays near 1e-7 of the scale: held to OFFB_REL.  The 5 x 5 x 5 and 3 x 5 x 5 windows take 4 and
    3 column passes."""
    x = inputs.generate_dsa3d(wl, names=("Q", "Wc", "bc", "Wl", "bl", "d_offsets"))
    dQ0 = inputs.generate_dsa3d(wl, seed=3, names=("dO",))["dO"]
    got = _gpu_offsets_bwd(sda, wl, x, dQ0)
    ref = D.dsa3d_offsets_bwd(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], x["d_offsets"], wl.T, wl.H, wl.W)
    ref = [ref[0] + dQ0.astype(np.float64)] + list(ref[1:])
    for name, g, r in zip(("dQ", "dWc", "dbc", "dWl", "dbl"), got, ref):
        check_fp32(g, r, name, rel=OFFB_REL)


def test_dsa3d_full_backward_chain(sda):
    """Attention backward, then the offset network's: the total dQ and the weight gradients match the oracle's
    chain (dsa3d_bwd's d_offsets fed to dsa3d_offsets_bwd), with the offsets the network predicts."""
    wl = WLS["dsa3d_ragged_d64"]
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "dO", "Wc", "bc", "Wl", "bl"))
    off = D.dsa3d_offsets(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], wl.T, wl.H, wl.W)
    dQa, dK, dV, doff = _gpu_bwd(sda, wl, x, off)
    rQ, rK, rV, roff = D.dsa3d_bwd(x["Q"], x["K"], x["V"], off, x["dO"], wl.T, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    y = dict(x, d_offsets=doff)
    got = _gpu_offsets_bwd(sda, wl, y, dQa)
    ref = D.dsa3d_offsets_bwd(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], roff, wl.T, wl.H, wl.W)
    ref = [ref[0] + rQ] + list(ref[1:])
    for name, g, r in zip(("dQ total", "dWc", "dbc", "dWl", "dbl"), got, ref):
        check_fp32(g, r, name, rel=BWD_REL)


@pytest.mark.parametrize("wl", [inputs.Dsa3dWorkload("dsa3d_5x5x5_d128", 1, 2, 6, 7, 9, 128, 5, 5, 5, 1.5),
                                inputs.Dsa3dWorkload("dsa3d_one_token_d128", 2, 3, 1, 1, 1, 128, 3, 3, 3, 0.5),
                                inputs.Dsa3dWorkload("dsa3d_line_d64", 1, 1, 1, 1, 37, 64, 1, 1, 7, 2.0),
                                inputs.Dsa3dWorkload("dsa3d_ragged_tail_d64", 3, 1, 2, 5, 13, 64, 3, 3, 3, 1.0)],
                         ids=lambda w: w.name)
def test_dsa3d_backward_edge_shapes(sda, wl):
    """Both backward calls on the largest window at d = 128 (125 points: four column passes of the offset
    network, 125-entry sample records per token), a single-token grid (a 2 x 2 x 2 cell grid, every
    corner but the token's own outside), a 1 x 1 x 37 line, and 130 tokens per batch entry (a partial
    CTA of the per-token and row kernels, three batch entries sharing one bucket workspace)."""
    x = inputs.generate_dsa3d(wl, names=("Q", "K", "V", "dO", "offsets", "Wc", "bc", "Wl", "bl", "d_offsets"))
    dQ, dK, dV, doff = _gpu_bwd(sda, wl, x, x["offsets"])
    rQ, rK, rV, roff = D.dsa3d_bwd(x["Q"], x["K"], x["V"], x["offsets"], x["dO"], wl.T, wl.H, wl.W, wl.kt, wl.kh,
                                   wl.kw)
    one_point = wl.N == 1
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV), ("d_offsets", doff, roff)):
        # On a one-token grid every sampled k~ and v~ is a multiple (its corner weight c_s) of the one K or
        # V row, so both dq and the row's dK reduce to sum_s da_s c_s = (dO.V_0) Var_P(c): a variance of
        # nearly equal weights, ~1e-4 of the terms it comes from.  fp32 logits near 100 fix P only to
        # ~1e-5 relative, which puts an absolute error of ~1e-5 on them whatever the order of the sums:
        # their relative Frobenius error has no fp32 meaning there, and only the max-abs bound applies.
        check_fp32(got, ref, name, rel=BWD_REL, frob=not (one_point and name in ("dQ", "dK")))
    got = _gpu_offsets_bwd(sda, wl, x, np.zeros_like(x["Q"]))
    ref = D.dsa3d_offsets_bwd(x["Q"], x["Wc"], x["bc"], x["Wl"], x["bl"], x["d_offsets"], wl.T, wl.H, wl.W)
    for name, g, r in zip(("dQ", "dWc", "dbc", "dWl", "dbl"), got, ref):
        check_fp32(g, r, name, rel=OFFB_REL)
