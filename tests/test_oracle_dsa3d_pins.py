"""Pins of the 3D deformable sliding attention oracle (CPU only).

Each test ties `oracle.dsa3d_oracle` to something other than itself: explicit neighbourhood loops, integer
gathers, SciPy's n-D correlation and linear interpolation, closed forms of trilinear interpolation and of a
one-point softmax.  "MegaSlide-DiT" (gist.science explainer), section 2 "3D deformable sliding attention".
"""
import math

import numpy as np
import pytest

from oracle import dsa3d_oracle as D
from tests.parity_util import reaching_tokens

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _grid(rng, T, H, W, Hh, d, B=1):
    N = T * H * W
    return tuple(rng.standard_normal((B, N, Hh, d)) for _ in range(3))


def _brute(Q, K, V, T, H, W, shifts, scale):
    """Attention of every token over explicitly listed integer sample positions: shifts[n][s] = (dt, dh, dw)
    relative to the token; positions off the raster give zero k and v (logit 0)."""
    B, N, Hh, d = Q.shape
    O = np.zeros_like(Q)
    L = np.zeros((B, Hh, N))
    for b in range(B):
        for h in range(Hh):
            for t in range(T):
                for y in range(H):
                    for x in range(W):
                        n = (t * H + y) * W + x
                        logits, vals = [], []
                        for (a, c, e) in shifts[n]:
                            tt, yy, xx = t + a, y + c, x + e
                            if 0 <= tt < T and 0 <= yy < H and 0 <= xx < W:
                                m = (tt * H + yy) * W + xx
                                logits.append(scale * float(Q[b, n, h] @ K[b, m, h]))
                                vals.append(V[b, m, h])
                            else:
                                logits.append(0.0)
                                vals.append(np.zeros(d))
                        lg = np.array(logits)
                        mx = lg.max()
                        w = np.exp(lg - mx)
                        O[b, n, h] = (w[:, None] * np.array(vals)).sum(0) / w.sum()
                        L[b, h, n] = mx + math.log(w.sum())
    return O, L


def test_window_points_are_centred_raster_order():
    g = D.window_points(3, 1, 5)
    assert g.shape == (15, 3)
    assert g[0].tolist() == [-1, 0, -2] and g[4].tolist() == [-1, 0, 2] and g[5].tolist() == [0, 0, -2]
    assert g[-1].tolist() == [1, 0, 2]
    with pytest.raises(ValueError):
        D.window_points(2, 3, 3)


def test_zero_offsets_is_neighbourhood_attention():
    rng = np.random.default_rng(1)
    T, H, W, Hh, d = 3, 4, 5, 2, 4
    Q, K, V = _grid(rng, T, H, W, Hh, d)
    N = T * H * W
    O, L = D.dsa3d_fwd(Q, K, V, np.zeros((1, N, Hh, 27, 3)), T, H, W, 3, 3, 3)
    win = [(a, c, e) for a in (-1, 0, 1) for c in (-1, 0, 1) for e in (-1, 0, 1)]
    Ob, Lb = _brute(Q, K, V, T, H, W, [win] * N, 1 / math.sqrt(d))
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


def test_integer_offsets_gather_the_shifted_rows():
    rng = np.random.default_rng(2)
    T, H, W, Hh, d = 3, 3, 4, 1, 6
    Q, K, V = _grid(rng, T, H, W, Hh, d)
    N = T * H * W
    kt, kh, kw = 1, 3, 3
    off = rng.integers(-2, 3, size=(1, N, Hh, 9, 3)).astype(np.float64)
    O, L = D.dsa3d_fwd(Q, K, V, off, T, H, W, kt, kh, kw, scale=0.7)
    g = D.window_points(kt, kh, kw)
    shifts = [[tuple(int(v) for v in g[s] + off[0, n, 0, s]) for s in range(9)] for n in range(N)]
    Ob, Lb = _brute(Q, K, V, T, H, W, shifts, 0.7)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


def test_trilinear_reproduces_affine_rows_and_grid_points():
    rng = np.random.default_rng(3)
    T, H, W, d = 4, 5, 6, 3
    c = D.token_coords(T, H, W)
    A = rng.standard_normal((3, d))
    b0 = rng.standard_normal(d)
    X = c @ A + b0  # affine in (t, h, w)
    pos = rng.uniform([0, 0, 0], [T - 1, H - 1, W - 1], size=(50, 3))  # inside the raster: no zero padding
    np.testing.assert_allclose(D.trilinear(X, pos, T, H, W), pos @ A + b0, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(D.trilinear(X, c, T, H, W), X)  # grid points: the rows themselves
    far = np.array([[-2.0, 0, 0], [0, H + 0.5, 0], [0, 0, -1.0], [np.nan, 1, 1], [1, np.inf, 1], [1, 1, -np.inf]])
    assert np.all(D.trilinear(X, far, T, H, W) == 0.0)  # wholly outside or not finite: zero rows


def test_trilinear_matches_scipy_linear_interpolation_with_zero_padding():
    ndimage = pytest.importorskip("scipy.ndimage")
    rng = np.random.default_rng(4)
    T, H, W, d = 3, 4, 5, 2
    X = rng.standard_normal((T * H * W, d))
    pos = rng.uniform([-1.5, -1.5, -1.5], [T + 0.5, H + 0.5, W + 0.5], size=(200, 3))
    got = D.trilinear(X, pos, T, H, W)
    for ch in range(d):
        ref = ndimage.map_coordinates(X[:, ch].reshape(T, H, W), pos.T, order=1, mode="grid-constant", cval=0.0)
        np.testing.assert_allclose(got[:, ch], ref, rtol=0, atol=1e-12)


def test_uniform_attention_is_the_mean_of_the_samples():
    ndimage = pytest.importorskip("scipy.ndimage")
    rng = np.random.default_rng(5)
    T, H, W, Hh, d = 2, 3, 4, 1, 3
    N = T * H * W
    _, K, V = _grid(rng, T, H, W, Hh, d)
    Q = np.zeros((1, N, Hh, d))  # every logit 0: softmax weights 1/S
    off = rng.normal(0, 0.8, size=(1, N, Hh, 27, 3))
    O, L = D.dsa3d_fwd(Q, K, V, off, T, H, W, 3, 3, 3)
    np.testing.assert_allclose(L, math.log(27), rtol=0, atol=1e-12)
    g = D.window_points(3, 3, 3)
    pos = D.token_coords(T, H, W)[:, None, :] + g[None] + off[0, :, 0]
    for ch in range(d):
        grid = V[0, :, 0, ch].reshape(T, H, W)
        ref = ndimage.map_coordinates(grid, pos.reshape(-1, 3).T, order=1, mode="grid-constant").reshape(N, 27)
        np.testing.assert_allclose(O[0, :, 0, ch], ref.mean(axis=1), rtol=0, atol=1e-12)


def test_one_point_window_returns_the_sampled_value():
    rng = np.random.default_rng(6)
    T, H, W, Hh, d = 2, 3, 3, 2, 5
    Q, K, V = _grid(rng, T, H, W, Hh, d)
    N = T * H * W
    O, L = D.dsa3d_fwd(Q, K, V, np.zeros((1, N, Hh, 1, 3)), T, H, W, 1, 1, 1, scale=0.3)
    np.testing.assert_allclose(O, V, rtol=0, atol=1e-12)  # softmax over one sample
    np.testing.assert_allclose(L, 0.3 * np.einsum("bnhd,bnhd->bhn", Q, K), rtol=0, atol=1e-12)


def test_query_subset_matches_the_full_forward():
    rng = np.random.default_rng(7)
    T, H, W, Hh, d = 2, 3, 4, 2, 4
    Q, K, V = _grid(rng, T, H, W, Hh, d)
    N = T * H * W
    off = rng.normal(0, 1.0, size=(1, N, Hh, 27, 3))
    O, L = D.dsa3d_fwd(Q, K, V, off, T, H, W, 3, 3, 3)
    toks = [0, 5, 23, 11]
    Os, Ls = D.dsa3d_fwd(Q, K, V, off, T, H, W, 3, 3, 3, tokens=toks)
    np.testing.assert_array_equal(Os, O[:, toks])
    np.testing.assert_array_equal(Ls, L[:, :, toks])
    Ot, Lt = D.dsa3d_fwd(Q, K, V, off[:, toks], T, H, W, 3, 3, 3, tokens=toks, offsets_of_tokens=True)
    np.testing.assert_array_equal(Ot, Os)
    np.testing.assert_array_equal(Lt, Ls)


def test_offsets_network_matches_scipy_correlation_and_a_matmul():
    ndimage = pytest.importorskip("scipy.ndimage")
    rng = np.random.default_rng(8)
    T, H, W, Hh, d, S = 3, 4, 5, 2, 3, 27
    N = T * H * W
    Q = rng.standard_normal((1, N, Hh, d))
    Wc = rng.standard_normal((Hh, d, 3, 3, 3))
    bc = rng.standard_normal((Hh, d))
    Wl = rng.standard_normal((Hh, d, 3 * S))
    bl = rng.standard_normal((Hh, 3 * S))
    got = D.dsa3d_offsets(Q, Wc, bc, Wl, bl, T, H, W)
    for h in range(Hh):
        Y = np.stack([ndimage.correlate(Q[0, :, h, c].reshape(T, H, W), Wc[h, c], mode="constant", cval=0.0)
                      for c in range(d)], axis=-1).reshape(N, d) + bc[h]
        ref = (Y @ Wl[h] + bl[h]).reshape(N, S, 3)
        np.testing.assert_allclose(got[0, :, h], ref, rtol=0, atol=1e-10)
    # a centre-tap-only kernel with identity-like weights moves the query values straight into offsets
    Wc2 = np.zeros_like(Wc)
    Wc2[:, :, 1, 1, 1] = 1.0
    Wl2 = np.zeros((Hh, d, 3 * S))
    Wl2[:, 0, 0] = 1.0  # dt of sample 0 = channel 0
    got2 = D.dsa3d_offsets(Q, Wc2, np.zeros((Hh, d)), Wl2, np.zeros((Hh, 3 * S)), T, H, W)
    np.testing.assert_array_equal(got2[0, :, :, 0, 0], Q[0, :, :, 0])
    assert np.all(got2[0, :, :, 1:] == 0.0) and np.all(got2[0, :, :, 0, 1:] == 0.0)


def test_offsets_of_a_token_subset_match_all_tokens():
    rng = np.random.default_rng(9)
    T, H, W, Hh, d, S = 2, 3, 4, 2, 3, 9
    N = T * H * W
    Q = rng.standard_normal((2, N, Hh, d))
    Wc, bc = rng.standard_normal((Hh, d, 3, 3, 3)), rng.standard_normal((Hh, d))
    Wl, bl = rng.standard_normal((Hh, d, 3 * S)), rng.standard_normal((Hh, 3 * S))
    full = D.dsa3d_offsets(Q, Wc, bc, Wl, bl, T, H, W)
    toks = [23, 0, 7, 12]
    np.testing.assert_allclose(D.dsa3d_offsets(Q, Wc, bc, Wl, bl, T, H, W, tokens=toks), full[:, toks],
                               rtol=0, atol=1e-12)


def _torch_dsa3d(Q, K, V, off, T, H, W, kt, kh, kw, scale):
    """The forward written with torch's grid_sample (trilinear, zero padding, corner-aligned grid): an
    independent statement of readings D1-D4 whose autograd gives the gradients."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, N, Hh, d = Q.shape
    g = torch.as_tensor(D.window_points(kt, kh, kw))
    p = torch.as_tensor(D.token_coords(T, H, W))
    O = torch.zeros(B, N, Hh, d, dtype=torch.float64)
    outs = []
    for b in range(B):
        for h in range(Hh):
            pos = p[:, None, :] + g[None] + off[b, :, h]  # [N, S, 3] as (t, h, w)
            grid = torch.stack([2 * pos[..., 2] / (W - 1) - 1, 2 * pos[..., 1] / (H - 1) - 1,
                                2 * pos[..., 0] / (T - 1) - 1], dim=-1)[None, :, :, None, :]
            vol = lambda X: X[b, :, h, :].reshape(T, H, W, d).permute(3, 0, 1, 2)[None]
            ks = F.grid_sample(vol(K), grid, mode="bilinear", padding_mode="zeros", align_corners=True)
            vs = F.grid_sample(vol(V), grid, mode="bilinear", padding_mode="zeros", align_corners=True)
            ks, vs = ks[0, :, :, :, 0].permute(1, 2, 0), vs[0, :, :, :, 0].permute(1, 2, 0)  # [N, S, d]
            a = scale * torch.einsum("nd,nsd->ns", Q[b, :, h, :], ks)
            outs.append(((b, h), torch.einsum("ns,nsd->nd", torch.softmax(a, dim=1), vs)))
    for (b, h), o in outs:
        O = O.index_put((torch.tensor(b), torch.arange(N), torch.tensor(h)), o)
    return O


def test_backward_matches_torch_autograd_through_grid_sample():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    T, H, W, Hh, d = 3, 4, 5, 2, 6
    N = T * H * W
    Q, K, V, dO = (rng.standard_normal((1, N, Hh, d)) for _ in range(4))
    off = rng.normal(0, 0.8, size=(1, N, Hh, 27, 3))
    scale = 0.45
    dQ, dK, dV, doff = D.dsa3d_bwd(Q, K, V, off, dO, T, H, W, 3, 3, 3, scale=scale)
    tQ, tK, tV, toff = (torch.tensor(x, requires_grad=True) for x in (Q, K, V, off))
    O = _torch_dsa3d(tQ, tK, tV, toff, T, H, W, 3, 3, 3, scale)
    Or, _ = D.dsa3d_fwd(Q, K, V, off, T, H, W, 3, 3, 3, scale=scale)
    np.testing.assert_allclose(O.detach().numpy(), Or, rtol=0, atol=1e-12)  # the same forward
    (O * torch.tensor(dO)).sum().backward()
    for name, got, ref in (("dQ", dQ, tQ.grad), ("dK", dK, tK.grad), ("dV", dV, tV.grad), ("doff", doff, toff.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-10, err_msg=name)


def test_offset_gradient_matches_finite_differences():
    rng = np.random.default_rng(11)
    T, H, W, Hh, d = 2, 3, 4, 1, 4
    N = T * H * W
    Q, K, V, dO = (rng.standard_normal((1, N, Hh, d)) for _ in range(4))
    off = rng.normal(0, 0.6, size=(1, N, Hh, 9, 3))
    _, _, _, doff = D.dsa3d_bwd(Q, K, V, off, dO, T, H, W, 1, 3, 3)
    eps = 1e-6
    for (n, s, ax) in [(0, 0, 0), (5, 4, 1), (11, 8, 2), (23, 3, 2), (17, 6, 0)]:
        e = np.zeros_like(off)
        e[0, n, 0, s, ax] = eps
        Op, _ = D.dsa3d_fwd(Q, K, V, off + e, T, H, W, 1, 3, 3)
        Om, _ = D.dsa3d_fwd(Q, K, V, off - e, T, H, W, 1, 3, 3)
        fd = float(((Op - Om) * dO).sum() / (2 * eps))
        assert abs(fd - doff[0, n, 0, s, ax]) <= 1e-6 * max(1.0, abs(fd)), (n, s, ax, fd, doff[0, n, 0, s, ax])


def test_offset_network_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    T, H, W, Hh, d, S = 3, 4, 5, 2, 3, 9
    N = T * H * W
    Q = rng.standard_normal((2, N, Hh, d))
    Wc, bc = rng.standard_normal((Hh, d, 3, 3, 3)), rng.standard_normal((Hh, d))
    Wl, bl = rng.standard_normal((Hh, d, 3 * S)), rng.standard_normal((Hh, 3 * S))
    G = rng.standard_normal((2, N, Hh, S, 3))
    dQ, dWc, dbc, dWl, dbl = D.dsa3d_offsets_bwd(Q, Wc, bc, Wl, bl, G, T, H, W)
    tQ, tWc, tbc, tWl, tbl = (torch.tensor(x, requires_grad=True) for x in (Q, Wc, bc, Wl, bl))
    loss = 0
    for h in range(Hh):
        X = tQ[:, :, h, :].reshape(2, T, H, W, d).permute(0, 4, 1, 2, 3)  # [B, d, T, H, W]
        Y = torch.nn.functional.conv3d(X, tWc[h][:, None], tbc[h], padding=1, groups=d)
        off = Y.permute(0, 2, 3, 4, 1).reshape(2, N, d) @ tWl[h] + tbl[h]
        loss = loss + (off * torch.tensor(G[:, :, h].reshape(2, N, 3 * S))).sum()
    loss.backward()
    for name, got, ref in (("dQ", dQ, tQ.grad), ("dWc", dWc, tWc.grad), ("dbc", dbc, tbc.grad),
                           ("dWl", dWl, tWl.grad), ("dbl", dbl, tbl.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-9, err_msg=name)


def test_backward_of_a_token_subset_matches_all_tokens():
    """The subset mode only selects: dQ and d_offsets of the chosen tokens are the full call's rows, and dK, dV
    of chosen rows are the full call's when every token that reaches them is selected, and less when not."""
    rng = np.random.default_rng(14)
    T, H, W, Hh, d = 6, 9, 14, 2, 4
    N = T * H * W
    Q, K, V, dO = (rng.standard_normal((2, N, Hh, d)) for _ in range(4))
    off = rng.normal(0, 0.4, size=(2, N, Hh, 27, 3))
    full = D.dsa3d_bwd(Q, K, V, off, dO, T, H, W, 3, 3, 3)
    toks = np.sort(rng.choice(N, 37, replace=False))
    sub = D.dsa3d_bwd(Q, K, V, off, dO, T, H, W, 3, 3, 3, tokens=toks)
    np.testing.assert_allclose(sub[0], full[0][:, toks], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sub[3], full[3][:, toks], rtol=0, atol=1e-12)
    rows = np.array([0, 417, N - 1])
    near = reaching_tokens(rows, off, T, H, W, 3, 3, 3)
    assert len(near) < N
    part = D.dsa3d_bwd(Q, K, V, off, dO, T, H, W, 3, 3, 3, tokens=near, rows=rows)
    np.testing.assert_allclose(part[1], full[1][:, rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(part[2], full[2][:, rows], rtol=0, atol=1e-12)
    few = D.dsa3d_bwd(Q, K, V, off, dO, T, H, W, 3, 3, 3, tokens=near[::2], rows=rows)
    assert np.abs(few[2] - full[2][:, rows]).max() > 1e-3  # half the reaching tokens miss part of dV
