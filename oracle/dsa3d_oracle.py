"""Oracle for 3D deformable sliding attention: a plain, slow, fp64 CPU statement.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
call it.  It shares no code with the CUDA path.

What it follows: "MegaSlide-DiT" (gist.science explainer), section 2 "3D
deformable sliding attention (3D-DSA)": each token attends to keys and values
sampled in a local kt x kh x kw space-time neighbourhood rather than to the
whole sequence; the sampling points are moved by offsets that a light 3D
convolution followed by a linear layer predicts from the input; the samples
are taken by trilinear interpolation; the cost is linear in the number of
tokens for a fixed window.

Readings taken where the page is silent (each is restated in the design notes):

D1. The window sizes kt, kh, kw are odd; the S = kt kh kw base points of token
    (t, h, w) are (t + a, h + b, w + c) for a in -(kt-1)/2 .. (kt-1)/2 (and so
    on), in (a, b, c) raster order.
D2. The offsets are predicted per head from that head's queries: a depthwise
    3 x 3 x 3 convolution over the token grid (zero padding, per-channel bias),
    then a linear layer from d channels to 3 S outputs (with bias), giving one
    (dt, dh, dw) offset per sampling point, in token units.
D3. Sampling point s of token n is p_n + g_s + offset_{n,s}.  Keys and values
    there are the trilinear interpolation of the grid's K and V rows; grid
    points outside the T x H x W raster count as zero vectors (zero padding),
    so a sample wholly outside the grid has k = v = 0 and still takes part in
    the softmax with logit 0.  A sampling point with a non-finite coordinate
    counts as wholly outside.
D4. Attention over the S samples of a token: logits scale * q . k_s (scale
    1/sqrt(d) unless given), softmax over s, O = sum_s softmax_s v_s, and the
    natural-log log-sum-exp of the logits, per (batch, head, token).
"""
from __future__ import annotations

import math

import numpy as np


def window_points(kt, kh, kw):
    """Base offsets g_s of the window (reading D1), shape [S, 3] in (t, h, w) order."""
    for k in (kt, kh, kw):
        if k < 1 or k % 2 == 0:
            raise ValueError("window sizes must be odd and positive")
    pts = []
    for a in range(kt):
        for b in range(kh):
            for c in range(kw):
                pts.append((a - (kt - 1) // 2, b - (kh - 1) // 2, c - (kw - 1) // 2))
    return np.asarray(pts, dtype=np.float64)


def token_coords(T, H, W):
    """(t, h, w) of every raster token n = (t H + h) W + w, shape [N, 3]."""
    t, h, w = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    return np.stack([t.ravel(), h.ravel(), w.ravel()], axis=1).astype(np.float64)


def dsa3d_offsets(Q, Wc, bc, Wl, bl, T, H, W, tokens=None):
    """Offsets of every sampling point (reading D2).

    Q: [B, N, Hh, d] with N = T H W in raster order; Wc: [Hh, d, 3, 3, 3]
    (depthwise kernel, taps in (dt, dh, dw) order, centre at [1, 1, 1]);
    bc: [Hh, d]; Wl: [Hh, d, 3 S]; bl: [Hh, 3 S].
    Returns [B, Nq, Hh, S, 3] fp64: Y = conv(Q_h) + bc, offsets = Y Wl[h] + bl[h],
    for every token or, when given, only the raster indices `tokens`.
    """
    Q = np.asarray(Q, dtype=np.float64)
    B, N, Hh, d = Q.shape
    assert N == T * H * W
    S3 = Wl.shape[2]
    toks = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)
    p = token_coords(T, H, W)[toks].astype(np.int64)
    out = np.empty((B, len(toks), Hh, S3 // 3, 3))
    for h in range(Hh):
        Y = np.broadcast_to(np.asarray(bc[h], dtype=np.float64), (B, len(toks), d)).copy()
        for a in range(3):
            for b in range(3):
                for c in range(3):
                    t, y, x = p[:, 0] + a - 1, p[:, 1] + b - 1, p[:, 2] + c - 1
                    inside = (t >= 0) & (t < T) & (y >= 0) & (y < H) & (x >= 0) & (x < W)
                    m = np.where(inside, (t * H + y) * W + x, 0)
                    Y += np.where(inside[None, :, None], Q[:, m, h, :], 0.0) * np.asarray(Wc[h, :, a, b, c],
                                                                                          dtype=np.float64)
        off = Y @ np.asarray(Wl[h], dtype=np.float64) + np.asarray(bl[h], dtype=np.float64)
        out[:, :, h] = off.reshape(B, len(toks), S3 // 3, 3)
    return out


def trilinear(X, pos, T, H, W):
    """Trilinear interpolation of grid rows (reading D3).

    X: [N, d] rows of one (batch, head) in raster order; pos: [..., 3] fractional
    (t, h, w) positions.  Each of the 8 surrounding grid points weighs the product
    of (1 - |distance|) along the three axes; points outside the raster are zero
    rows.  Returns [..., d].
    """
    pos = np.asarray(pos, dtype=np.float64)
    # a position with a non-finite coordinate lies outside the raster (reading D3)
    pos = np.where(np.isfinite(pos).all(axis=-1, keepdims=True), pos, -2.0)
    base = np.floor(pos)
    frac = pos - base
    out = np.zeros(pos.shape[:-1] + (X.shape[1],))
    for ct in (0, 1):
        for ch in (0, 1):
            for cw in (0, 1):
                t = base[..., 0] + ct
                h = base[..., 1] + ch
                w = base[..., 2] + cw
                wt = np.where(ct, frac[..., 0], 1.0 - frac[..., 0])
                wh = np.where(ch, frac[..., 1], 1.0 - frac[..., 1])
                ww = np.where(cw, frac[..., 2], 1.0 - frac[..., 2])
                inside = (t >= 0) & (t < T) & (h >= 0) & (h < H) & (w >= 0) & (w < W)
                n = np.where(inside, (t * H + h) * W + w, 0).astype(np.int64)
                out += (np.where(inside, wt * wh * ww, 0.0))[..., None] * X[n]
    return out


def dsa3d_fwd(Q, K, V, offsets, T, H, W, kt, kh, kw, scale=None, tokens=None, offsets_of_tokens=False):
    """3D deformable sliding attention forward (readings D1, D3, D4).

    Q, K, V: [B, N, Hh, d]; offsets: [B, N, Hh, S, 3] (or [B, Nq, Hh, S, 3], the
    selected tokens' rows only, with offsets_of_tokens).  Returns (O [B, Nq, Hh, d],
    LSE [B, Hh, Nq]) fp64, Nq = N, or the number of `tokens` when only those
    query tokens (raster indices) are wanted.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.float64)
    B, N, Hh, d = Q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    g = window_points(kt, kh, kw)
    toks = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)
    p = token_coords(T, H, W)[toks]
    O = np.zeros((B, len(toks), Hh, d))
    L = np.zeros((B, Hh, len(toks)))
    chunk = 256
    for b in range(B):
        for h in range(Hh):
            for c0 in range(0, len(toks), chunk):
                sl = slice(c0, c0 + chunk)
                orow = offsets[b, sl, h] if offsets_of_tokens else offsets[b, toks[sl], h]
                pos = p[sl, None, :] + g[None, :, :] + orow  # [n, S, 3]
                ks = trilinear(K[b, :, h, :], pos, T, H, W)
                vs = trilinear(V[b, :, h, :], pos, T, H, W)
                logit = scale * np.einsum("nd,nsd->ns", Q[b, toks[sl], h, :], ks)
                m = logit.max(axis=1, keepdims=True)
                e = np.exp(logit - m)
                z = e.sum(axis=1, keepdims=True)
                O[b, sl, h, :] = np.einsum("ns,nsd->nd", e / z, vs)
                L[b, h, sl] = (m + np.log(z))[:, 0]
    return O, L


# --------------------------------------------------------------------------- backward
# D5. The backward differentiates readings D1-D4 as written, with dLSE = 0 (the loss reaches the
#     attention through O): for every token n and window point s, with k~_s, v~_s the sampled rows,
#     a_s = scale q.k~_s, P = softmax(a), dP_s = dO.v~_s and da_s = P_s (dP_s - sum_u P_u dP_u):
#       dq_n = scale sum_s da_s k~_s,
#       dK[m] += w_c scale da_s q_n and dV[m] += w_c P_s dO_n for every corner c (row m, weight w_c) of
#       every sample inside the raster,
#       d offset_s = sum_c (d w_c / d pos) (scale da_s q.K[m_c] + P_s dO.V[m_c]),
#     where d w_c / d pos along an axis is -1 or +1 (lower or upper neighbour on that axis) times the
#     other two axes' weights: the derivative of the interpolation at a position off the integer grid
#     (on the grid, the one-sided derivative from above, as floor() sees it).  The offset network's
#     backward follows from D2: dY = d offsets Wl^T, dWl = Y^T d offsets, dbl = sum d offsets,
#     dWc[c, tap] = sum_n dY[n, c] Q[n + tap, c], dbc = sum_n dY, and dQ += the transposed convolution
#     of dY (zero padding).


def _corners(pos, T, H, W):
    """The 8 trilinear corners of every position: (row index, inside, weight, d weight / d (t, h, w))."""
    pos = np.where(np.isfinite(pos).all(axis=-1, keepdims=True), pos, -2.0)
    base = np.floor(pos)
    f = pos - base
    out = []
    for ct in (0, 1):
        for ch in (0, 1):
            for cw in (0, 1):
                t = base[..., 0] + ct
                h = base[..., 1] + ch
                w = base[..., 2] + cw
                wt = np.where(ct, f[..., 0], 1.0 - f[..., 0])
                wh = np.where(ch, f[..., 1], 1.0 - f[..., 1])
                ww = np.where(cw, f[..., 2], 1.0 - f[..., 2])
                st, sh, sw = (1.0 if ct else -1.0), (1.0 if ch else -1.0), (1.0 if cw else -1.0)
                inside = (t >= 0) & (t < T) & (h >= 0) & (h < H) & (w >= 0) & (w < W)
                n = np.where(inside, (t * H + h) * W + w, 0).astype(np.int64)
                m = inside.astype(np.float64)
                dw = np.stack([st * wh * ww, sh * wt * ww, sw * wt * wh], axis=-1) * m[..., None]
                out.append((n, inside, wt * wh * ww * m, dw))
    return out


def dsa3d_bwd(Q, K, V, offsets, dO, T, H, W, kt, kh, kw, scale=None, tokens=None, rows=None):
    """Gradients of 3D deformable sliding attention (reading D5).

    Q, K, V, dO: [B, N, Hh, d]; offsets: [B, N, Hh, S, 3].  Returns (dQ, dK, dV [B, N, Hh, d],
    d_offsets [B, N, Hh, S, 3]) fp64; dQ is the attention's part only.

    tokens (sorted raster indices) restricts the work to those tokens: dQ and d_offsets then hold their rows
    only, and dK, dV hold, for the raster rows `rows` (sorted; default: tokens), the sum over the selected
    tokens' samples alone.  A row's dK, dV are its full value when every token whose samples touch it is
    selected.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.float64)
    B, N, Hh, d = Q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    g = window_points(kt, kh, kw)
    p = token_coords(T, H, W)
    toks = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)
    rows = toks if rows is None else np.asarray(rows, dtype=np.int64)
    dQ = np.zeros((B, len(toks), Hh, d))
    dK = np.zeros((B, len(rows), Hh, d))
    dV = np.zeros((B, len(rows), Hh, d))
    doff = np.zeros((B, len(toks)) + offsets.shape[2:])
    chunk = 256
    for b in range(B):
        for h in range(Hh):
            Kh, Vh = K[b, :, h, :], V[b, :, h, :]
            for c0 in range(0, len(toks), chunk):
                sl = slice(c0, min(len(toks), c0 + chunk))
                tk = toks[sl]
                q, do = Q[b, tk, h, :], dO[b, tk, h, :]
                pos = p[tk, None, :] + g[None, :, :] + offsets[b, tk, h]  # [n, S, 3]
                cs = _corners(pos, T, H, W)
                ks = sum(w[..., None] * Kh[n] for n, _, w, _ in cs)  # [n, S, d]
                vs = sum(w[..., None] * Vh[n] for n, _, w, _ in cs)
                a = scale * np.einsum("nd,nsd->ns", q, ks)
                P = np.exp(a - a.max(axis=1, keepdims=True))
                P /= P.sum(axis=1, keepdims=True)
                dP = np.einsum("nd,nsd->ns", do, vs)
                da = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dQ[b, sl, h, :] = scale * np.einsum("ns,nsd->nd", da, ks)
                for n, inside, w, dw in cs:
                    gk = (w * scale * da)[..., None] * q[:, None, :]  # [n, S, d]
                    gv = (w * P)[..., None] * do[:, None, :]
                    r = np.minimum(np.searchsorted(rows, n), len(rows) - 1)  # the corner row's place in rows
                    hit = inside & (rows[r] == n)
                    np.add.at(dK[b, :, h, :], r[hit], gk[hit])
                    np.add.at(dV[b, :, h, :], r[hit], gv[hit])
                    qk = np.einsum("nd,nsd->ns", q, Kh[n])
                    dv = np.einsum("nd,nsd->ns", do, Vh[n])
                    doff[b, sl, h] += dw * (scale * da * qk + P * dv)[..., None]
    return dQ, dK, dV, doff


def dsa3d_offsets_bwd(Q, Wc, bc, Wl, bl, d_offsets, T, H, W):
    """Gradients of the offset network (reading D5): (dQ_net [B, N, Hh, d], dWc, dbc, dWl, dbl) fp64."""
    Q = np.asarray(Q, dtype=np.float64)
    B, N, Hh, d = Q.shape
    S3 = Wl.shape[2]
    X = Q.reshape(B, T, H, W, Hh, d)
    Xp = np.zeros((B, T + 2, H + 2, W + 2, Hh, d))
    Xp[:, 1:-1, 1:-1, 1:-1] = X
    dQ = np.zeros((B, T + 2, H + 2, W + 2, Hh, d))
    dWc = np.zeros((Hh, d, 3, 3, 3))
    dbc = np.zeros((Hh, d))
    dWl = np.zeros((Hh, d, S3))
    dbl = np.zeros((Hh, S3))
    for h in range(Hh):
        Y = np.broadcast_to(np.asarray(bc[h], dtype=np.float64), (B, T, H, W, d)).copy()
        for a in range(3):
            for b_ in range(3):
                for c in range(3):
                    Y += Xp[:, a:a + T, b_:b_ + H, c:c + W, h, :] * np.asarray(Wc[h, :, a, b_, c], dtype=np.float64)
        G = np.asarray(d_offsets[:, :, h], dtype=np.float64).reshape(B, N, S3)
        Yf = Y.reshape(B, N, d)
        dWl[h] = np.einsum("bnd,bnj->dj", Yf, G)
        dbl[h] = G.sum(axis=(0, 1))
        dY = (G @ np.asarray(Wl[h], dtype=np.float64).T).reshape(B, T, H, W, d)
        dbc[h] = dY.sum(axis=(0, 1, 2, 3))
        for a in range(3):
            for b_ in range(3):
                for c in range(3):
                    dWc[h, :, a, b_, c] = (dY * Xp[:, a:a + T, b_:b_ + H, c:c + W, h, :]).sum(axis=(0, 1, 2, 3))
                    dQ[:, a:a + T, b_:b_ + H, c:c + W, h, :] += dY * np.asarray(Wc[h, :, a, b_, c], dtype=np.float64)
    return dQ[:, 1:-1, 1:-1, 1:-1].reshape(B, N, Hh, d), dWc, dbc, dWl, dbl
