"""Pins for the CPU oracle: checks against facts the pages and the mathematics fix, not against itself.

Each test targets a step of the oracle with something independent of it: a
closed form, a library routine (torch's scaled-dot-product attention and
autograd in fp64, torch's bfloat16 conversion), brute-force enumeration,
finite differences or an exact invariant.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
from dynamic_block_sparse_rank_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(tok):
    tok = tok.strip()
    if tok == "-inf":
        return -math.inf
    if tok.startswith("ln"):
        return math.log(float(tok[2:]))
    return float(tok)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            vals[k.strip()] = v.strip()
    return vals


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _block_id_brute(geom):
    """Block id of every raster token from integer division alone (t-major tile numbering)."""
    ids = np.empty(geom.N, dtype=np.int64)
    for t in range(geom.T):
        for h in range(geom.H):
            for w in range(geom.W):
                ids[(t * geom.H + h) * geom.W + w] = ((t // geom.bt) * geom.nH + h // geom.bh) * geom.nW + w // geom.bw
    return ids


def _sdpa(Q, K, V, mask, scale):
    """torch fp64 scaled-dot-product attention per head; mask[i, j] True = attend. Returns O, LSE."""
    q = torch.from_numpy(np.ascontiguousarray(np.transpose(Q, (0, 2, 1, 3))))
    k = torch.from_numpy(np.ascontiguousarray(np.transpose(K, (0, 2, 1, 3))))
    v = torch.from_numpy(np.ascontiguousarray(np.transpose(V, (0, 2, 1, 3))))
    m = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~m, -math.inf), dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


# ------------------------------------------------------------------ rounding, k, geometry
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-5, 5, 20000)
    # exact half-way cases between adjacent bf16 values, both parities
    base = torch.tensor(rng.standard_normal(2000), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    ulp = np.abs(base) * 2.0 ** -7
    ties = np.concatenate([base + 0.5 * np.ldexp(1.0, np.frexp(base)[1] - 8), base - 0.5 * ulp]).astype(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1.0, -3.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(orc.to_bf16(x.astype(np.float64)), want)
    assert np.array_equal(inputs.round_to_bf16(x).astype(np.float64), want)


@pytest.mark.parametrize("keep,nb,k", [(0.5, 4, 2), (0.10, 64, 6), (0.05, 480, 24), (0.05, 4096, 204),
                                       (0.10, 1144, 114), (0.29, 100, 29), (1e-6, 50, 1), (1.0, 7, 7),
                                       (2.0, 7, 7)])
def test_keep_count(keep, nb, k):
    assert orc.keep_count(keep, nb) == k


@pytest.mark.parametrize("dims", [(4, 8, 8, 1, 8, 8), (21, 60, 104, 2, 8, 8), (3, 5, 7, 2, 2, 3)])
def test_geometry_partitions_grid(dims):
    geom = orc.Geometry(*dims)
    ids = _block_id_brute(geom)
    seen = np.zeros(geom.N, dtype=np.int64)
    for I in range(geom.n_blocks):
        toks = geom.tokens(I)
        assert np.all(ids[toks] == I)
        seen[toks] += 1
        # (tt, hh, ww) order inside the tile is raster order of the tile's tokens
        assert np.all(np.diff(toks) > 0)
    assert np.all(seen == 1)


def test_geometry_ragged_counts():
    geom = orc.Geometry(21, 60, 104, 2, 8, 8)
    sizes = np.array([len(geom.tokens(I)) for I in range(geom.n_blocks)])
    assert geom.n_blocks == 11 * 8 * 13
    assert (sizes == 128).sum() == 910 and (sizes == 64).sum() == 221 and (sizes == 32).sum() == 13


# ------------------------------------------------------------------ forward
def test_golden_two_key_attention():
    g = _read_golden("two_key_attention.txt")
    vec = lambda k: np.array([_num(t) for t in g[k].split()])
    geom = orc.Geometry(1, 1, 2, 1, 1, 1)
    Q = np.stack([vec("q0"), vec("q1")])[None, :, None, :]
    K = np.stack([vec("k0"), vec("k1")])[None, :, None, :]
    V = np.stack([vec("v0"), vec("v1")])[None, :, None, :]
    idx = np.array([[[[0, 1], [0, 1]]]], dtype=np.int32)
    O, L = orc.attn_fwd(Q, K, V, idx, geom, scale=1.0)
    assert np.allclose(O[0, 0, 0], vec("O0"), atol=1e-14) and np.allclose(O[0, 1, 0], vec("O1"), atol=1e-14)
    assert abs(L[0, 0, 0] - _num(g["LSE0"])) < 1e-14 and abs(L[0, 0, 1] - _num(g["LSE1"])) < 1e-14


@pytest.mark.parametrize("dims", [(2, 4, 4, 1, 2, 2), (3, 5, 7, 2, 2, 3)])
def test_keep_all_equals_dense_softmax(dims):
    geom = orc.Geometry(*dims)
    B, Hh, d = 1, 2, 8
    Q, K, V = (_rand((B, geom.N, Hh, d), s) for s in (1, 2, 3))
    idx = np.broadcast_to(np.arange(geom.n_blocks, dtype=np.int32), (B, Hh, geom.n_blocks, geom.n_blocks))
    O, L = orc.attn_fwd(Q, K, V, idx, geom)
    mask = np.ones((geom.N, geom.N), dtype=bool)
    Oref, Lref = _sdpa(Q, K, V, mask, 1 / math.sqrt(d))
    assert np.abs(O - Oref).max() < 1e-12 and np.abs(L - Lref).max() < 1e-12
    # an independent plain softmax as well
    for h in range(Hh):
        S = Q[0, :, h] @ K[0, :, h].T / math.sqrt(d)
        P = np.exp(S - S.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        assert np.abs(P @ V[0, :, h] - O[0, :, h]).max() < 1e-12


def _random_map(geom, B, Hh, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.empty((B, Hh, geom.n_blocks, k), dtype=np.int32)
    for b in range(B):
        for h in range(Hh):
            for I in range(geom.n_blocks):
                idx[b, h, I] = np.sort(rng.choice(geom.n_blocks, k, replace=False))
    return idx


def _mask_from_map(geom, idx_bh):
    ids = _block_id_brute(geom)
    mask = np.zeros((geom.N, geom.N), dtype=bool)
    for i in range(geom.N):
        mask[i] = np.isin(ids, idx_bh[ids[i]])
    return mask


@pytest.mark.parametrize("dims,k", [((2, 4, 4, 1, 2, 2), 3), ((3, 5, 7, 2, 2, 3), 2)])
def test_sparse_forward_equals_masked_sdpa(dims, k):
    geom = orc.Geometry(*dims)
    B, Hh, d = 1, 2, 6
    Q, K, V = (_rand((B, geom.N, Hh, d), s, 2.0) for s in (4, 5, 6))
    idx = _random_map(geom, B, Hh, k, 7)
    O, L = orc.attn_fwd(Q, K, V, idx, geom)
    for h in range(Hh):
        mask = _mask_from_map(geom, idx[0, h])
        Oref, Lref = _sdpa(Q[:, :, h:h + 1], K[:, :, h:h + 1], V[:, :, h:h + 1], mask, 1 / math.sqrt(d))
        assert np.abs(O[:, :, h:h + 1] - Oref).max() < 1e-12
        assert np.abs(L[:, h:h + 1] - Lref).max() < 1e-12


def test_forward_row_facts():
    geom = orc.Geometry(2, 4, 4, 1, 2, 2)
    Q, K, V = (_rand((1, geom.N, 1, 4), s, 3.0) for s in (8, 9, 10))
    idx = _random_map(geom, 1, 1, 2, 11)
    O, L = orc.attn_fwd(Q, K, V, idx, geom)
    for I in range(geom.n_blocks):
        keys = np.concatenate([geom.tokens(J) for J in idx[0, 0, I]])
        for i in geom.tokens(I):
            s = Q[0, i, 0] @ K[0, keys, 0].T / 2.0
            assert L[0, 0, i] >= s.max() - 1e-15  # LSE bounds the row max
            assert abs(np.exp(s - L[0, 0, i]).sum() - 1.0) < 1e-13  # P rows sum to one


def test_single_token_block_returns_v():
    geom = orc.Geometry(1, 1, 3, 1, 1, 1)
    Q, K, V = (_rand((1, 3, 1, 5), s) for s in (12, 13, 14))
    idx = np.array([[[[2], [0], [1]]]], dtype=np.int32)
    O, L = orc.attn_fwd(Q, K, V, idx, geom)
    for i, j in enumerate([2, 0, 1]):
        assert np.array_equal(O[0, i, 0], V[0, j, 0])
        assert abs(L[0, 0, i] - Q[0, i, 0] @ K[0, j, 0] / math.sqrt(5)) < 1e-14


def test_empty_range_and_inactive_blocks():
    geom = orc.Geometry(2, 4, 4, 1, 2, 2)
    Q, K, V = (_rand((1, geom.N, 1, 4), s) for s in (15, 16, 17))
    idx = np.broadcast_to(np.array([0, 1], dtype=np.int32), (1, 1, geom.n_blocks, 2))
    O, L = orc.attn_fwd(Q, K, V, idx, geom, kb_begin=4, kb_end=8)
    assert np.all(O == 0) and np.all(np.isneginf(L))
    act = np.zeros(geom.n_blocks, dtype=bool)
    act[3] = True
    O2, L2 = orc.attn_fwd(Q, K, V, idx, geom, qb_active=act)
    rows = geom.tokens(3)
    assert np.all(np.isfinite(O2[0, rows])) and np.isnan(O2[0, geom.tokens(0)]).all()


# ------------------------------------------------------------------ merge
def test_golden_merge():
    g = _read_golden("merge_states.txt")
    for r in ("row0", "row1"):
        lse = [_num(t) for t in g[r + "_lse"].split()]
        os_ = [np.array([_num(t) for t in part.split()]) for part in g[r + "_o"].split("|")]
        O, L = orc.merge_states([o[None] for o in os_], [np.array([x]) for x in lse])
        want_l = _num(g[r + "_expect_lse"])
        want_o = np.array([_num(t) for t in g[r + "_expect_o"].split()])
        assert (np.isneginf(L[0]) and np.isneginf(want_l)) or abs(L[0] - want_l) < 1e-14
        assert np.allclose(O[0], want_o, atol=1e-14)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_of_partitions_equals_union(seed):
    rng = np.random.default_rng(seed)
    geom = orc.Geometry(3, 4, 6, 1, 2, 2)
    B, Hh, d = 1, 2, 5
    Q, K, V = (_rand((B, geom.N, Hh, d), seed * 10 + s, 2.0) for s in range(3))
    k = 5
    idx = _random_map(geom, B, Hh, k, seed)
    full_O, full_L = orc.attn_fwd(Q, K, V, idx, geom)
    cuts = np.sort(rng.integers(0, geom.n_blocks + 1, size=4))  # uneven, possibly empty parts
    bounds = list(zip([0, *cuts], [*cuts, geom.n_blocks]))
    states = [orc.attn_fwd(Q, K, V, idx, geom, kb_begin=b0, kb_end=b1) for b0, b1 in bounds]
    Ls = [np.transpose(L, (0, 2, 1)) for _, L in states]
    O, L = orc.merge_states([s[0] for s in states], Ls)
    assert np.abs(O - full_O).max() < 1e-12
    assert np.abs(np.transpose(L, (0, 2, 1)) - full_L).max() < 1e-12
    # order of merging does not matter (associative, commutative)
    perm = rng.permutation(len(states))
    O2, L2 = orc.merge_states([states[p][0] for p in perm], [Ls[p] for p in perm])
    a = orc.merge_states([s[0] for s in states[:2]], Ls[:2])
    O3, L3 = orc.merge_states([a[0]] + [s[0] for s in states[2:]], [a[1]] + Ls[2:])
    assert np.abs(O2 - O).max() < 1e-12 and np.abs(O3 - O).max() < 1e-12
    assert np.abs(L2 - L).max() < 1e-12 and np.abs(L3 - L).max() < 1e-12


# ------------------------------------------------------------------ predictor + top-k
def _brute_scores(qt, kt, geom):
    nb = geom.n_blocks
    ids = _block_id_brute(geom)
    s = np.full((nb, nb), -np.inf)
    for i in range(geom.N):
        for j in range(geom.N):
            v = sum(qt[i, c] * kt[j, c] for c in range(qt.shape[1]))
            if v > s[ids[i], ids[j]]:
                s[ids[i], ids[j]] = v
    return s


def _brute_select(row, k):
    best, best_sum = None, -np.inf
    for sub in itertools.combinations(range(len(row)), k):  # lexicographic order
        tot = sum(row[j] for j in sub)
        if tot > best_sum:
            best, best_sum = sub, tot
    return np.array(best, dtype=np.int32)


@pytest.mark.parametrize("dims,k,r", [((2, 4, 4, 1, 2, 2), 3, 3), ((2, 4, 4, 2, 2, 2), 2, 2), ((3, 3, 5, 2, 2, 2), 4, 2)])
def test_predictor_brute_force(dims, k, r):
    geom = orc.Geometry(*dims)
    d = 4
    Q, K = (_rand((1, geom.N, 1, d), s) for s in (20, 21))
    Wq, Wk = (_rand((1, d, r), s, 0.5) for s in (22, 23))
    keep = k / geom.n_blocks
    idx, scores = orc.predict_blocks(Q, K, Wq, Wk, geom, keep, "f32")
    qt = np.array([[sum(Q[0, i, 0, c] * Wq[0, c, a] for c in range(d)) for a in range(r)] for i in range(geom.N)])
    kt = np.array([[sum(K[0, i, 0, c] * Wk[0, c, a] for c in range(d)) for a in range(r)] for i in range(geom.N)])
    bs = _brute_scores(qt, kt, geom)
    assert np.abs(scores[0, 0] - bs).max() < 1e-12
    for I in range(geom.n_blocks):
        assert np.array_equal(idx[0, 0, I], _brute_select(bs[I], k))


def test_predictor_exact_ties_go_to_lower_index():
    geom = orc.Geometry(2, 4, 4, 1, 2, 2)  # 8 blocks of 4 tokens
    d, r = 4, 2
    rng = np.random.default_rng(3)
    Q = rng.integers(-3, 4, size=(1, geom.N, 1, d)).astype(np.float64)
    block = rng.integers(-3, 4, size=(4, d)).astype(np.float64)
    K = np.empty_like(Q)
    for J in range(geom.n_blocks):
        K[0, geom.tokens(J), 0] = block  # every key block identical -> all scores tie
    W = np.zeros((1, d, r))
    W[0, :r, :r] = np.eye(r)
    idx, scores = orc.predict_blocks(Q, K, W, W, geom, 3 / 8, "bf16")
    assert np.all(scores[0, 0] == scores[0, 0, :, :1])
    assert np.all(idx == np.array([0, 1, 2], dtype=np.int32))
    # two blocks above the rest, then a three-way tie for the last slot
    K2 = K.copy()
    K2[0, geom.tokens(6), 0] *= 2.0
    K2[0, geom.tokens(5), 0] *= 2.0
    idx2, sc2 = orc.predict_blocks(Q, K2, W, W, geom, 3 / 8, "bf16")
    for I in range(geom.n_blocks):
        row = sc2[0, 0, I]
        want = _brute_select(row, 3)
        assert np.array_equal(idx2[0, 0, I], want)


def test_rank1_closed_form():
    geom = orc.Geometry(2, 4, 6, 1, 2, 3)
    d = 3
    Q, K = (_rand((1, geom.N, 1, d), s) for s in (30, 31))
    Wq, Wk = (_rand((1, d, 1), s) for s in (32, 33))
    qt, kt = orc.project(Q, Wq, "f32"), orc.project(K, Wk, "f32")
    s = orc.block_scores(qt, kt, geom)[0, 0]
    for I in range(geom.n_blocks):
        a = qt[0, 0, geom.tokens(I), 0]
        for J in range(geom.n_blocks):
            c = kt[0, 0, geom.tokens(J), 0]
            want = max(a.max() * c.max(), a.min() * c.min())
            assert abs(s[I, J] - want) < 1e-13


def test_identity_projection_gives_block_max_logits():
    geom = orc.Geometry(2, 4, 4, 1, 2, 2)
    d = 4
    Q, K = (_rand((1, geom.N, 1, d), s) for s in (34, 35))
    W = np.eye(d)[None]
    s = orc.block_scores(orc.project(Q, W, "f32"), orc.project(K, W, "f32"), geom)[0, 0]
    logits = Q[0, :, 0] @ K[0, :, 0].T
    for I in range(geom.n_blocks):
        for J in range(geom.n_blocks):
            assert abs(s[I, J] - logits[np.ix_(geom.tokens(I), geom.tokens(J))].max()) < 1e-13


def test_projection_rounds_to_bf16_for_bf16_problems():
    Q = _rand((1, 16, 2, 8), 36)
    W = _rand((2, 8, 3), 37)
    exact = np.einsum("bnhd,hdr->bhnr", Q, W)
    got = orc.project(Q, W, "bf16")
    want = torch.from_numpy(exact).float().to(torch.bfloat16).double().numpy()
    # torch rounds via fp32 first; the two agree except for rare double-rounding cases
    assert np.mean(got == want) > 0.99
    assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-300)


# ------------------------------------------------------------------ backward
def _loss(Q, K, V, dO, idx, geom):
    O, _ = orc.attn_fwd(Q, K, V, idx, geom)
    return float((O * dO).sum())


def test_backward_finite_differences():
    geom = orc.Geometry(2, 2, 4, 1, 2, 2)
    B, Hh, d = 1, 1, 3
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s) for s in (40, 41, 42, 43))
    idx = _random_map(geom, B, Hh, 2, 44)
    dQ, dK, dV = orc.attn_bwd(Q, K, V, dO, idx, geom)
    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for pos in np.ndindex(X.shape):
            x0 = X[pos]
            X[pos] = x0 + h
            lp = _loss(Q, K, V, dO, idx, geom)
            X[pos] = x0 - h
            lm = _loss(Q, K, V, dO, idx, geom)
            X[pos] = x0
            num[pos] = (lp - lm) / (2 * h)
        assert np.abs(num - G).max() <= 1e-6 * max(1.0, np.abs(G).max())


def test_backward_matches_torch_autograd():
    geom = orc.Geometry(2, 4, 4, 1, 2, 2)
    B, Hh, d = 1, 2, 4
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s, 1.5) for s in (50, 51, 52, 53))
    idx = _random_map(geom, B, Hh, 3, 54)
    dQ, dK, dV = orc.attn_bwd(Q, K, V, dO, idx, geom)
    for h in range(Hh):
        mask = torch.from_numpy(_mask_from_map(geom, idx[0, h]))
        q, k, v = (torch.tensor(X[0, :, h], requires_grad=True) for X in (Q, K, V))
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask[None])[0]
        (o * torch.from_numpy(dO[0, :, h])).sum().backward()
        assert np.abs(q.grad.numpy() - dQ[0, :, h]).max() < 1e-12
        assert np.abs(k.grad.numpy() - dK[0, :, h]).max() < 1e-12
        assert np.abs(v.grad.numpy() - dV[0, :, h]).max() < 1e-12


def test_backward_sum_invariants():
    geom = orc.Geometry(3, 4, 6, 1, 2, 2)
    B, Hh, d = 1, 2, 6
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s, 2.0) for s in (60, 61, 62, 63))
    idx = _random_map(geom, B, Hh, 4, 64)
    dQ, dK, dV = orc.attn_bwd(Q, K, V, dO, idx, geom)
    assert np.abs(dK.sum(axis=1)).max() < 1e-11
    assert np.abs(dV.sum(axis=1) - dO.sum(axis=1)).max() < 1e-11


def test_backward_blocks_agree_with_full():
    geom = orc.Geometry(2, 4, 6, 1, 2, 2)
    B, Hh, d = 1, 2, 4
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s) for s in (70, 71, 72, 73))
    idx = _random_map(geom, B, Hh, 3, 74)
    dQ, dK, dV = orc.attn_bwd(Q, K, V, dO, idx, geom)
    dq, dkv = orc.attn_bwd_blocks(Q, K, V, dO, idx, geom, query_blocks=[0, 5], key_blocks=[1, 4])
    for (b, h, I), v in dq.items():
        assert np.abs(v - dQ[b, geom.tokens(I), h]).max() < 1e-12
    for (b, h, J), (dk, dv) in dkv.items():
        assert np.abs(dk - dK[b, geom.tokens(J), h]).max() < 1e-12
        assert np.abs(dv - dV[b, geom.tokens(J), h]).max() < 1e-12


# ------------------------------------------------------------------ partitions and reuse
def test_frame_partitions_for_the_ragged_grid():
    geom = orc.Geometry(21, 60, 104, 2, 8, 8)
    per = 8 * 13
    assert orc.frame_partitions(geom, 4) == [(0, 3 * per), (3 * per, 6 * per), (6 * per, 9 * per), (9 * per, 11 * per)]
    reuse = orc.reuse_mask(geom, 4, 2)
    assert np.all(reuse.sum(axis=0) == 2)
    assert reuse[2, 0] and reuse[3, 0] and not reuse[0, 0]  # block in partition 0: far = 3, 2
    I3 = 10 * per  # in partition 3: distances 3, 2, 1, 0 -> reuse 0, 1
    assert reuse[0, I3] and reuse[1, I3]
    I1 = 4 * per  # in partition 1: distances 1, 0, 1, 2 -> reuse 3 and the lower of the tie (0)
    assert reuse[3, I1] and reuse[0, I1] and not reuse[2, I1]


def test_reuse_merge_limits():
    geom = orc.Geometry(4, 2, 4, 1, 2, 2)  # 4 slabs of 2 blocks
    B, Hh, d = 1, 1, 4
    Q, K, V = (_rand((B, geom.N, Hh, d), s) for s in (80, 81, 82))
    Qp, Kp, Vp = Q + 0.3, K - 0.2, V * 1.1
    idx = _random_map(geom, B, Hh, 4, 83)
    idxp = _random_map(geom, B, Hh, 4, 84)
    now = orc.partition_states(Q, K, V, idx, geom, 4)
    prev = orc.partition_states(Qp, Kp, Vp, idxp, geom, 4)
    O0, L0 = orc.reuse_merge(now, prev, geom, 4, 0)
    Of, Lf = orc.attn_fwd(Q, K, V, idx, geom)
    assert np.abs(O0 - Of).max() < 1e-12 and np.abs(L0 - Lf).max() < 1e-12
    O4, L4 = orc.reuse_merge(now, prev, geom, 4, 4)
    Op, Lp = orc.attn_fwd(Qp, Kp, Vp, idxp, geom)
    assert np.abs(O4 - Op).max() < 1e-12 and np.abs(L4 - Lp).max() < 1e-12


# ------------------------------------------------------------------ generator
def test_generator_is_seeded_and_head_separable():
    wl = inputs.WORKLOADS["tiny_f32_256"]
    a = inputs.generate(wl, names=("Q", "K", "V", "dO", "Wq", "Wk", "Qp"))
    b = inputs.generate(wl, names=("Q", "K", "V", "dO", "Wq", "Wk", "Qp"), threads=1)
    assert inputs.digest(a) == inputs.digest(b)
    one = inputs.generate(wl, names=("Q", "Wq"), heads=[1])
    assert np.array_equal(one["Q"][:, :, 0], a["Q"][:, :, 1]) and np.array_equal(one["Wq"][0], a["Wq"][1])
    wl16 = inputs.WORKLOADS["fwd_8k"].with_(heads=1)
    g = inputs.generate(wl16, names=("Q", "K", "Qp"))
    assert np.array_equal(inputs.round_to_bf16(g["Q"]), g["Q"])
    # Q and K share the field: their correlation is A^2 / (A^2 + 1) = 0.9 for A = 3
    q, k = g["Q"].ravel().astype(np.float64), g["K"].ravel().astype(np.float64)
    assert abs(np.corrcoef(q, k)[0, 1] - 0.9) < 0.05
    assert abs(q.var() - 10.0) < 1.5
    assert 0.03 < np.std(g["Qp"] - g["Q"]) < 0.07


def test_backward_is_the_sum_over_query_block_splits():
    geom = orc.Geometry(2, 4, 6, 1, 2, 2)
    B, Hh, d = 1, 1, 4
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s) for s in (90, 91, 92, 93))
    idx = _random_map(geom, B, Hh, 3, 94)
    full = orc.attn_bwd(Q, K, V, dO, idx, geom)
    part_a = [0, 2, 5]
    part_b = [I for I in range(geom.n_blocks) if I not in part_a]
    ga = orc.attn_bwd(Q, K, V, dO, idx[:, :, part_a], geom, query_blocks=part_a)
    gb = orc.attn_bwd(Q, K, V, dO, idx[:, :, part_b], geom, query_blocks=part_b)
    for f, a, b in zip(full, ga, gb):
        assert np.abs(a + b - f).max() < 1e-12


# ------------------------------------------------------------------ training through the merge
def _merge_loss(Os, Ls, dO, dLSE):
    O, L = orc.merge_states(Os, Ls)
    live = np.isfinite(L)
    return float((O * dO).sum() + (np.where(live, L, 0.0) * dLSE).sum())


def _merge_case(seed, P=3, rows=(2, 3), d=4):
    rng = np.random.default_rng(seed)
    Os = [rng.standard_normal(rows + (d,)) for _ in range(P)]
    Ls = [rng.standard_normal(rows) * 2 for _ in range(P)]
    Ls[1][0, 1] = -np.inf  # one empty part in a live row
    for L in Ls:
        L[1, 2] = -np.inf  # one row where every part is empty
    dO = rng.standard_normal(rows + (d,))
    dLSE = rng.standard_normal(rows)
    return Os, Ls, dO, dLSE


def test_golden_merge_bwd():
    g = _read_golden("merge_states_bwd.txt")
    for r in ("row0", "row1"):
        lse = [_num(t) for t in g[r + "_lse"].split()]
        os_ = [np.array([_num(t) for t in part.split()]) for part in g[r + "_o"].split("|")]
        dO = np.array([[_num(t) for t in g[r + "_do"].split()]])
        dL = np.array([_num(g[r + "_dlse"])])
        dOs, dLs = orc.merge_states_bwd([o[None] for o in os_], [np.array([x]) for x in lse], dO, dL)
        want_do = [np.array([_num(t) for t in part.split()]) for part in g[r + "_expect_do"].split("|")]
        want_dl = [_num(t) for t in g[r + "_expect_dlse"].split()]
        for p in range(len(os_)):
            assert np.abs(dOs[p][0] - want_do[p]).max() < 1e-14
            assert abs(dLs[p][0] - want_dl[p]) < 1e-14


@pytest.mark.parametrize("seed", [0, 1])
def test_merge_bwd_finite_differences(seed):
    Os, Ls, dO, dLSE = _merge_case(seed)
    dOs, dLs = orc.merge_states_bwd(Os, Ls, dO, dLSE)
    h = 1e-6
    for p in range(len(Os)):
        for X, G in ((Os[p], dOs[p]), (Ls[p], dLs[p])):
            num = np.zeros_like(X)
            for pos in np.ndindex(X.shape):
                x0 = X[pos]
                if np.isneginf(x0):  # an empty part stays empty under any finite change of the others
                    continue
                X[pos] = x0 + h
                lp = _merge_loss(Os, Ls, dO, dLSE)
                X[pos] = x0 - h
                lm = _merge_loss(Os, Ls, dO, dLSE)
                X[pos] = x0
                num[pos] = (lp - lm) / (2 * h)
            assert np.abs(num - G).max() <= 1e-6 * max(1.0, np.abs(G).max())


def test_merge_bwd_invariants_and_special_cases():
    Os, Ls, dO, dLSE = _merge_case(3)
    dOs, dLs = orc.merge_states_bwd(Os, Ls, dO, dLSE)
    live = np.isfinite(orc.merge_states(Os, Ls)[1])
    # the weights sum to 1 and sum_p w_p (O_p - O) = 0 on every live row
    assert np.abs((sum(dOs) - dO)[live]).max() < 1e-12
    assert np.abs((sum(dLs) - dLSE)[live]).max() < 1e-12
    # empty rows and empty parts get nothing
    assert all(np.all(x[~live] == 0) for x in dOs) and all(np.all(x[~live] == 0) for x in dLs)
    assert np.all(dOs[1][0, 1] == 0) and dLs[1][0, 1] == 0
    # one state: the merge is the identity
    a, b = orc.merge_states_bwd(Os[:1], [np.zeros((2, 3))], dO, dLSE)
    assert np.array_equal(a[0], dO) and np.abs(b[0] - dLSE).max() < 1e-15


def _lse_loss_torch(q, k, v, mask, dO, dLSE, scale):
    s = (q @ k.T) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=1)
    o = torch.softmax(s, dim=1) @ v
    return (o * dO).sum() + (lse * dLSE).sum()


def test_partition_backward_matches_torch_autograd():
    """A key range, inactive query blocks and an LSE gradient, against autograd through logsumexp + softmax."""
    geom = orc.Geometry(4, 2, 4, 1, 2, 2)  # 4 slabs of 2 blocks
    B, Hh, d = 1, 2, 4
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s, 1.5) for s in (110, 111, 112, 113))
    dLSE = _rand((B, Hh, geom.N), 114)
    idx = _random_map(geom, B, Hh, 4, 115)
    kb0, kb1 = 2, 6
    active = np.array([1, 0, 1, 1, 0, 1, 1, 1], dtype=bool)
    dQ, dK, dV = orc.attn_bwd(Q, K, V, dO, idx, geom, kb_begin=kb0, kb_end=kb1, qb_active=active, dLSE=dLSE)
    ids = _block_id_brute(geom)
    scale = 1.0 / math.sqrt(d)
    for h in range(Hh):
        mask = _mask_from_map(geom, idx[0, h]) & ((ids >= kb0) & (ids < kb1))[None, :]
        rows = active[ids] & mask.any(axis=1)  # rows of active blocks with at least one key in the range
        q, k, v = (torch.tensor(X[0, :, h], requires_grad=True) for X in (Q, K, V))
        r = torch.from_numpy(np.nonzero(rows)[0])
        loss = _lse_loss_torch(q[r], k, v, torch.from_numpy(mask[rows]), torch.from_numpy(dO[0, rows, h]),
                               torch.from_numpy(dLSE[0, h, rows]), scale)
        loss.backward()
        assert np.abs(q.grad.numpy() - dQ[0, :, h]).max() < 1e-12
        assert np.abs(k.grad.numpy() - dK[0, :, h]).max() < 1e-12
        assert np.abs(v.grad.numpy() - dV[0, :, h]).max() < 1e-12


def test_merge_and_partition_backward_compose_to_full():
    """Partitions covering every key, merged: the chain rule through the merge gives the full gradient."""
    geom = orc.Geometry(5, 2, 4, 1, 2, 2)
    B, Hh, d, P = 1, 2, 4, 3
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s) for s in (120, 121, 122, 123))
    dLSE = _rand((B, Hh, geom.N), 124)
    idx = _random_map(geom, B, Hh, 5, 125)
    states = orc.partition_states(Q, K, V, idx, geom, P)
    tr = lambda L: np.transpose(L, (0, 2, 1))  # [B, Hh, N] <-> [B, N, Hh]
    dOs, dLs = orc.merge_states_bwd([s[0] for s in states], [tr(s[1]) for s in states], dO, tr(dLSE))
    total = [np.zeros_like(X) for X in (Q, K, V)]
    for p, (b0, b1) in enumerate(orc.frame_partitions(geom, P)):
        part = orc.attn_bwd(Q, K, V, dOs[p], idx, geom, kb_begin=b0, kb_end=b1, dLSE=tr(dLs[p]))
        for acc, x in zip(total, part):
            acc += x
    full = orc.attn_bwd(Q, K, V, dO, idx, geom, dLSE=dLSE)
    for a, b in zip(total, full):
        assert np.abs(a - b).max() < 1e-12


def test_reuse_backward_finite_differences():
    """The reuse-aware training gradient: reused states are constants, fresh ones carry the gradient."""
    geom = orc.Geometry(4, 2, 2, 1, 2, 2)  # 4 slabs of 1 block
    B, Hh, d, P, n_reuse = 1, 1, 3, 4, 2
    Q, K, V, dO = (_rand((B, geom.N, Hh, d), s) for s in (130, 131, 132, 133))
    dLSE = _rand((B, Hh, geom.N), 134)
    idx = _random_map(geom, B, Hh, 3, 135)
    prev = orc.partition_states(Q + 0.3, K - 0.2, V * 1.1, _random_map(geom, B, Hh, 3, 136), geom, P)
    dQ, dK, dV = orc.reuse_bwd(Q, K, V, dO, idx, geom, P, n_reuse, prev, dLSE=dLSE)

    def loss():
        O, L = orc.reuse_merge(orc.partition_states(Q, K, V, idx, geom, P), prev, geom, P, n_reuse)
        return float((O * dO).sum() + (L * dLSE).sum())

    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for pos in np.ndindex(X.shape):
            x0 = X[pos]
            X[pos] = x0 + h
            lp = loss()
            X[pos] = x0 - h
            lm = loss()
            X[pos] = x0
            num[pos] = (lp - lm) / (2 * h)
        assert np.abs(num - G).max() <= 1e-6 * max(1.0, np.abs(G).max())
    assert np.abs(dK).max() > 0 and np.abs(dV).max() > 0


def test_reuse_backward_reads_fresh_states_as_stored():
    """Reading 9: a bf16 problem's fresh O_p enters the merge's backward rounded to bf16.  Special case: with
    one-token blocks and one kept key block per query block, each fresh state is a single v_j, which is
    already a bf16 value when V is, so the rounding changes nothing.  With several keys per state O_p is an
    average that bf16 cannot hold; the gradient then moves, by no more than the rounding's first-order effect
    (states move by 2^-9 relative, so gradients by a few 2^-9 of their scale)."""
    geom = orc.Geometry(4, 1, 4, 1, 1, 1)  # one-token blocks, 4 slabs of 4
    B, Hh, d, P, n_reuse = 1, 1, 4, 4, 2
    Q, K, dO = (_rand((B, geom.N, Hh, d), s) for s in (150, 151, 152))
    V = orc.to_bf16(_rand((B, geom.N, Hh, d), 153))
    idx = _random_map(geom, B, Hh, 1, 154)
    prev = orc.partition_states(Q + 0.1, K, V, _random_map(geom, B, Hh, 1, 155), geom, P)
    plain = orc.reuse_bwd(Q, K, V, dO, idx, geom, P, n_reuse, prev)
    stored = orc.reuse_bwd(Q, K, V, dO, idx, geom, P, n_reuse, prev, state_dtype="bf16")
    for a, b in zip(plain, stored):
        assert np.array_equal(a, b)
    V2 = _rand((B, geom.N, Hh, d), 156)
    idx3 = _random_map(geom, B, Hh, 6, 157)
    plain = orc.reuse_bwd(Q, K, V2, dO, idx3, geom, P, n_reuse, prev)
    stored = orc.reuse_bwd(Q, K, V2, dO, idx3, geom, P, n_reuse, prev, state_dtype="bf16")
    diffs = [np.abs(a - b).max() for a, b in zip(plain, stored)]
    scale = max(np.abs(x).max() for x in plain + stored)
    assert max(diffs) > 0 and max(diffs) < 8 * 2.0 ** -9 * scale, (diffs, scale)


# ------------------------------------------------------------------ predictor training signal
def _distill_case(seed, dims=(2, 4, 4, 1, 2, 2), d=5, r=3, Hh=2):
    geom = orc.Geometry(*dims)
    Q, K = (_rand((1, geom.N, Hh, d), seed + s) for s in (0, 1))
    Wq, Wk = (_rand((Hh, d, r), seed + s, 0.5) for s in (2, 3))
    return geom, Q, K, Wq, Wk


def test_distill_gradient_finite_differences():
    geom, Q, K, Wq, Wk = _distill_case(140)
    L, dWq, dWk, _, _ = orc.predictor_distill_grad(Q, K, Wq, Wk, geom, "f32")
    h = 1e-6
    for W, G in ((Wq, dWq), (Wk, dWk)):
        num = np.zeros_like(W)
        for pos in np.ndindex(W.shape):
            w0 = W[pos]
            W[pos] = w0 + h
            lp = orc.predictor_distill_grad(Q, K, Wq, Wk, geom, "f32")[0]
            W[pos] = w0 - h
            lm = orc.predictor_distill_grad(Q, K, Wq, Wk, geom, "f32")[0]
            W[pos] = w0
            num[pos] = (lp - lm) / (2 * h)
        assert np.abs(num - G).max() <= 1e-6 * max(1.0, np.abs(G).max())


def test_distill_gradient_matches_torch_autograd():
    geom, Q, K, Wq, Wk = _distill_case(150, dims=(3, 4, 6, 1, 2, 3), d=6, r=4)
    L, dWq, dWk, s, t = orc.predictor_distill_grad(Q, K, Wq, Wk, geom, "f32")
    order = np.concatenate([geom.tokens(J) for J in range(geom.n_blocks)])
    sizes = [len(geom.tokens(J)) for J in range(geom.n_blocks)]
    loss = 0.0
    wq, wk = torch.tensor(Wq, requires_grad=True), torch.tensor(Wk, requires_grad=True)
    for h in range(Q.shape[2]):
        q, k = torch.from_numpy(Q[0, order, h]), torch.from_numpy(K[0, order, h])
        S = (q @ wq[h]) @ (k @ wk[h]).T
        T = q @ k.T
        for Sb, Tb in zip(torch.split(S, sizes, 0), torch.split(T, sizes, 0)):
            for Sbb, Tbb in zip(torch.split(Sb, sizes, 1), torch.split(Tb, sizes, 1)):
                loss = loss + 0.5 * (Sbb.amax() - Tbb.amax()) ** 2
    loss.backward()
    assert abs(loss.item() - L) < 1e-9 * max(1.0, L)
    assert np.abs(wq.grad.numpy() - dWq).max() < 1e-10
    assert np.abs(wk.grad.numpy() - dWk).max() < 1e-10


def test_distill_scores_are_the_predictor_scores_and_identity_is_exact():
    geom, Q, K, Wq, Wk = _distill_case(160)
    _, _, _, s, t = orc.predictor_distill_grad(Q, K, Wq, Wk, geom, "f32")
    assert np.array_equal(s, orc.block_scores(orc.project(Q, Wq, "f32"), orc.project(K, Wk, "f32"), geom))
    d = Q.shape[3]
    eye = np.stack([np.eye(d)] * Q.shape[2])
    L, dWq, dWk, s, t = orc.predictor_distill_grad(Q, K, eye, eye, geom, "f32")
    assert L < 1e-20 and np.abs(dWq).max() < 1e-12 and np.abs(dWk).max() < 1e-12
    assert np.abs(s - t).max() < 1e-12
