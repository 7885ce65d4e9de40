"""Oracle for dynamic block-sparse attention: a plain, slow, fp64 CPU statement of the method.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
call it.  It shares no code with the CUDA path (no helpers, tables or
constants); the only thing both sides share is the seeded input generator.

What it follows:

* "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
  Training" (gist.science explainer), section 3a "low-rank predictor": a cheap
  low-rank estimate picks the ~10% of attention worth computing; section 3b
  "query grouping": neighbouring tokens share that decision; section 4 stage 2:
  attention is computed only on the predicted parts.  The explainer gives no
  formula; the form used here is the plainest one consistent with it:
  q~ = Q Wq, k~ = K Wk (rank r), block score s(I, J) = max over i in I, j in J
  of q~_i . k~_j, keep the k highest-scoring key blocks per query block with
  ties going to the lower block index.
* "DiTango: Cost-Effective Parallel Diffusion Generation with Selective
  Attention State Reuse" (gist.science explainer): attention over near context
  partitions is recomputed, far partitions reuse a cached state from an
  earlier step.  The state of a partition is read here as the pair (O, LSE) of
  softmax attention restricted to that partition's keys, and the reuse is the
  log-sum-exp merge of those states.

Readings taken where the pages are silent (each is restated in the design notes):

1. Blocks are compact bt x bh x bw space-time tiles numbered t-major
   (I = (it * nH + ih) * nW + iw); edge tiles of a non-divisible grid are
   clipped and hold only real tokens.  Inside a tile, tokens are ordered
   (tt, hh, ww).
2. For bf16 problems the projected q~, k~ are rounded to bf16 (round to
   nearest even) after an exact product; score dot products are then exact in
   fp64.  For fp32 problems q~, k~ are kept unrounded.
3. k = min(n_b, max(1, floor(keep * n_b + 1e-9))).
4. The kept key blocks of a query block are reported in ascending order.
5. Softmax scale 1/sqrt(d) unless given; the log-sum-exp uses the natural log.
6. The backward pass holds the block map fixed (no gradient through top-k).
7. A query block with no kept key in the requested key range has state
   (O = 0, LSE = -inf); the merge of all-(-inf) states is (0, -inf).
8. State-reuse partitions are contiguous ranges of tile slabs along t split
   as evenly as possible (first slabs get the extra one); the distance of
   partition p from query block I is |p - p(I)|, and the n_reuse partitions
   of largest distance (ties to the lower p) are taken from the previous
   step, whose states come from its own inputs and its own block selection.
9. Training through the merge: the pages describe the reuse for generation
   only.  Read for training, the reused states are constants of this step
   (they were computed from an earlier step's inputs) and carry no gradient;
   the fresh states are differentiated by the chain rule through the merge
   and through softmax attention restricted to their key range.  A state is
   read by the merge's backward as it is stored: in the problem's dtype, so a
   bf16 problem's fresh O_p enters it rounded to bf16 (the reused states are
   stored the same way by the step that computed them).
10. The predictor's own training signal (DSV trains it in a stage of its
    own; the pages give no loss): the block score s(I, J) is read as an
    estimate of the full-rank block-max logit t(I, J) = max over i in I,
    j in J of q_i . k_j (with r = d and identity projections the two
    coincide), distilled by L = 1/2 sum (s - t)^2.  The max passes its
    gradient to its maximising pair, the first in token order on ties; the
    bf16 rounding of q~, k~ passes it unchanged.
"""
from __future__ import annotations

import math

import numpy as np


# --------------------------------------------------------------------------- geometry
class Geometry:
    """Tiling of a T x H x W raster of tokens into bt x bh x bw blocks (reading 1)."""

    def __init__(self, T, H, W, bt, bh, bw):
        self.T, self.H, self.W = int(T), int(H), int(W)
        self.bt, self.bh, self.bw = int(bt), int(bh), int(bw)
        self.nT = -(-self.T // self.bt)
        self.nH = -(-self.H // self.bh)
        self.nW = -(-self.W // self.bw)
        self.n_blocks = self.nT * self.nH * self.nW
        self.N = self.T * self.H * self.W
        self._tokens = [self._block_tokens(I) for I in range(self.n_blocks)]

    def block_coords(self, I):
        return I // (self.nH * self.nW), (I // self.nW) % self.nH, I % self.nW

    def _block_tokens(self, I):
        it, ih, iw = self.block_coords(I)
        toks = []
        for t in range(it * self.bt, min(self.T, (it + 1) * self.bt)):
            for h in range(ih * self.bh, min(self.H, (ih + 1) * self.bh)):
                for w in range(iw * self.bw, min(self.W, (iw + 1) * self.bw)):
                    toks.append((t * self.H + h) * self.W + w)
        return np.asarray(toks, dtype=np.int64)

    def tokens(self, I):
        """Raster indices of the real tokens of block I, in (tt, hh, ww) order."""
        return self._tokens[I]


def keep_count(keep: float, n_blocks: int) -> int:
    """Reading 3: number of key blocks kept per query block."""
    return min(n_blocks, max(1, int(math.floor(keep * n_blocks + 1e-9))))


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def to_bf16(x):
    """Nearest bfloat16 value of each fp64 entry, ties to even, returned as fp64.

    Works on the binary64 encoding: bfloat16 keeps the top 7 of the 52 stored
    mantissa bits, so the low 45 bits are rounded away (half-way cases go to the
    even kept value).  Values are assumed finite and within bf16's normal range.
    """
    x = np.asarray(x, dtype=np.float64)
    bits = x.view(np.uint64)
    drop = np.uint64(45)
    half = np.uint64(1) << np.uint64(44)
    low_mask = (np.uint64(1) << drop) - np.uint64(1)
    low = bits & low_mask
    kept = bits >> drop
    round_up = (low > half) | ((low == half) & ((kept & np.uint64(1)) == np.uint64(1)))
    kept = kept + round_up.astype(np.uint64)
    return (kept << drop).view(np.float64)


# --------------------------------------------------------------------------- step 1: predictor
def project(X, Wt, dtype):
    """q~ = X Wt per head (DSV section 3a, reading 2).

    X: [B, N, Hh, d]; Wt: [Hh, d, r].  Returns [B, Hh, N, r] fp64, rounded to
    bf16 when dtype == "bf16".
    """
    X = np.asarray(X, dtype=np.float64)
    Wt = np.asarray(Wt, dtype=np.float64)
    B, N, Hh, d = X.shape
    out = np.empty((B, Hh, N, Wt.shape[2]), dtype=np.float64)
    for b in range(B):
        for h in range(Hh):
            out[b, h] = X[b, :, h, :] @ Wt[h]
    return to_bf16(out) if dtype == "bf16" else out


def block_scores(qt, kt, geom: Geometry, query_blocks=None):
    """s(I, J) = max_{i in I, j in J} q~_i . k~_j for each requested query block I and every J.

    qt, kt: [B, Hh, N, r] (from `project`).  Returns [B, Hh, len(query_blocks), n_blocks].
    """
    qb = list(range(geom.n_blocks)) if query_blocks is None else list(query_blocks)
    B, Hh = qt.shape[:2]
    order = np.concatenate([geom.tokens(J) for J in range(geom.n_blocks)])
    starts = np.cumsum([0] + [len(geom.tokens(J)) for J in range(geom.n_blocks - 1)])
    out = np.empty((B, Hh, len(qb), geom.n_blocks), dtype=np.float64)
    for b in range(B):
        for h in range(Hh):
            kord = kt[b, h][order]  # keys grouped by block
            for a, I in enumerate(qb):
                S = qt[b, h][geom.tokens(I)] @ kord.T  # every (i, j) product
                col_max = S.max(axis=0)  # max over the query group i in I
                out[b, h, a] = np.maximum.reduceat(col_max, starts)  # then over j in J
    return out


def topk_blocks(score_row, k):
    """The k best key blocks: score descending, ties to the lower index; reported ascending (reading 4)."""
    J = np.arange(len(score_row))
    order = np.lexsort((J, -np.asarray(score_row)))  # primary: -score, secondary: J
    return np.sort(order[:k]).astype(np.int32)


def predict_blocks(Q, K, Wq, Wk, geom: Geometry, keep, dtype, query_blocks=None):
    """Low-rank predictor + top-k (DSV section 3a/3b).  Returns (idx [B,Hh,nq,k] int32, scores fp64)."""
    k = keep_count(keep, geom.n_blocks)
    scores = block_scores(project(Q, Wq, dtype), project(K, Wk, dtype), geom, query_blocks)
    B, Hh, nq, _ = scores.shape
    idx = np.empty((B, Hh, nq, k), dtype=np.int32)
    for b in range(B):
        for h in range(Hh):
            for a in range(nq):
                idx[b, h, a] = topk_blocks(scores[b, h, a], k)
    return idx, scores


def predictor_distill_grad(Q, K, Wq, Wk, geom: Geometry, dtype):
    """Training signal of the low-rank predictor (DSV stage 1, reading 10).

    For every (b, h, I, J): s = q~_i* . k~_j* at the pair maximising q~_i . k~_j
    over i in I, j in J (first in the tiles' token order on ties), and the
    target t = max over the same pairs of q_i . k_j.  With e = s - t and
    L = 1/2 sum e^2:
      dL/dWq[h] = sum e Q_i*^T k~_j*,   dL/dWk[h] = sum e K_j*^T q~_i*.
    Returns (L, dWq [Hh, d, r], dWk [Hh, d, r], s, t), s and t [B, Hh, n_b, n_b].
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    qt, kt = project(Q, Wq, dtype), project(K, Wk, dtype)
    B, N, Hh, d = Q.shape
    r = qt.shape[3]
    nb = geom.n_blocks
    dWq = np.zeros((Hh, d, r))
    dWk = np.zeros((Hh, d, r))
    s_all = np.empty((B, Hh, nb, nb))
    t_all = np.empty((B, Hh, nb, nb))
    L = 0.0
    for b in range(B):
        for h in range(Hh):
            for I in range(nb):
                rows = geom.tokens(I)
                qI, QI = qt[b, h][rows], Q[b, rows, h]
                for J in range(nb):
                    cols = geom.tokens(J)
                    kJ, KJ = kt[b, h][cols], K[b, cols, h]
                    S = qI @ kJ.T
                    i, j = divmod(int(np.argmax(S)), len(cols))  # first maximum in row-major (i, j) order
                    t = (QI @ KJ.T).max()
                    e = S[i, j] - t
                    s_all[b, h, I, J] = S[i, j]
                    t_all[b, h, I, J] = t
                    L += 0.5 * e * e
                    dWq[h] += e * np.outer(QI[i], kJ[j])
                    dWk[h] += e * np.outer(KJ[j], qI[i])
    return L, dWq, dWk, s_all, t_all


# --------------------------------------------------------------------------- step 2: sparse attention
def _kept_keys(geom, sel, kb_begin, kb_end):
    blocks = [int(J) for J in sel if kb_begin <= J < kb_end]
    if not blocks:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([geom.tokens(J) for J in blocks])


def attn_fwd(Q, K, V, idx, geom: Geometry, scale=None, kb_begin=0, kb_end=None, qb_active=None,
             query_blocks=None, out=None):
    """Block-sparse softmax attention over the kept key blocks (DSV section 4, stage 2).

    For row i of query block I, over keys j of the kept blocks J with
    kb_begin <= J < kb_end: S_ij = scale q_i . k_j, LSE_i = log sum_j exp(S_ij),
    O_i = sum_j exp(S_ij - LSE_i) v_j.  Rows with no kept key get (0, -inf)
    (reading 7).  Query blocks with qb_active[I] == 0 are not written.

    idx: [B, Hh, n_blocks (or len(query_blocks)), k].  Returns (O [B,N,Hh,d], LSE [B,Hh,N]) in
    fp64; rows that were not written hold NaN unless `out` supplies arrays.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, N, Hh, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    kb_end = geom.n_blocks if kb_end is None else kb_end
    qb = list(range(geom.n_blocks)) if query_blocks is None else list(query_blocks)
    if out is None:
        O = np.full((B, N, Hh, V.shape[3]), np.nan)
        LSE = np.full((B, Hh, N), np.nan)
    else:
        O, LSE = out
    for b in range(B):
        for h in range(Hh):
            for a, I in enumerate(qb):
                if qb_active is not None and not qb_active[I]:
                    continue
                rows = geom.tokens(I)
                keys = _kept_keys(geom, idx[b, h, a], kb_begin, kb_end)
                if len(keys) == 0:
                    O[b, rows, h] = 0.0
                    LSE[b, h, rows] = -np.inf
                    continue
                S = scale * (Q[b, rows, h] @ K[b, keys, h].T)
                m = S.max(axis=1, keepdims=True)
                lse = m + np.log(np.exp(S - m).sum(axis=1, keepdims=True))
                O[b, rows, h] = np.exp(S - lse) @ V[b, keys, h]
                LSE[b, h, rows] = lse[:, 0]
    return O, LSE


def attn_bwd(Q, K, V, dO, idx, geom: Geometry, scale=None, query_blocks=None, kb_begin=0, kb_end=None,
             qb_active=None, dLSE=None):
    """Gradients of block-sparse attention with the block map held fixed (reading 6).

    With P_ij = exp(S_ij - LSE_i) over the kept keys and D_i = dO_i . O_i:
    dV_j = sum_i P_ij dO_i, dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - D_i),
    dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i.
    query_blocks restricts the sums over i to those query blocks (idx rows
    then follow that list); by linearity the full gradient is the sum over any
    split of the query blocks.  Returns (dQ, dK, dV), each [B, N, Hh, d] fp64.

    Partition states (reading 9): kb_begin, kb_end and qb_active select the
    state (O_p, LSE_p) that attn_fwd computes with the same arguments; dO is
    then dL/dO_p and dLSE ([B, Hh, N], None = 0) is dL/dLSE_p.  Since
    d LSE_i / d S_ij = P_ij, the LSE gradient enters as dS_ij = P_ij (dP_ij -
    D_i + dLSE_i).  Query blocks with qb_active[I] == 0 contribute nothing.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, N, Hh, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    kb_end = geom.n_blocks if kb_end is None else kb_end
    qb = list(range(geom.n_blocks)) if query_blocks is None else list(query_blocks)
    for b in range(B):
        for h in range(Hh):
            for a, I in enumerate(qb):
                if qb_active is not None and not qb_active[I]:
                    continue
                rows = geom.tokens(I)
                keys = _kept_keys(geom, idx[b, h, a], kb_begin, kb_end)
                if len(keys) == 0:
                    continue
                q, kk, v, do = Q[b, rows, h], K[b, keys, h], V[b, keys, h], dO[b, rows, h]
                S = scale * (q @ kk.T)
                m = S.max(axis=1, keepdims=True)
                lse = m + np.log(np.exp(S - m).sum(axis=1, keepdims=True))
                P = np.exp(S - lse)
                o = P @ v
                D = (do * o).sum(axis=1, keepdims=True)
                g = 0.0 if dLSE is None else np.asarray(dLSE, dtype=np.float64)[b, h, rows][:, None]
                dP = do @ v.T
                dS = P * (dP - D + g)
                dV[b, keys, h] += P.T @ do
                dQ[b, rows, h] += scale * (dS @ kk)
                dK[b, keys, h] += scale * (dS.T @ q)
    return dQ, dK, dV


def attn_bwd_blocks(Q, K, V, dO, idx, geom: Geometry, scale=None, query_blocks=(), key_blocks=()):
    """The same gradients as `attn_bwd`, evaluated only for some blocks.

    dQ rows of each block in `query_blocks` (needs only that block's kept list)
    and dK/dV rows of each block in `key_blocks` (sums over every query block
    that kept it).  idx must cover all query blocks.  Returns dicts
    {(b, h, I): dQ rows} and {(b, h, J): (dK rows, dV rows)}.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, N, Hh, d = Q.shape
    scale = default_scale(d) if scale is None else scale

    def row_terms(b, h, I):
        rows = geom.tokens(I)
        sel = [int(J) for J in idx[b, h, I]]
        keys = _kept_keys(geom, sel, 0, geom.n_blocks)
        q, kk, v, do = Q[b, rows, h], K[b, keys, h], V[b, keys, h], dO[b, rows, h]
        S = scale * (q @ kk.T)
        m = S.max(axis=1, keepdims=True)
        lse = m + np.log(np.exp(S - m).sum(axis=1, keepdims=True))
        P = np.exp(S - lse)
        D = (do * (P @ v)).sum(axis=1, keepdims=True)
        dS = P * (do @ v.T - D)
        return sel, q, kk, do, P, dS

    dq_out, dkv_out = {}, {}
    for b in range(B):
        for h in range(Hh):
            for I in query_blocks:
                sel, q, kk, do, P, dS = row_terms(b, h, I)
                dq_out[(b, h, I)] = scale * (dS @ kk)
            # dK/dV of each requested key block J: a sum over the query blocks that kept J; every such
            # query block's terms are formed once and added to each requested block it kept
            acc = {J: (np.zeros((len(geom.tokens(J)), d)), np.zeros((len(geom.tokens(J)), V.shape[3])))
                   for J in key_blocks}
            for I in range(geom.n_blocks):
                sel = [int(x) for x in idx[b, h, I]]
                hit = [J for J in key_blocks if J in sel]
                if not hit:
                    continue
                _, q, kk, do, P, dS = row_terms(b, h, I)
                for J in hit:
                    nJ = len(geom.tokens(J))
                    off = sum(len(geom.tokens(x)) for x in sel if x < J)
                    dk, dv = acc[J]
                    dv += P[:, off:off + nJ].T @ do
                    dk += scale * (dS[:, off:off + nJ].T @ q)
            for J in key_blocks:
                dkv_out[(b, h, J)] = acc[J]
    return dq_out, dkv_out


# --------------------------------------------------------------------------- step 3: state merge
def _merge_weights(L):
    """Per row of the stacked LSE_p [P, rows...]: (LSE, w_p = exp(LSE_p - LSE)); all -inf rows give (-inf, 0)."""
    m = L.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    s = np.exp(L - m_safe).sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, s)))
    w = np.where(empty[None], 0.0, np.exp(L - np.where(empty, 0.0, lse)[None]))
    return lse, w


def merge_states(O_parts, LSE_parts):
    """LSE merge of partial attention states (DiTango's state reuse, reading 7).

    LSE = log sum_p exp(LSE_p);  O = sum_p exp(LSE_p - LSE) O_p.
    O_parts: list of [..., d]; LSE_parts: list of matching [...] (row shapes).
    Rows where every LSE_p is -inf give (0, -inf).
    """
    L = np.stack([np.asarray(x, dtype=np.float64) for x in LSE_parts])  # [P, rows...]
    O = np.stack([np.asarray(x, dtype=np.float64) for x in O_parts])  # [P, rows..., d]
    lse, w = _merge_weights(L)
    out = (w[..., None] * O).sum(axis=0)
    return out, lse


def merge_states_bwd(O_parts, LSE_parts, dO, dLSE=None):
    """Gradient of merge_states (training through DiTango's merge, reading 9).

    With w_p = exp(LSE_p - LSE) and O = sum_p w_p O_p, the chain rule gives
    dLSE/dLSE_p = w_p and dO/dLSE_p = w_p (O_p - O), so
      dL/dO_p = w_p dO,   dL/dLSE_p = w_p (dO . (O_p - O) + dLSE).
    Shapes as merge_states; dO matches O's rows x d, dLSE the LSE rows (None =
    0).  Rows where every LSE_p is -inf give zeros.  Returns (list of dO_p,
    list of dLSE_p).
    """
    L = np.stack([np.asarray(x, dtype=np.float64) for x in LSE_parts])
    O = np.stack([np.asarray(x, dtype=np.float64) for x in O_parts])
    dO = np.asarray(dO, dtype=np.float64)
    _, w = _merge_weights(L)
    Om = (w[..., None] * O).sum(axis=0)
    g = 0.0 if dLSE is None else np.asarray(dLSE, dtype=np.float64)
    dot = (dO[None] * (np.where(w[..., None] > 0, O, 0.0) - Om[None])).sum(axis=-1)
    dL = w * (dot + g)
    dOp = w[..., None] * dO[None]
    return [dOp[p] for p in range(len(O_parts))], [dL[p] for p in range(len(O_parts))]


def frame_partitions(geom: Geometry, P):
    """Reading 8: P contiguous key-block ranges [begin, end) on tile-slab (t) boundaries."""
    per_slab = geom.nH * geom.nW
    base, extra = divmod(geom.nT, P)
    bounds, s = [], 0
    for p in range(P):
        n = base + (1 if p < extra else 0)
        bounds.append((s * per_slab, (s + n) * per_slab))
        s += n
    return bounds


def reuse_mask(geom: Geometry, P, n_reuse):
    """Reading 8: reuse[p, I] is True when partition p's state for query block I comes from the previous step."""
    bounds = frame_partitions(geom, P)
    reuse = np.zeros((P, geom.n_blocks), dtype=bool)
    for I in range(geom.n_blocks):
        pI = next(p for p, (b0, b1) in enumerate(bounds) if b0 <= I < b1)
        dist = [abs(p - pI) for p in range(P)]
        order = sorted(range(P), key=lambda p: (-dist[p], p))
        for p in order[:n_reuse]:
            reuse[p, I] = True
    return reuse


def partition_states(Q, K, V, idx, geom, P, scale=None, query_blocks=None):
    """Per-partition states (O_p, LSE_p) for every partition p (DiTango)."""
    return [attn_fwd(Q, K, V, idx, geom, scale, b0, b1, query_blocks=query_blocks)
            for (b0, b1) in frame_partitions(geom, P)]


def reuse_merge(states_now, states_prev, geom, P, n_reuse):
    """Merged attention where far partitions use the previous step's states (DiTango, reading 8).

    states_*: lists of (O_p [B,N,Hh,d], LSE_p [B,Hh,N]).  Returns (O, LSE).
    """
    reuse = reuse_mask(geom, P, n_reuse)
    Os, Ls = [], []
    for p in range(P):
        O_p = states_now[p][0].copy()
        L_p = states_now[p][1].copy()
        for I in range(geom.n_blocks):
            if reuse[p, I]:
                rows = geom.tokens(I)
                O_p[:, rows] = states_prev[p][0][:, rows]
                L_p[:, :, rows] = states_prev[p][1][:, :, rows]
        Os.append(O_p)
        Ls.append(np.transpose(L_p, (0, 2, 1)))  # [B, N, Hh] to match O's row layout
    O, L = merge_states(Os, Ls)
    return O, np.transpose(L, (0, 2, 1))


def reuse_bwd(Q, K, V, dO, idx, geom, P, n_reuse, states_prev, dLSE=None, scale=None, state_dtype=None):
    """Gradient of reuse_merge with respect to this step's Q, K, V (reading 9).

    The reused states come from an earlier step and are constants here; only
    the fresh ones carry gradient.  dL/d(state) comes from merge_states_bwd of
    the states reuse_merge merged, then each fresh partition state (key range
    of partition p, query blocks that recompute it) is differentiated with
    attn_bwd.  dO: [B, N, Hh, d]; dLSE: [B, Hh, N] or None.  state_dtype
    "bf16": the fresh O_p are read by the merge's backward as stored in bf16
    (reading 9); None or "f32": as computed.  Returns (dQ, dK, dV).
    """
    now = partition_states(Q, K, V, idx, geom, P, scale)
    reuse = reuse_mask(geom, P, n_reuse)
    Os, Ls = [], []
    for p in range(P):
        O_p, L_p = now[p][0].copy(), now[p][1].copy()
        if state_dtype == "bf16":
            O_p = to_bf16(O_p)
        for I in range(geom.n_blocks):
            if reuse[p, I]:
                rows = geom.tokens(I)
                O_p[:, rows] = states_prev[p][0][:, rows]
                L_p[:, :, rows] = states_prev[p][1][:, :, rows]
        Os.append(O_p)
        Ls.append(np.transpose(L_p, (0, 2, 1)))
    g = None if dLSE is None else np.transpose(np.asarray(dLSE, dtype=np.float64), (0, 2, 1))
    dOs, dLs = merge_states_bwd(Os, Ls, dO, g)
    grads = [np.zeros(np.shape(X)) for X in (Q, K, V)]
    for p, (b0, b1) in enumerate(frame_partitions(geom, P)):
        part = attn_bwd(Q, K, V, dOs[p], idx, geom, scale, kb_begin=b0, kb_end=b1, qb_active=~reuse[p],
                        dLSE=np.transpose(dLs[p], (0, 2, 1)))
        for acc, x in zip(grads, part):
            acc += x
    return tuple(grads)
