"""Seeded synthetic workloads for dynamic block-sparse attention over T x H x W video latents.

This module only *draws inputs*: it holds the workload shapes and the random
generators that both the CUDA path and the CPU oracle consume.  It contains none
of the method's arithmetic (no projection, score, selection, softmax or merge).

Workloads follow the problem statement of "DSV: Exploiting Dynamic Sparsity to
Accelerate Large-Scale Video DiT Training" (gist.science explainer, section 3a
"low-rank predictor" and 3b "query grouping"): tokens of a T x H x W latent
grid, several heads, a head dimension, space-time tile sizes for query/key
blocks, a predictor rank and a keep ratio.  The last workload adds the
partitioned state-reuse setting of "DiTango: Cost-Effective Parallel Diffusion
Generation with Selective Attention State Reuse".

Input recipe (all fp64, then rounded once to the workload dtype):

* Q = A * F + N(0,1), K = A * F + N(0,1), with one shared random Fourier field
  F per (batch, head) and independent noise.  F_c(t,h,w) =
  sqrt(2/M) * sum_m cos(2 pi w_m . (t,h,w) + phi_{m,c}) has unit variance;
  frequencies w_m ~ U(-1/8, 1/8)^3 cycles per token step, phases ~ U[0, 2pi).
  The shared field makes attention local in space-time, as the pages describe.
* V, dO ~ N(0,1); Wq, Wk ~ N(0, 1/d) of shape [heads, d, r].
* Previous diffusion step (state-reuse workload): Q' = Q + 0.05 N(0,1), and the
  same for K' and V' with independent draws, re-rounded to the dtype.

Every (stream, batch, head) has its own counter-free SeedSequence spawn key, so
any head can be generated alone and the bytes do not depend on which heads are
asked for.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

# Stream ids for SeedSequence spawn keys: one child stream per quantity.
_FIELD, _QNOISE, _KNOISE, _V, _WQ, _WK, _DO, _PREV = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and generator parameters of one synthetic problem."""

    name: str
    B: int
    heads: int
    T: int
    H: int
    W: int
    d: int
    bt: int
    bh: int
    bw: int
    rank: int
    keep: float
    dtype: str  # "f32" or "bf16"
    amp: float  # Fourier-field amplitude A
    n_terms: int  # Fourier terms M
    backward: bool = False
    partitions: int = 0  # key partitions for the state-reuse workload (0 = none)
    n_reuse: int = 0  # partitions per query block taken from the previous step

    @property
    def N(self) -> int:
        return self.T * self.H * self.W

    @property
    def block_tokens(self) -> int:
        return self.bt * self.bh * self.bw

    @property
    def grid(self) -> tuple[int, int, int]:
        return (-(-self.T // self.bt), -(-self.H // self.bh), -(-self.W // self.bw))

    @property
    def n_blocks(self) -> int:
        a, b, c = self.grid
        return a * b * c

    @property
    def k(self) -> int:
        """Kept key blocks per query block: floor(keep * n_b) clamped to [1, n_b]."""
        return min(self.n_blocks, max(1, int(math.floor(self.keep * self.n_blocks + 1e-9))))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    # 256-token fp32 forward: 1x8x8 tiles, keep top-2 of 4 key blocks.
    "tiny_f32_256": Workload("tiny_f32_256", 1, 2, 4, 8, 8, 64, 1, 8, 8, 16, 0.5, "f32", 3.0, 16),
    # 8,192-token bf16 forward, d=64, 2x8x8 tiles, keep 6 of 64.
    "fwd_8k": Workload("fwd_8k", 1, 12, 8, 32, 32, 64, 2, 8, 8, 16, 0.10, "bf16", 3.0, 16),
    # 61,440-token bf16 forward, d=128, sharply local field, keep 24 of 480.
    "fwd_61k": Workload("fwd_61k", 1, 24, 16, 48, 80, 128, 2, 8, 8, 32, 0.05, "bf16", 4.0, 32),
    # 524,288-token bf16 training step (forward + backward), keep 204 of 4096.
    "train_524k": Workload("train_524k", 1, 8, 32, 128, 128, 128, 2, 8, 8, 32, 0.05, "bf16", 4.0, 32,
                           backward=True),
    # 131,040-token ragged grid, 4 frame partitions, 2 farthest partitions reused.
    "merge_131k": Workload("merge_131k", 1, 16, 21, 60, 104, 128, 2, 8, 8, 32, 0.10, "bf16", 4.0, 32,
                           partitions=4, n_reuse=2),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (ties to even); returned as float32.

    x = m * 2**e with 0.5 <= |m| < 1; bfloat16 keeps 8 significant bits, so
    m * 2**8 is rounded half-to-even to an integer and scaled back.  The
    result is exactly representable in float32.
    """
    x64 = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x64)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8).astype(np.float32)


def _to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    raise ValueError(dtype)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(key))))


def _field(wl: Workload, seed: int, b: int, h: int, n0: int, n1: int) -> np.ndarray:
    """Unit-variance random Fourier field for tokens [n0, n1) (raster order), [n, d] fp64."""
    rng = _rng(seed, _FIELD, b, h)
    M = wl.n_terms
    omega = rng.uniform(-0.125, 0.125, size=(M, 3))
    phase = rng.uniform(0.0, 2.0 * np.pi, size=(M, wl.d))
    n = np.arange(n0, n1, dtype=np.int64)
    w = n % wl.W
    hh = (n // wl.W) % wl.H
    t = n // (wl.W * wl.H)
    # separable phasors exp(i 2 pi omega . x) per token, [n, M]
    arg = 2.0 * np.pi * (np.outer(t, omega[:, 0]) + np.outer(hh, omega[:, 1]) + np.outer(w, omega[:, 2]))
    E = np.exp(1j * arg)
    A = np.exp(1j * phase)  # [M, d]
    return math.sqrt(2.0 / M) * (E @ A).real


def _head_arrays(wl: Workload, seed: int, b: int, h: int, want: frozenset) -> dict[str, np.ndarray]:
    """Draw every per-head [N, d] array requested in `want` (already dtype-rounded)."""
    N, d = wl.N, wl.d
    out: dict[str, np.ndarray] = {}
    need_field = bool(want & {"Q", "K", "Qp", "Kp"})
    if need_field:
        F = np.empty((N, d), dtype=np.float64)
        chunk = 1 << 16
        for n0 in range(0, N, chunk):
            F[n0:n0 + chunk] = _field(wl, seed, b, h, n0, min(N, n0 + chunk))
        F *= wl.amp
    if want & {"Q", "Qp"}:
        q = F + _rng(seed, _QNOISE, b, h).standard_normal((N, d))
        out["Q"] = _to_dtype(q, wl.dtype)
    if want & {"K", "Kp"}:
        kk = F + _rng(seed, _KNOISE, b, h).standard_normal((N, d))
        out["K"] = _to_dtype(kk, wl.dtype)
    if need_field:
        del F
    if want & {"V", "Vp"}:
        out["V"] = _to_dtype(_rng(seed, _V, b, h).standard_normal((N, d)), wl.dtype)
    if "dO" in want:
        out["dO"] = _to_dtype(_rng(seed, _DO, b, h).standard_normal((N, d)), wl.dtype)
    for j, name in enumerate(("Q", "K", "V")):
        if name + "p" in want:
            noise = _rng(seed, _PREV, b, h, j).standard_normal((N, d))
            out[name + "p"] = _to_dtype(out[name].astype(np.float64) + 0.05 * noise, wl.dtype)
    for name in ("Q", "K", "V"):
        if name not in want and name in out:
            del out[name]
    return out


def generate(wl: Workload, seed: int = 0, names=("Q", "K", "V", "Wq", "Wk"), heads=None,
             threads: int | None = None) -> dict[str, np.ndarray]:
    """Draw the seeded inputs of `wl`.

    names: any of Q, K, V, dO (per-token [B, N, heads_sel, d]), Qp, Kp, Vp (the
    previous diffusion step's tensors, same layout) and Wq, Wk ([heads_sel, d, r]).
    heads: optional list of head indices; the values of a head do not depend on
    which other heads are generated.  Arrays are float32 holding values exactly
    representable in the workload dtype.
    """
    heads = list(range(wl.heads)) if heads is None else list(heads)
    want = frozenset(names)
    tok = [n for n in ("Q", "K", "V", "dO", "Qp", "Kp", "Vp") if n in want]
    out: dict[str, np.ndarray] = {}
    for n in tok:
        out[n] = np.empty((wl.B, wl.N, len(heads), wl.d), dtype=np.float32)
    jobs = [(b, hi, h) for b in range(wl.B) for hi, h in enumerate(heads)]

    def run(job):
        b, hi, h = job
        arrs = _head_arrays(wl, seed, b, h, want)
        for n in tok:
            out[n][b, :, hi, :] = arrs[n]

    if tok:
        nthreads = threads or min(len(jobs), max(1, len(os.sched_getaffinity(0))))
        if nthreads > 1 and len(jobs) > 1:
            with _cf.ThreadPoolExecutor(nthreads) as ex:
                list(ex.map(run, jobs))
        else:
            for j in jobs:
                run(j)
    for name, stream in (("Wq", _WQ), ("Wk", _WK)):
        if name in want:
            Wt = np.stack([_rng(seed, stream, h).standard_normal((wl.d, wl.rank)) / math.sqrt(wl.d)
                           for h in heads])
            out[name] = _to_dtype(Wt, wl.dtype)
    return out


def scattered_block_map(wl: Workload, seed: int = 0, sigma: float = 0.5) -> np.ndarray:
    """A seeded block map [B, heads, n_b, k] (int32, rows ascending) shaped like the predictor's maps on
    these inputs: each query block keeps k distinct key blocks scattered over the whole grid, and key
    blocks differ in popularity, so the number of query blocks that keep one key block is heavy-tailed
    (with the predictor on the 61K- and 131K-token workloads it runs from 0 to 4.5-6 k with a median
    near 0.85 k; sigma = 0.5 gives a median of 0.89 k and a maximum of 4-6 k at 524K tokens).  Per
    (batch, head) every key block gets a weight exp(sigma z), z ~ N(0, 1); each row is a weighted draw of
    k blocks without replacement (the k largest of log-weight + Gumbel noise).  Used where a test needs one
    fixed map shared by both sides for more rows than the oracle's predictor can produce in test time."""
    nb, k = wl.n_blocks, wl.k
    out = np.empty((wl.B, wl.heads, nb, k), dtype=np.int32)
    rows_per_chunk = max(1, (1 << 22) // nb)
    for b in range(wl.B):
        for h in range(wl.heads):
            rng = _rng(seed, 101, b, h)
            logw = sigma * rng.standard_normal(nb)
            for r0 in range(0, nb, rows_per_chunk):
                r1 = min(nb, r0 + rows_per_chunk)
                keys = logw[None, :] + rng.gumbel(size=(r1 - r0, nb))
                top = np.argpartition(-keys, k - 1, axis=1)[:, :k] if k < nb else np.tile(np.arange(nb), (r1 - r0, 1))
                out[b, h, r0:r1] = np.sort(top, axis=1)
    return out


def digest(arrays: dict[str, np.ndarray]) -> str:
    """sha256 over the named arrays' bytes (sorted by name), to log that both sides saw the same inputs."""
    import hashlib

    hsh = hashlib.sha256()
    for k in sorted(arrays):
        hsh.update(k.encode())
        hsh.update(np.ascontiguousarray(arrays[k]).tobytes())
    return hsh.hexdigest()


# --------------------------------------------------------------------------- 3D deformable sliding attention
# Workloads of "MegaSlide-DiT" (gist.science explainer, section 2 "3D deformable sliding attention"): the
# same T x H x W latent grids, a kt x kh x kw window per token.  Recipe: Q, K as above (shared Fourier field
# plus noise, so attention is local in space-time), V ~ N(0,1), all rounded to bf16; offsets ~ N(0, off_std^2)
# in token units (fp32, drawn directly for the attention alone); offset-network weights in fp32:
# Wc ~ N(0, 1/27), bc ~ N(0, 0.1^2), Wl ~ N(0, off_std^2 / (d (amp^2 + 1))), bl ~ N(0, 0.1^2), which gives
# predicted offsets of about off_std tokens.
_DSA_OFF, _DSA_WC, _DSA_BC, _DSA_WL, _DSA_BL, _DSA_DOFF = range(20, 26)


@dataclasses.dataclass(frozen=True)
class Dsa3dWorkload:
    """Shape and generator parameters of one 3D-DSA problem (bf16 activations)."""

    name: str
    B: int
    heads: int
    T: int
    H: int
    W: int
    d: int
    kt: int
    kh: int
    kw: int
    off_std: float
    amp: float = 3.0
    n_terms: int = 16
    dtype: str = "bf16"

    @property
    def N(self) -> int:
        return self.T * self.H * self.W

    @property
    def S(self) -> int:
        return self.kt * self.kh * self.kw

    def with_(self, **kw) -> "Dsa3dWorkload":
        return dataclasses.replace(self, **kw)


DSA3D_WORKLOADS = {
    # ragged grid, d = 64, 3 x 3 x 3 window
    "dsa3d_ragged_d64": Dsa3dWorkload("dsa3d_ragged_d64", 1, 3, 5, 12, 20, 64, 3, 3, 3, 1.0),
    # two batch entries, d = 128, a flat 1 x 5 x 5 window, larger offsets
    "dsa3d_d128_1x5x5": Dsa3dWorkload("dsa3d_d128_1x5x5", 2, 2, 4, 9, 11, 128, 1, 5, 5, 1.5, 4.0),
    # offsets of several tokens: many samples leave the raster
    "dsa3d_far": Dsa3dWorkload("dsa3d_far", 1, 2, 3, 8, 10, 128, 3, 3, 3, 6.0),
    # the 524,288-token grid of the block-sparse workloads, 8 heads, d = 128, 3 x 3 x 3
    "dsa3d_524k": Dsa3dWorkload("dsa3d_524k", 1, 8, 32, 128, 128, 128, 3, 3, 3, 1.0, 4.0, 32),
}


def generate_dsa3d(wl: Dsa3dWorkload, seed: int = 0, names=("Q", "K", "V", "offsets"), heads=None,
                   threads: int | None = None) -> dict[str, np.ndarray]:
    """Draw the seeded inputs of a 3D-DSA workload.

    names: Q, K, V, dO ([B, N, heads_sel, d] float32 holding bf16 values), offsets and d_offsets (an upstream
    gradient of the offsets, unit normal) ([B, N, heads_sel, S, 3] float32), Wc ([heads_sel, d, 3, 3, 3]), bc ([heads_sel, d]), Wl ([heads_sel, d, 3 S]), bl
    ([heads_sel, 3 S]).  As for `generate`, a head's values do not depend on which heads are asked for.
    """
    heads = list(range(wl.heads)) if heads is None else list(heads)
    want = frozenset(names)
    out = generate(wl, seed, names=tuple(n for n in ("Q", "K", "V", "dO") if n in want), heads=heads,
                   threads=threads) if want & {"Q", "K", "V", "dO"} else {}
    S, d = wl.S, wl.d
    if "offsets" in want:
        off = np.empty((wl.B, wl.N, len(heads), S, 3), dtype=np.float32)
        for b in range(wl.B):
            for hi, h in enumerate(heads):
                off[b, :, hi] = wl.off_std * _rng(seed, _DSA_OFF, b, h).standard_normal((wl.N, S, 3))
        out["offsets"] = off
    if "d_offsets" in want:
        g = np.empty((wl.B, wl.N, len(heads), S, 3), dtype=np.float32)
        for b in range(wl.B):
            for hi, h in enumerate(heads):
                g[b, :, hi] = _rng(seed, _DSA_DOFF, b, h).standard_normal((wl.N, S, 3))
        out["d_offsets"] = g
    wscale = wl.off_std / math.sqrt(d * (wl.amp ** 2 + 1.0))
    for name, stream, shape, sd in (("Wc", _DSA_WC, (d, 3, 3, 3), 1.0 / math.sqrt(27.0)),
                                    ("bc", _DSA_BC, (d,), 0.1),
                                    ("Wl", _DSA_WL, (d, 3 * S), wscale),
                                    ("bl", _DSA_BL, (3 * S,), 0.1)):
        if name in want:
            out[name] = np.stack([sd * _rng(seed, stream, h).standard_normal(shape) for h in heads]).astype(np.float32)
    return out
