"""Helpers shared by the GPU parity tests and the smoke check.

Tolerances: bf16 problems max-abs <= 2e-2 and relative Frobenius <= 1e-2;
fp32 problems 1e-4 for both.  Block selection: exact wherever the oracle's gap
between the k-th and (k+1)-th score exceeds 1e-3 relative; otherwise (a
near-tie) every selected block must score within 1e-3 of the (k+1)-th.
"""
from __future__ import annotations

import numpy as np

TOL = {"bf16": (2e-2, 1e-2), "f32": (1e-4, 1e-4)}
GAP_REL = 1e-3


def dev(x: np.ndarray, dtype: str):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    return t.to(torch.bfloat16) if dtype == "bf16" else t.float()


def host(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray) -> tuple[float, float]:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    if not np.array_equal(fin, np.isfinite(got)) or not np.array_equal(got[~fin], ref[~fin]):
        return float("inf"), float("inf")
    d = got[fin] - ref[fin]
    mx = float(np.abs(d).max()) if d.size else 0.0
    nrm = float(np.linalg.norm(ref[fin]))
    rel = float(np.linalg.norm(d) / nrm) if nrm > 0 else float(np.linalg.norm(d))
    return mx, rel


def assert_close(got, ref, dtype: str, what: str):
    atol, rtol = TOL[dtype]
    mx, rel = errors(got, ref)
    assert mx <= atol and rel <= rtol, f"{what}: max-abs {mx:.3e} (tol {atol}), rel-frob {rel:.3e} (tol {rtol})"
    return mx, rel


def assert_close_stored(got, ref, dtype: str, out_dtype: str, what: str):
    """Like assert_close, for a result stored in `out_dtype`: a bf16 output cannot be closer to the
    exact value than its own rounding (2^-9 relative), so each element may differ by
    atol + 2^-8 |ref| (rounding plus the computation's share); rel-Frobenius keeps its bound."""
    if out_dtype != "bf16":
        return assert_close(got, ref, dtype, what)
    atol, rtol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    excess = np.abs(got - ref) - (atol + 2.0 ** -8 * np.abs(ref))
    _, rel = errors(got, ref)
    assert excess.max() <= 0 and rel <= rtol, f"{what}: worst excess {excess.max():.3e}, rel-frob {rel:.3e}"
    return rel


def check_scores(got, ref):
    """Block scores of a bf16 problem: fp32 accumulation of exact bf16 products, so they match the oracle
    to ~1e-6 except where a q~ or k~ element was rounded to the neighbouring bf16 value (the GPU rounds an
    fp32-accumulated projection, the oracle an exact one; q~ and k~ are rounded after the product): such a
    flip moves a score by about 2^-8 of one of its r terms.  Nearly every score must agree to 1e-5 of the
    largest, and every one to 4e-3."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref) / np.abs(ref).max()
    assert np.mean(err > 1e-5) < 0.02, np.mean(err > 1e-5)
    assert err.max() < 4e-3, err.max()


def check_selection(gpu_idx: np.ndarray, scores: np.ndarray, k: int) -> dict:
    """Compare GPU index rows [..., k] with the oracle's scores [..., n_b] under the gap rule."""
    gi = gpu_idx.reshape(-1, k)
    sc = scores.reshape(-1, scores.shape[-1])
    nb = sc.shape[1]
    stats = {"rows": gi.shape[0], "exact": 0, "near_tie": 0, "near_tie_differs": 0, "fail": 0}
    for row in range(gi.shape[0]):
        s = sc[row]
        order = np.lexsort((np.arange(nb), -s))
        want = np.sort(order[:k])
        got = gi[row]
        if k == nb:
            rel = np.inf
        else:
            sk, sk1 = s[order[k - 1]], s[order[k]]
            rel = (sk - sk1) / max(abs(sk), abs(sk1), 1e-30)
        if rel > GAP_REL:
            if np.array_equal(got, want):
                stats["exact"] += 1
            else:
                stats["fail"] += 1
            continue
        stats["near_tie"] += 1
        sk, sk1 = s[order[k - 1]], s[order[k]]
        floor = sk1 - GAP_REL * max(abs(sk), abs(sk1))
        valid = (len(set(got.tolist())) == k and np.all(np.diff(got) > 0) and np.all(got >= 0) and np.all(got < nb)
                 and np.all(s[got] >= floor))
        if not valid:
            stats["fail"] += 1
        elif not np.array_equal(got, want):
            stats["near_tie_differs"] += 1
    return stats


def reaching_tokens(rows, offsets, T, H, W, kt, kh, kw):
    """Every token one of whose samples can have a trilinear corner on one of `rows`: the tokens within the
    window's half-size plus the largest |offset| plus one of a row, per axis."""
    r = np.ceil(np.nanmax(np.abs(offsets), axis=(0, 1, 2, 3))).astype(int) + 1 + np.array([kt, kh, kw]) // 2
    out = set()
    for m in np.asarray(rows):
        t, y, x = m // (H * W), (m // W) % H, m % W
        for tt in range(max(0, t - r[0]), min(T, t + r[0] + 1)):
            for yy in range(max(0, y - r[1]), min(H, y + r[1] + 1)):
                for xx in range(max(0, x - r[2]), min(W, x + r[2] + 1)):
                    out.add((tt * H + yy) * W + xx)
    return np.array(sorted(out), dtype=np.int64)

