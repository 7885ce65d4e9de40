"""The C-ABI library: it loads, exports every symbol include/sda.h declares, and its
host-only calls (block counts, workspace sizes, argument validation) behave
without a GPU.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

from dynamic_block_sparse_rank_gb300 import inputs, sda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from dynamic_block_sparse_rank_gb300 import build

    build.build()
    return sda.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "sda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sda_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert set(names) >= set(sda.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_exported_symbols_have_c_linkage(L):
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", sda.LIB_PATH], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in _declared():
        assert n in syms, n


@pytest.mark.parametrize("name,nb,k", [("tiny_f32_256", 4, 2), ("fwd_8k", 64, 6), ("fwd_61k", 480, 24),
                                       ("train_524k", 4096, 204), ("merge_131k", 1144, 114)])
def test_block_counts(L, name, nb, k):
    wl = inputs.WORKLOADS[name]
    assert sda.sda_num_blocks(sda.problem_from_workload(wl)) == (nb, k)
    assert wl.n_blocks == nb and wl.k == k


def test_keep_count_matches_the_oracle_for_every_keep(L):
    """k from the C ABI equals the oracle's reading of the keep ratio for keep in {0.01, ..., 0.99} on block
    counts from 4 to 4096, including products such as 0.29 x 100 that double arithmetic leaves just below an
    integer (the 1e-9 guard lifts them)."""
    import oracle as orc

    mismatches = []
    for nb in (4, 10, 20, 64, 100, 480, 1144, 4096):
        for i in range(1, 100):
            keep = i / 100
            p = sda.problem(1, 1, nb, 1, 1, 64, 1, 1, 1, 16, keep, "f32")
            got = sda.sda_num_blocks(p)
            want = orc.keep_count(keep, nb)
            if got != (nb, want):
                mismatches.append((keep, nb, got[1], want))
    assert not mismatches, mismatches[:10]
    assert orc.keep_count(0.29, 100) == 29 and sda.sda_num_blocks(sda.problem(1, 1, 100, 1, 1, 64, 1, 1, 1, 16, 0.29,
                                                                              "f32"))[1] == 29


def test_workspace_sizes(L):
    wl = inputs.WORKLOADS["train_524k"]
    p = sda.problem_from_workload(wl)
    pred = sda.sda_workspace_size(p, sda.SDA_OP_PREDICT)
    assert pred == 2 * wl.heads * wl.n_blocks * 128 * wl.rank * 2  # q~ and k~ in bf16, tile order
    bwd = sda.sda_workspace_size(p, sda.SDA_OP_BWD)
    assert bwd >= wl.heads * wl.n_blocks * (2 * 128 * 4 + wl.k * 4)
    f32 = sda.problem_from_workload(inputs.WORKLOADS["tiny_f32_256"])
    assert sda.sda_workspace_size(f32, sda.SDA_OP_PREDICT) > 0 and sda.sda_workspace_size(f32, sda.SDA_OP_BWD) > 0
    with pytest.raises(sda.SdaError) as e:
        sda.sda_workspace_size(p, 7)
    assert e.value.status == sda.SDA_ERR_INVALID_ARG


def _bad(p_kw):
    base = dict(B=1, heads=2, T=4, H=8, W=8, head_dim=64, bt=2, bh=8, bw=8, rank=16, keep_ratio=0.5, dtype="bf16")
    base.update(p_kw)
    return sda.problem(**base)


@pytest.mark.parametrize("kw,status", [
    ({"B": 0}, sda.SDA_ERR_INVALID_ARG), ({"T": -1}, sda.SDA_ERR_INVALID_ARG), ({"bw": 0}, sda.SDA_ERR_INVALID_ARG),
    ({"keep_ratio": 0.0}, sda.SDA_ERR_INVALID_ARG), ({"keep_ratio": float("nan")}, sda.SDA_ERR_INVALID_ARG),
    ({"dtype": 7}, sda.SDA_ERR_INVALID_ARG), ({"softmax_scale": -1.0}, sda.SDA_ERR_INVALID_ARG),
    ({"head_dim": 96}, sda.SDA_ERR_UNSUPPORTED), ({"bt": 1}, sda.SDA_ERR_UNSUPPORTED),
    ({"rank": 24}, sda.SDA_ERR_UNSUPPORTED), ({"dtype": "f32", "head_dim": 256}, sda.SDA_ERR_UNSUPPORTED),
])
def test_invalid_problems_are_rejected_on_the_host(L, kw, status):
    p = _bad(kw)
    with pytest.raises(sda.SdaError) as e:
        sda.sda_workspace_size(p, sda.SDA_OP_PREDICT)
    assert e.value.status == status


def test_null_and_range_arguments_return_before_any_launch(L):
    p = _bad({})
    # null tensors: rejected synchronously, no CUDA call is made
    assert L.sda_predict_blocks(ctypes.byref(p), None, None, None, None, None, None, None, 0, None) == \
        sda.SDA_ERR_INVALID_ARG
    assert L.sda_attn_fwd(ctypes.byref(p), 16, 16, 16, 16, 0, 99, None, 16, 16, 1, None) == sda.SDA_ERR_INVALID_ARG
    assert L.sda_attn_fwd(ctypes.byref(p), 16, 16, 16, 16, 3, 2, None, 16, 16, 1, None) == sda.SDA_ERR_INVALID_ARG
    # misaligned pointers on the tensor-core path
    assert L.sda_attn_fwd(ctypes.byref(p), 18, 16, 16, 16, 0, 2, None, 16, 16, 1, None) == sda.SDA_ERR_INVALID_ARG
    # bad output dtype
    assert L.sda_attn_fwd(ctypes.byref(p), 16, 16, 16, 16, 0, 2, None, 16, 16, 5, None) == sda.SDA_ERR_INVALID_ARG
    # workspace too small
    assert L.sda_predict_blocks(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, 8, None) == sda.SDA_ERR_WORKSPACE
    # bad gradient dtype
    assert L.sda_attn_bwd(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 5, 16, 1 << 40, None) == \
        sda.SDA_ERR_INVALID_ARG
    # merge: bad state count, unsupported width
    arr = (ctypes.c_void_p * 1)(16)
    assert L.sda_merge_states(0, arr, arr, 1, 4, 1, 64, 1, 16, 16, None) == sda.SDA_ERR_INVALID_ARG
    assert L.sda_merge_states(17, arr, arr, 1, 4, 1, 64, 1, 16, 16, None) == sda.SDA_ERR_INVALID_ARG
    assert L.sda_merge_states(1, arr, arr, 1, 4, 1, 12, 1, 16, 16, None) == sda.SDA_ERR_UNSUPPORTED


def test_training_through_the_merge_validates_on_the_host(L):
    """sda_merge_states_bwd and sda_attn_bwd_partition reject bad arguments before any launch."""
    arr = (ctypes.c_void_p * 1)(16)
    farr = (ctypes.c_void_p * 1)(16)
    mb = L.sda_merge_states_bwd
    assert mb(0, arr, arr, 16, None, 1, 4, 1, 64, 1, arr, farr, None) == sda.SDA_ERR_INVALID_ARG
    assert mb(17, arr, arr, 16, None, 1, 4, 1, 64, 1, arr, farr, None) == sda.SDA_ERR_INVALID_ARG
    assert mb(1, arr, arr, None, None, 1, 4, 1, 64, 1, arr, farr, None) == sda.SDA_ERR_INVALID_ARG  # no dO
    assert mb(1, arr, arr, 16, None, 1, 4, 1, 12, 1, arr, farr, None) == sda.SDA_ERR_UNSUPPORTED  # 24-byte rows
    assert mb(1, arr, arr, 18, None, 1, 4, 1, 64, 1, arr, farr, None) == sda.SDA_ERR_INVALID_ARG  # misaligned dO
    none = (ctypes.c_void_p * 1)(None)
    assert mb(1, arr, arr, 16, None, 1, 4, 1, 64, 1, none, farr, None) == sda.SDA_ERR_INVALID_ARG  # no dO_0
    p = _bad({})  # n_b = 2
    bp = L.sda_attn_bwd_partition
    t = [16] * 5
    # key range outside [0, n_b] or reversed
    assert bp(ctypes.byref(p), *t[:4], 16, t[4], None, 16, 0, 3, None, 16, 16, 16, 1, 16, 1 << 40, None) == \
        sda.SDA_ERR_INVALID_ARG
    assert bp(ctypes.byref(p), *t[:4], 16, t[4], None, 16, 2, 1, None, 16, 16, 16, 1, 16, 1 << 40, None) == \
        sda.SDA_ERR_INVALID_ARG
    assert bp(ctypes.byref(p), *t[:4], 16, t[4], None, 16, -1, 1, None, 16, 16, 16, 1, 16, 1 << 40, None) == \
        sda.SDA_ERR_INVALID_ARG
    # bad gradient dtype, small workspace, missing dQ
    assert bp(ctypes.byref(p), *t[:4], 16, t[4], None, 16, 0, 2, None, 16, 16, 16, 5, 16, 1 << 40, None) == \
        sda.SDA_ERR_INVALID_ARG
    assert bp(ctypes.byref(p), *t[:4], 16, t[4], None, 16, 0, 2, None, 16, 16, 16, 1, 16, 8, None) == \
        sda.SDA_ERR_WORKSPACE
    assert bp(ctypes.byref(p), *t[:4], 16, t[4], None, 16, 0, 2, None, None, 16, 16, 1, 16, 1 << 40, None) == \
        sda.SDA_ERR_INVALID_ARG


def test_training_pair_validates_on_the_host(L):
    p = _bad({})
    ws_need = sda.sda_workspace_size(p, sda.SDA_OP_TRAIN)
    assert ws_need > sda.sda_workspace_size(p, sda.SDA_OP_BWD)  # + the fp32 O
    fw, bw = L.sda_attn_fwd_train, L.sda_attn_bwd_train
    assert fw(ctypes.byref(p), None, 16, 16, 16, 16, 16, 16, ws_need, None) == sda.SDA_ERR_INVALID_ARG
    assert fw(ctypes.byref(p), 18, 16, 16, 16, 16, 16, 16, ws_need, None) == sda.SDA_ERR_INVALID_ARG  # misaligned
    assert fw(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, ws_need - 1, None) == sda.SDA_ERR_WORKSPACE
    assert bw(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 1, 0, 16, ws_need, None) == sda.SDA_ERR_INVALID_ARG  # phases
    assert bw(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 1, 8, 16, ws_need, None) == sda.SDA_ERR_INVALID_ARG
    assert bw(ctypes.byref(p), 16, 16, 16, None, 16, 16, 1, 2, 16, ws_need, None) == sda.SDA_ERR_INVALID_ARG  # dQ
    assert bw(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 5, 7, 16, ws_need, None) == sda.SDA_ERR_INVALID_ARG  # dtype
    assert bw(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 1, 7, 16, ws_need - 1, None) == sda.SDA_ERR_WORKSPACE
    f32 = _bad({"dtype": "f32"})
    with pytest.raises(sda.SdaError) as e:
        sda.sda_workspace_size(f32, sda.SDA_OP_TRAIN)
    assert e.value.status == sda.SDA_ERR_UNSUPPORTED


def test_predictor_training_signal_validates_on_the_host(L):
    p = _bad({})
    need = sda.sda_workspace_size(p, sda.SDA_OP_PREDICTOR_GRAD)
    assert need > sda.sda_workspace_size(p, sda.SDA_OP_PREDICT)  # q~, k~ tiles + norms + per-token sums
    g = L.sda_predictor_grad
    assert g(ctypes.byref(p), None, 16, 16, 16, 16, 16, 16, None, None, 16, need, None) == sda.SDA_ERR_INVALID_ARG
    assert g(ctypes.byref(p), 16, 16, 16, 16, 16, 16, None, None, None, 16, need, None) == sda.SDA_ERR_INVALID_ARG
    assert g(ctypes.byref(p), 18, 16, 16, 16, 16, 16, 16, None, None, 16, need, None) == sda.SDA_ERR_INVALID_ARG
    assert g(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, None, None, 16, need - 1, None) == sda.SDA_ERR_WORKSPACE
    f32 = _bad({"dtype": "f32"})
    assert g(ctypes.byref(f32), 16, 16, 16, 16, 16, 16, 16, None, None, 16, 1 << 40, None) == sda.SDA_ERR_UNSUPPORTED


def test_status_strings(L):
    for s in range(8):
        assert sda.status_string(s) and "unknown" not in sda.status_string(s)
    assert "unknown" in sda.status_string(42)


def test_binding_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sda, "_lib", None)
    monkeypatch.setattr(sda, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        sda.lib()


def test_dsa3d_host_validation(L):
    """Argument checks of the 3D-DSA calls happen before any launch (no GPU needed)."""
    import ctypes

    from dynamic_block_sparse_rank_gb300 import sda

    fake = 1 << 20  # 16-byte aligned, never dereferenced: every call below fails validation first
    f = lambda p: sda.lib().sda_dsa3d_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, None)
    g = lambda p: sda.lib().sda_dsa3d_offsets(ctypes.byref(p), fake, fake, fake, fake, fake, fake, None)
    good = dict(B=1, T=4, H=5, W=6, heads=2, d=64, kt=3, kh=3, kw=3)
    bad = [(dict(kt=2), sda.SDA_ERR_INVALID_ARG), (dict(T=0), sda.SDA_ERR_INVALID_ARG),
           (dict(heads=0), sda.SDA_ERR_INVALID_ARG), (dict(d=96), sda.SDA_ERR_UNSUPPORTED),
           (dict(kt=7, kh=7, kw=3), sda.SDA_ERR_UNSUPPORTED), (dict(kw=-1), sda.SDA_ERR_INVALID_ARG)]
    for change, want in bad:
        p = sda.dsa3d_problem(**{**good, **change})
        assert f(p) == want and g(p) == want, change
    p = sda.dsa3d_problem(**good)
    assert sda.lib().sda_dsa3d_fwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None) == sda.SDA_ERR_INVALID_ARG
    assert sda.lib().sda_dsa3d_fwd(ctypes.byref(p), fake + 8, fake, fake, fake, fake, fake, None) == \
        sda.SDA_ERR_INVALID_ARG  # misaligned Q
    assert sda.lib().sda_dsa3d_offsets(ctypes.byref(p), fake, fake, None, fake, fake, fake, None) == \
        sda.SDA_ERR_INVALID_ARG
    assert sda.lib().sda_dsa3d_fwd(None, fake, fake, fake, fake, fake, fake, None) == sda.SDA_ERR_INVALID_ARG


def test_dsa3d_backward_host_validation(L):
    """The 3D-DSA backward calls check their arguments and workspace before any launch."""
    import ctypes

    from dynamic_block_sparse_rank_gb300 import sda

    fake = 1 << 20
    good = dict(B=2, T=4, H=5, W=6, heads=3, d=128, kt=3, kh=3, kw=3)
    p = sda.dsa3d_problem(**good)
    assert sda.sda_dsa3d_offsets_bwd_workspace_size(p) == 2 * 4 * 5 * 6 * 3 * 128 * 4
    need = sda.sda_dsa3d_offsets_bwd_workspace_size(p)
    ob = lambda p, ws_bytes, *ptrs: sda.lib().sda_dsa3d_offsets_bwd(
        ctypes.byref(p), *(ptrs or (fake,) * 10), fake, ws_bytes, None)
    assert ob(p, need - 4) == sda.SDA_ERR_WORKSPACE
    assert ob(sda.dsa3d_problem(**{**good, "d": 96}), need) == sda.SDA_ERR_UNSUPPORTED
    assert ob(sda.dsa3d_problem(**{**good, "kh": 4}), need) == sda.SDA_ERR_INVALID_ARG
    assert ob(p, need, fake + 8, *(fake,) * 9) == sda.SDA_ERR_INVALID_ARG  # misaligned Q
    assert ob(p, need, fake, fake, None, *(fake,) * 7) == sda.SDA_ERR_INVALID_ARG  # no bc
    assert sda.lib().sda_dsa3d_offsets_bwd(ctypes.byref(p), *(fake,) * 10, fake + 4, need, None) == \
        sda.SDA_ERR_INVALID_ARG  # misaligned workspace
    assert sda.lib().sda_dsa3d_offsets_bwd_workspace_size(ctypes.byref(p), None) == sda.SDA_ERR_INVALID_ARG
    samples, cells = 2 * 3 * 120 * 27, 2 * 3 * (5 * 6 * 7 + 1)
    bneed = sda.sda_dsa3d_bwd_workspace_size(p)
    assert 32 * samples + 8 * cells <= bneed <= 32 * samples + 8 * cells + 5 * 256
    def bw(*ptrs, ws=fake, n=bneed):  # Q, K, V, offsets, LSE, dO, dQ, dK, dV, d_offsets; every case fails its checks
        assert len(ptrs) == 10
        return sda.lib().sda_dsa3d_bwd(ctypes.byref(p), *ptrs, ws, n, None)

    assert bw(*(fake,) * 6, fake + 4, *(fake,) * 3) == sda.SDA_ERR_INVALID_ARG  # misaligned dQ
    assert bw(*(fake,) * 8, None, fake) == sda.SDA_ERR_INVALID_ARG  # no dV
    assert bw(*(fake,) * 10, n=bneed - 1) == sda.SDA_ERR_WORKSPACE
    assert bw(*(fake,) * 10, ws=fake + 8) == sda.SDA_ERR_INVALID_ARG  # misaligned workspace
    assert bw(*(fake,) * 10, ws=None) == sda.SDA_ERR_INVALID_ARG
    big = sda.dsa3d_problem(**{**good, "B": 1, "heads": 1, "d": 64, "T": 100, "H": 1000, "W": 1000})
    size = ctypes.c_size_t()
    assert sda.lib().sda_dsa3d_bwd_workspace_size(ctypes.byref(big), ctypes.byref(size)) == \
        sda.SDA_ERR_UNSUPPORTED  # N S = 2.7e9 samples: past the 32-bit bucket indices
    assert sda.lib().sda_dsa3d_offsets_bwd_workspace_size(ctypes.byref(big), ctypes.byref(size)) == sda.SDA_OK
