"""Thin ctypes binding of libsda.so (include/sda.h): argument marshalling only.

Every entry point keeps the C name and takes device tensors (torch) or raw
device pointers (int).  Outputs and workspace are allocated by the caller;
nothing here computes.  A missing or unloadable library raises immediately:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsda.so")

(SDA_OK, SDA_ERR_INVALID_ARG, SDA_ERR_UNSUPPORTED, SDA_ERR_WORKSPACE, SDA_ERR_CUDA, SDA_ERR_DEVICE_TIMEOUT,
 SDA_ERR_DEVICE_BAD_INDEX, SDA_ERR_DEVICE_RANGE) = range(8)
SDA_F32, SDA_BF16 = 0, 1
SDA_OP_PREDICT, SDA_OP_BWD, SDA_OP_TRAIN, SDA_OP_PREDICTOR_GRAD = 0, 1, 2, 3

EXPORTS = ("sda_num_blocks", "sda_workspace_size", "sda_predict_blocks", "sda_attn_fwd", "sda_attn_bwd",
           "sda_attn_fwd_train", "sda_attn_bwd_train", "sda_predictor_grad",
           "sda_attn_bwd_prepare", "sda_attn_bwd_dq", "sda_attn_bwd_dkdv", "sda_attn_bwd_partition", "sda_merge_states", "sda_merge_states_bwd",
           "sda_get_device_status", "sda_kernel_launch_count", "sda_predict_blocks_noalloc", "sda_selftest_wait_timeout", "sda_status_string",
           "sda_dsa3d_offsets", "sda_dsa3d_fwd", "sda_dsa3d_bwd", "sda_dsa3d_bwd_workspace_size", "sda_dsa3d_offsets_bwd_workspace_size",
           "sda_dsa3d_offsets_bwd")


class SdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("heads", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("W", ctypes.c_int), ("head_dim", ctypes.c_int), ("bt", ctypes.c_int), ("bh", ctypes.c_int),
                ("bw", ctypes.c_int), ("rank", ctypes.c_int), ("keep_ratio", ctypes.c_double),
                ("dtype", ctypes.c_int), ("softmax_scale", ctypes.c_float)]


class Dsa3dProblem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("heads", ctypes.c_int), ("d", ctypes.c_int), ("kt", ctypes.c_int), ("kh", ctypes.c_int),
                ("kw", ctypes.c_int), ("scale", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libsda.so (built by `dynamic_block_sparse_rank_gb300.build`); raise if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m dynamic_block_sparse_rank_gb300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, pr = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(Problem)
        L.sda_num_blocks.argtypes = [pr, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.sda_workspace_size.argtypes = [pr, i32, ctypes.POINTER(sz)]
        L.sda_predict_blocks.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sda_attn_fwd.argtypes = [pr, vp, vp, vp, vp, i32, i32, vp, vp, vp, i32, vp]
        L.sda_attn_bwd.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]
        L.sda_attn_bwd_prepare.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sda_attn_fwd_train.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sda_predictor_grad.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sda_attn_bwd_train.argtypes = [pr, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz, vp]
        L.sda_attn_bwd_partition.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, i32, vp, sz,
                                             vp]
        L.sda_attn_bwd_dq.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]
        L.sda_attn_bwd_dkdv.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]
        L.sda_predict_blocks_noalloc.argtypes = [pr, vp, vp, vp, vp, vp, vp, vp]
        L.sda_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp, vp]
        L.sda_kernel_launch_count.argtypes = []
        L.sda_kernel_launch_count.restype = ctypes.c_ulonglong
        L.sda_merge_states.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, i32, i32, i32, i32, vp, vp, vp]
        L.sda_merge_states_bwd.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp, i32, i32, i32, i32,
                                           i32, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
        dp = ctypes.POINTER(Dsa3dProblem)
        L.sda_dsa3d_offsets.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp]
        L.sda_dsa3d_fwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp]
        L.sda_dsa3d_bwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sda_dsa3d_bwd_workspace_size.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        L.sda_dsa3d_offsets_bwd_workspace_size.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        L.sda_dsa3d_offsets_bwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sda_get_device_status.argtypes = [vp]
        L.sda_status_string.argtypes = [i32]
        L.sda_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name not in ("sda_status_string", "sda_kernel_launch_count"):
                getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().sda_status_string(int(s)).decode()


def problem(B, heads, T, H, W, head_dim, bt, bh, bw, rank, keep_ratio, dtype, softmax_scale=0.0) -> Problem:
    dt = {"f32": SDA_F32, "bf16": SDA_BF16}.get(dtype, dtype)
    return Problem(B, heads, T, H, W, head_dim, bt, bh, bw, rank, float(keep_ratio), int(dt), float(softmax_scale))


def problem_from_workload(wl, softmax_scale=0.0) -> Problem:
    return problem(wl.B, wl.heads, wl.T, wl.H, wl.W, wl.d, wl.bt, wl.bh, wl.bw, wl.rank, wl.keep, wl.dtype,
                   softmax_scale)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != SDA_OK:
        raise SdaError(st, where)


def sda_num_blocks(p: Problem) -> tuple[int, int]:
    nb, k = ctypes.c_int(), ctypes.c_int()
    _check(lib().sda_num_blocks(ctypes.byref(p), ctypes.byref(nb), ctypes.byref(k)), "sda_num_blocks")
    return nb.value, k.value


def sda_workspace_size(p: Problem, op: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().sda_workspace_size(ctypes.byref(p), int(op), ctypes.byref(b)), "sda_workspace_size")
    return b.value


def _nbytes(ws):
    if ws is None:
        return 0
    if isinstance(ws, tuple):  # (pointer, bytes)
        return ws[1]
    return ws.numel() * ws.element_size()


def _wsptr(ws):
    return ws[0] if isinstance(ws, tuple) else _ptr(ws)


def sda_predict_blocks(p, Q, K, Wq, Wk, block_idx, block_score=None, ws=None, stream=None):
    _check(lib().sda_predict_blocks(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), _ptr(block_idx),
                                    _ptr(block_score), _wsptr(ws), _nbytes(ws), _stream(stream)),
           "sda_predict_blocks")


def sda_attn_fwd(p, Q, K, V, block_idx, O, LSE, kb_begin=0, kb_end=None, qb_active=None, stream=None,
                 out_dtype=None):
    """out_dtype: None (the problem's dtype), "f32" or "bf16"."""
    if kb_end is None:
        kb_end = sda_num_blocks(p)[0]
    od = p.dtype if out_dtype is None else {"f32": SDA_F32, "bf16": SDA_BF16}.get(out_dtype, out_dtype)
    _check(lib().sda_attn_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(block_idx), int(kb_begin),
                              int(kb_end), _ptr(qb_active), _ptr(O), _ptr(LSE), int(od), _stream(stream)),
           "sda_attn_fwd")


def sda_attn_bwd(p, Q, K, V, O, LSE, dO, block_idx, dQ, dK, dV, grad_dtype, ws, stream=None):
    gd = {"f32": SDA_F32, "bf16": SDA_BF16}.get(grad_dtype, grad_dtype)
    _check(lib().sda_attn_bwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO),
                              _ptr(block_idx), _ptr(dQ), _ptr(dK), _ptr(dV), int(gd), _wsptr(ws), _nbytes(ws),
                              _stream(stream)), "sda_attn_bwd")


def sda_predictor_grad(p, Q, K, Wq, Wk, dWq, dWk, loss, ws, s_out=None, t_out=None, stream=None):
    _check(lib().sda_predictor_grad(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), _ptr(dWq), _ptr(dWk),
                                    _ptr(loss), _ptr(s_out), _ptr(t_out), _wsptr(ws), _nbytes(ws), _stream(stream)),
           "sda_predictor_grad")


def sda_attn_fwd_train(p, Q, K, V, block_idx, O, LSE, ws, stream=None):
    _check(lib().sda_attn_fwd_train(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(block_idx), _ptr(O), _ptr(LSE),
                                    _wsptr(ws), _nbytes(ws), _stream(stream)), "sda_attn_fwd_train")


def sda_attn_bwd_train(p, LSE, dO, block_idx, dQ, dK, dV, grad_dtype, ws, phases=7, stream=None):
    gd = {"f32": SDA_F32, "bf16": SDA_BF16}.get(grad_dtype, grad_dtype)
    _check(lib().sda_attn_bwd_train(ctypes.byref(p), _ptr(LSE), _ptr(dO), _ptr(block_idx), _ptr(dQ), _ptr(dK),
                                    _ptr(dV), int(gd), int(phases), _wsptr(ws), _nbytes(ws), _stream(stream)),
           "sda_attn_bwd_train")


def sda_attn_bwd_partition(p, Q, K, V, O, LSE, dO, dLSE, block_idx, dQ, dK, dV, grad_dtype, ws, kb_begin=0,
                           kb_end=None, qb_active=None, stream=None):
    gd = {"f32": SDA_F32, "bf16": SDA_BF16}.get(grad_dtype, grad_dtype)
    if kb_end is None:
        kb_end = sda_num_blocks(p)[0]
    _check(lib().sda_attn_bwd_partition(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO),
                                        _ptr(dLSE), _ptr(block_idx), int(kb_begin), int(kb_end), _ptr(qb_active),
                                        _ptr(dQ), _ptr(dK), _ptr(dV), int(gd), _wsptr(ws), _nbytes(ws),
                                        _stream(stream)), "sda_attn_bwd_partition")


def sda_attn_bwd_prepare(p, Q, K, V, O, LSE, dO, block_idx, ws, stream=None):
    _check(lib().sda_attn_bwd_prepare(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO),
                                      _ptr(block_idx), _wsptr(ws), _nbytes(ws), _stream(stream)),
           "sda_attn_bwd_prepare")


def sda_attn_bwd_dq(p, Q, K, V, LSE, dO, block_idx, dQ, grad_dtype, ws, stream=None):
    gd = {"f32": SDA_F32, "bf16": SDA_BF16}.get(grad_dtype, grad_dtype)
    _check(lib().sda_attn_bwd_dq(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(LSE), _ptr(dO), _ptr(block_idx),
                                 _ptr(dQ), int(gd), _wsptr(ws), _nbytes(ws), _stream(stream)), "sda_attn_bwd_dq")


def sda_attn_bwd_dkdv(p, Q, K, V, LSE, dO, block_idx, dK, dV, grad_dtype, ws, stream=None):
    gd = {"f32": SDA_F32, "bf16": SDA_BF16}.get(grad_dtype, grad_dtype)
    _check(lib().sda_attn_bwd_dkdv(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(LSE), _ptr(dO),
                                   _ptr(block_idx), _ptr(dK), _ptr(dV), int(gd), _wsptr(ws), _nbytes(ws),
                                   _stream(stream)), "sda_attn_bwd_dkdv")


def sda_predict_blocks_noalloc(p, Q, K, Wq, Wk, block_idx, block_score=None, stream=None):
    """sda_predict_blocks with the library's built-in scratch instead of a caller workspace."""
    _check(lib().sda_predict_blocks_noalloc(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), _ptr(block_idx),
                                            _ptr(block_score), _stream(stream)), "sda_predict_blocks_noalloc")


def sda_selftest_wait_timeout(limit_us, completed, stream=None):
    _check(lib().sda_selftest_wait_timeout(int(limit_us), _ptr(completed), _stream(stream)),
           "sda_selftest_wait_timeout")


def sda_kernel_launch_count() -> int:
    return int(lib().sda_kernel_launch_count())


def sda_merge_states(O_parts, LSE_parts, B, N, heads, head_dim, dtype, O_out, LSE_out, stream=None):
    n = len(O_parts)
    dt = {"f32": SDA_F32, "bf16": SDA_BF16}.get(dtype, dtype)
    optrs = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in O_parts])
    lptrs = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in LSE_parts])
    _check(lib().sda_merge_states(n, optrs, lptrs, int(B), int(N), int(heads), int(head_dim), int(dt), _ptr(O_out),
                                  _ptr(LSE_out), _stream(stream)), "sda_merge_states")


def sda_merge_states_bwd(O_parts, LSE_parts, dO, dLSE, B, N, heads, head_dim, dtype, dO_parts, dLSE_parts,
                         stream=None):
    n = len(O_parts)
    dt = {"f32": SDA_F32, "bf16": SDA_BF16}.get(dtype, dtype)
    arr = lambda xs: (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in xs])
    _check(lib().sda_merge_states_bwd(n, arr(O_parts), arr(LSE_parts), _ptr(dO), _ptr(dLSE), int(B), int(N),
                                      int(heads), int(head_dim), int(dt), arr(dO_parts), arr(dLSE_parts),
                                      _stream(stream)), "sda_merge_states_bwd")


def sda_get_device_status(stream=None) -> int:
    return lib().sda_get_device_status(_stream(stream))


def dsa3d_problem(B, T, H, W, heads, d, kt, kh, kw, scale=0.0) -> Dsa3dProblem:
    return Dsa3dProblem(B, T, H, W, heads, d, kt, kh, kw, float(scale))


def sda_dsa3d_offsets(p: Dsa3dProblem, Q, Wc, bc, Wl, bl, offsets, stream=None):
    _check(lib().sda_dsa3d_offsets(ctypes.byref(p), _ptr(Q), _ptr(Wc), _ptr(bc), _ptr(Wl), _ptr(bl), _ptr(offsets),
                                   _stream(stream)), "sda_dsa3d_offsets")


def sda_dsa3d_fwd(p: Dsa3dProblem, Q, K, V, offsets, O, LSE, stream=None):
    _check(lib().sda_dsa3d_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(offsets), _ptr(O), _ptr(LSE),
                               _stream(stream)), "sda_dsa3d_fwd")


def sda_dsa3d_bwd_workspace_size(p: Dsa3dProblem) -> int:
    b = ctypes.c_size_t()
    _check(lib().sda_dsa3d_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b)), "sda_dsa3d_bwd_workspace_size")
    return b.value


def sda_dsa3d_bwd(p: Dsa3dProblem, Q, K, V, offsets, LSE, dO, dQ, dK, dV, d_offsets, ws, stream=None):
    _check(lib().sda_dsa3d_bwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(offsets), _ptr(LSE), _ptr(dO),
                               _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(d_offsets), _ptr(ws), _nbytes(ws),
                               _stream(stream)), "sda_dsa3d_bwd")


def sda_dsa3d_offsets_bwd_workspace_size(p: Dsa3dProblem) -> int:
    b = ctypes.c_size_t()
    _check(lib().sda_dsa3d_offsets_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b)),
           "sda_dsa3d_offsets_bwd_workspace_size")
    return b.value


def sda_dsa3d_offsets_bwd(p: Dsa3dProblem, Q, Wc, bc, Wl, d_offsets, dQ, dWc, dbc, dWl, dbl, ws, stream=None):
    _check(lib().sda_dsa3d_offsets_bwd(ctypes.byref(p), _ptr(Q), _ptr(Wc), _ptr(bc), _ptr(Wl), _ptr(d_offsets),
                                       _ptr(dQ), _ptr(dWc), _ptr(dbc), _ptr(dWl), _ptr(dbl), _ptr(ws), _nbytes(ws),
                                       _stream(stream)), "sda_dsa3d_offsets_bwd")
