"""The predictor entry point that allocates nothing (sda_predict_blocks_noalloc).

It exists for callers that cannot allocate device memory and so have no
workspace to hand over.  These tests call it through the C ABI and compare it
with sda_predict_blocks run on a caller workspace, on calls in a row that
reuse the same built-in scratch.  The file is named to be collected last.
"""
import numpy as np
import pytest

from dynamic_block_sparse_rank_gb300 import inputs
from tests.parity_util import dev, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_block_sparse_rank_gb300 import sda as s

    s.lib()
    return s


def _both(sda, wl, seed):
    x = inputs.generate(wl, seed=seed, names=("Q", "K", "Wq", "Wk"))
    p = sda.problem_from_workload(wl)
    nb, k = sda.sda_num_blocks(p)
    Q, K, Wq, Wk = (dev(x[n], wl.dtype) for n in ("Q", "K", "Wq", "Wk"))
    out = []
    for use_ws in (True, False):
        idx = torch.full((wl.B, wl.heads, nb, k), -1, dtype=torch.int32, device="cuda")
        score = torch.full((wl.B, wl.heads, nb, nb), float("nan"), dtype=torch.float32, device="cuda")
        if use_ws:
            ws = torch.empty(sda.sda_workspace_size(p, sda.SDA_OP_PREDICT), dtype=torch.uint8, device="cuda")
            sda.sda_predict_blocks(p, Q, K, Wq, Wk, idx, score, ws)
        else:
            sda.sda_predict_blocks_noalloc(p, Q, K, Wq, Wk, idx, score)
        torch.cuda.synchronize()
        out.append((idx.cpu().numpy(), host(score)))
    return out


def test_noalloc_predictor_matches_workspace_predictor_on_consecutive_calls(sda):
    cases = [
        (inputs.Workload("noalloc_a", 1, 3, 5, 12, 20, 64, 2, 8, 8, 16, 0.4, "bf16", 3.0, 16), 1),
        (inputs.Workload("noalloc_b", 1, 2, 4, 16, 17, 128, 2, 8, 8, 32, 0.3, "bf16", 4.0, 32), 2),
        (inputs.WORKLOADS["fwd_8k"], 0),
        (inputs.WORKLOADS["tiny_f32_256"], 0),
    ]
    for wl, seed in cases:  # consecutive calls on the shared scratch, different shapes and contents
        (idx_ws, sc_ws), (idx_na, sc_na) = _both(sda, wl, seed)
        assert np.array_equal(idx_na, idx_ws), wl.name
        assert np.all(np.isfinite(sc_na))
        rel = np.abs(sc_na - sc_ws).max() / np.abs(sc_ws).max()
        assert rel <= 1e-5, (wl.name, rel)
    assert sda.sda_get_device_status() == sda.SDA_OK


def test_noalloc_rejects_problems_beyond_its_scratch(sda):
    wl = inputs.WORKLOADS["train_524k"]  # needs 537 MB of predictor scratch
    p = sda.problem_from_workload(wl)
    assert sda.sda_workspace_size(p, sda.SDA_OP_PREDICT) > 32 << 20
    before = sda.sda_kernel_launch_count()
    with pytest.raises(sda.SdaError) as e:
        sda.sda_predict_blocks_noalloc(p, 16, 16, 16, 16, 16, None)
    assert e.value.status == sda.SDA_ERR_WORKSPACE
    assert sda.sda_kernel_launch_count() == before
