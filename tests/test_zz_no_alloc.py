"""The allocation-free pool entry point against the rollout's own pool.

Some callers cannot allocate device memory when they call into the library
(their memory is owned by a planner, or their allocator is locked while a
workload is captured).  For them the library offers a pool selection whose
scratch lives in a buffer compiled into the library.  This file is collected
last on purpose: if it fails, a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest

from speculative_decoding_draft_lm_gb300 import inputs

from helpers import cached_weights, device_requests, device_weights, gpu_debug, make_engine

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V,B,K", [(20000, 4, 300), (151936, 8, 2048)])
def test_static_scratch_pool_equals_rollout_pool(V, B, K):
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(V=V, dtype="bf16")
    w = cached_weights(sh, 0, ())
    r = inputs.make_requests(sh, list(range(60, 60 + B)))
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    ref = gpu_debug(eng, sh, device_requests(r), B, K, None)  # base logits and pool of the rollout
    logits = torch.from_numpy(ref["logits"]).cuda()
    for call in range(2):  # two calls in a row share (and overwrite) the scratch
        out = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
        assert R.domino_candidate_pool_static(logits, B, V, K, out) == R.DOMINO_OK
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), ref["pool"], err_msg=f"call {call}")
    eng.close()


def test_static_scratch_limits_are_reported():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    V = 151936
    B = R.DOMINO_STATIC_SCRATCH_FLOATS // V + 1
    logits = torch.zeros((1,), dtype=torch.float32, device="cuda")
    out = torch.zeros((1,), dtype=torch.int32, device="cuda")
    assert R.domino_candidate_pool_static(logits, B, V, 10, out) == R.DOMINO_ERR_SCRATCH_LIMIT
    assert R.domino_candidate_pool_static(logits, 1, V, 0, out) == R.DOMINO_ERR_INVALID_ARG
    assert R.domino_candidate_pool_static(logits, 1, V, V, out) == R.DOMINO_ERR_INVALID_ARG
    assert R.domino_candidate_pool_static(None, 1, V, 10, out) == R.DOMINO_ERR_INVALID_ARG
