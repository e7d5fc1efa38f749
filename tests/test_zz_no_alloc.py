"""The allocation-free pool entry point against the oracle and the rollout.

Some callers cannot allocate device memory when they call into the library:
their memory is owned by a planner that has handed out every byte, or their
allocator is locked while a workload is being captured.  For them the library
offers a pool selection whose scratch lives in a buffer compiled into the
library.  Its output must equal the oracle's pool on the same base logits
(ties at the cutoff included) and the rollout's own pool, on two calls in a
row that share the buffer, and a call must not allocate.  This file is
collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import cached_weights, device_requests, device_weights, gpu_debug, make_engine

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _oracle_pools(logits: np.ndarray, K: int) -> np.ndarray:
    rows = logits.astype(np.float64)[:, oracle.ROW_OFFSET:oracle.ROW_OFFSET + oracle.N_PROPOSALS]
    return np.stack([oracle.candidate_pool(rows[b], K) for b in range(logits.shape[0])]).astype(np.int32)


def _call_twice(logits_np: np.ndarray, K: int, want: np.ndarray):
    """Two calls in a row; the second must allocate nothing."""
    from speculative_decoding_draft_lm_gb300 import rollout as R
    B, _, V = logits_np.shape
    logits = torch.from_numpy(logits_np).cuda()
    outs = [torch.full((B, K), -1, dtype=torch.int32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):
        if call == 1:
            free0, _ = torch.cuda.mem_get_info()
            n_alloc0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        assert R.domino_candidate_pool_static(logits, B, V, K, outs[call]) == R.DOMINO_OK
        torch.cuda.synchronize()
        if call == 1:
            free1, _ = torch.cuda.mem_get_info()
            n_alloc1 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
            assert free1 == free0, (free0, free1)
            assert n_alloc1 == n_alloc0
        np.testing.assert_array_equal(outs[call].cpu().numpy(), want, err_msg=f"call {call}")


@pytest.mark.parametrize("V,B,K", [(20000, 4, 300), (151936, 8, 2048)])
def test_static_scratch_pool_equals_oracle_and_rollout_pool(V, B, K):
    sh = inputs.small_shape(V=V, dtype="bf16")
    w = cached_weights(sh, 0, ())
    r = inputs.make_requests(sh, list(range(60, 60 + B)))
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    ref = gpu_debug(eng, sh, device_requests(r), B, K, None)  # base logits and pool of the rollout
    eng.close()
    want = _oracle_pools(ref["logits"], K)
    np.testing.assert_array_equal(ref["pool"], want)
    _call_twice(ref["logits"], K, want)


@pytest.mark.parametrize("K", [1, 250, 2048])
def test_static_scratch_pool_cutoff_inside_a_tie_group(K):
    """600 ids share one exact score and the K-th place falls among them: the
    lowest ids of the group must be taken, as the oracle takes them."""
    V, B = 30011, 3
    rng = np.random.default_rng(K)
    logits = rng.standard_normal((B, 16, V)).astype(np.float32)
    for b in range(B):
        ids = rng.permutation(V)
        n_above = max(0, K - 300)
        above, tied = ids[:n_above], ids[n_above:n_above + 600]
        logits[b, :, :] = np.minimum(logits[b], 2.0)
        logits[b, 1 + rng.integers(0, 15, size=above.size), above] = 3.0 + rng.random(above.size, dtype=np.float32)
        logits[b, 1:, tied] = np.minimum(logits[b, 1:, tied], 2.5)
        logits[b, 1 + rng.integers(0, 15, size=tied.size), tied] = 2.75  # exactly equal maxima
        logits[b, 0, :] = 9.0  # row 0 is not part of the score
    want = _oracle_pools(logits, K)
    for b in range(B):
        score = logits[b, 1:].max(axis=0)
        kth = np.sort(score)[::-1][K - 1]
        assert kth == np.float32(2.75) and (score == kth).sum() == 600
    _call_twice(logits, K, want)


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
