"""Stage C of the tensor-parallel rollout on one GPU: the candidate pool
built from P shard-local top-K selections and a global merge equals the
direct selection (stage B) and the oracle's candidate_pool_compact, ties
included, and the proposal chain is unchanged."""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import (cached_oracle_weights, cached_weights, check_against_oracle, device_requests, device_weights,
                     gpu_debug, make_engine)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _scales(sh):
    return (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5), ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


def _compare(sh, w, r, B, K, parts, ow=None):
    ow = ow or oracle.OracleWeights(w)
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    dreq = device_requests(r)
    direct = gpu_debug(eng, sh, dreq, B, K, o["tokens"])
    free_direct = eng.run(*dreq, K=K).cpu().numpy()
    for P in parts:
        eng.set_vocab_partitions(P)
        g = gpu_debug(eng, sh, dreq, B, K, o["tokens"])
        for b in range(B):
            rows = o["L"][b, oracle.ROW_OFFSET:oracle.ROW_OFFSET + 15]
            assert g["pool"][b].tolist() == oracle.candidate_pool_compact(rows, K, P).tolist(), (P, b)
        np.testing.assert_array_equal(g["pool"], direct["pool"])
        np.testing.assert_array_equal(g["tokens"], direct["tokens"])
        check_against_oracle(ow, o, g, sh, K)
        free = eng.run(*dreq, K=K).cpu().numpy()
        assert eng.status() == 0
        np.testing.assert_array_equal(free, free_direct)
    eng.close()


@pytest.mark.parametrize("K", [1, 100, 300, 999])
def test_compact_pool_small(K):
    sh = inputs.small_shape(dtype="bf16")
    sc = _scales(sh)
    r = inputs.make_requests(sh, [21, 22, 23])
    _compare(sh, cached_weights(sh, 0, sc), r, 3, K, (2, 3, 4, 8), cached_oracle_weights(sh, 0, sc))


@pytest.mark.parametrize("K", [50, 300, 600])
def test_compact_pool_cutoff_inside_a_tie_group(K):
    sh = inputs.small_shape(V=2000, dtype="bf16")
    sc = _scales(sh)
    w = {k: v.copy() for k, v in cached_weights(sh, 0, sc).items()}
    w["lm_head"][1234] = inputs.to_bf16_bits((oracle.widen(w["lm_head"][1234]) * 6.0).astype(np.float32))
    for v in np.random.default_rng(3).choice(sh.V, size=600, replace=False):
        w["lm_head"][v] = w["lm_head"][1234]
    r = inputs.make_requests(sh, [5, 6])
    _compare(sh, w, r, 2, K, (2, 3, 8))


def test_compact_pool_full_size_tp2():
    """The pages' TP2 case: two shards of the Qwen3-8B-shaped vocabulary, B=8, K=2048."""
    wl = inputs.WORKLOADS["qwen3_8b_b8_k2048"]
    sh = wl.shape
    r = inputs.make_requests(sh, list(wl.request_seeds))
    _compare(sh, cached_weights(sh, 0, ()), r, wl.B, wl.K, (2,), cached_oracle_weights(sh, 0, ()))


def test_vocab_partitions_range():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    eng = make_engine(sh, max_B=1, max_K=10, dw=device_weights(cached_weights(sh, 0, _scales(sh))))
    for P in (0, 9, -2):
        with pytest.raises(R.DominoError):
            eng.set_vocab_partitions(P)
    eng.close()
