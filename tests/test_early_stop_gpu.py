"""Early-stopped rollout (the b8 serving variant: the block-16 draft is kept,
the target verifies fewer positions): the n proposals equal the first n of
the full rollout, on both drivers, in full-vocabulary and pool mode."""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import (TOL, cached_oracle_weights, cached_weights, device_requests, device_weights, gpu_debug,
                     make_engine, oracle_scores_at)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _scales(sh):
    return (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5), ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


def _check_prefix(ow, o, g, sh, K, n):
    tol = TOL[sh.dtype]
    full = K == 0 or K >= sh.V
    assert g["status"] == 0, g["status"]
    assert np.abs(g["logits"] - o["L"]).max() <= tol
    nh = max(2, n)  # GRU states written: the two-token prefix, then one per corrected step but the last
    assert np.abs(g["h"][:, :nh] - o["h"][:, :nh]).max() <= tol
    if n > 1:
        assert np.abs(g["z"][:, :n - 1] - o["z"][:, :n - 1]).max() <= tol
    assert (g["tokens"][:, n:] == -1).all()
    for b in range(o["tokens"].shape[0]):
        for j in range(n):
            gt, ot = int(g["tokens"][b, j]), int(o["tokens"][b, j])
            if j == 0:
                row = o["L"][b, oracle.ROW_OFFSET]
                gval, oval = row[gt], row[ot]
            else:
                if not full:
                    assert gt in set(g["pool"][b].tolist())
                gval, oval = oracle_scores_at(ow, o, b, j, [gt, ot])
            if o["margin"][b, j] > tol:
                assert gt == ot, f"request {b} proposal {j}: gpu {gt} oracle {ot}"
            else:
                assert gval >= oval - tol


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("B,K", [(1, 0), (1, 100), (3, 0), (3, 100)])
def test_early_stop_matches_full_prefix(dtype, B, K):
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype=dtype)
    sc = _scales(sh)
    w = cached_weights(sh, 0, sc)
    ow = cached_oracle_weights(sh, 0, sc)
    r = inputs.make_requests(sh, list(range(70, 70 + B)))
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    dreq = device_requests(r)
    drivers = [R.DOMINO_DRIVER_KERNELS]
    if K > 0 or B == 1:
        drivers += [R.DOMINO_DRIVER_PERSISTENT, R.DOMINO_DRIVER_PERSISTENT_GRID]
    for drv in drivers:
        eng.set_driver(drv)
        eng.set_proposals(15)
        whole = eng.run(*dreq, K=K).cpu().numpy()
        assert eng.status() == 0
        for n in (1, 2, 7, 14):
            eng.set_proposals(n)
            g = gpu_debug(eng, sh, dreq, B, K, o["tokens"])
            _check_prefix(ow, o, g, sh, K, n)
            part = eng.run(*dreq, K=K)
            torch.cuda.synchronize()
            assert eng.status() == 0
            part = part.cpu().numpy()
            # same kernels, same inputs: the prefix is bit-identical to the full run
            np.testing.assert_array_equal(part[:, :n], whole[:, :n])
            assert (part[:, n:] == -1).all()
    eng.close()


def test_set_proposals_rejects_out_of_range():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="fp32")
    eng = make_engine(sh, max_B=1, max_K=0, dw=device_weights(cached_weights(sh, 0, _scales(sh))))
    for n in (0, 16, -1):
        with pytest.raises(R.DominoError):
            eng.set_proposals(n)
    eng.close()
