"""The drivers of the 14 dependent steps (one launch per phase, and the two
persistent cooperative kernels: tagged data exchanges or grid barriers) agree
with the oracle and with each other."""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import (TOL, cached_oracle_weights, cached_weights, check_against_oracle, device_requests,
                     device_weights, gpu_debug, make_engine)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _scales(sh):
    return (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5), ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("B,K", [(1, 0), (1, 100), (3, 100), (5, 7), (8, 100)])
def test_persistent_matches_kernels_and_oracle(dtype, B, K):
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype=dtype)
    sc = _scales(sh)
    w = cached_weights(sh, 0, sc)
    ow = cached_oracle_weights(sh, 0, sc)
    r = inputs.make_requests(sh, list(range(40, 40 + B)))
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    dreq = device_requests(r)
    outs = {}
    persistent = (R.DOMINO_DRIVER_PERSISTENT, R.DOMINO_DRIVER_PERSISTENT_GRID)
    for drv in (R.DOMINO_DRIVER_KERNELS,) + persistent:
        eng.set_driver(drv)
        g = gpu_debug(eng, sh, dreq, B, K, o["tokens"], want_scores=True)
        check_against_oracle(ow, o, g, sh, K)
        free = eng.run(*dreq, K=K)
        torch.cuda.synchronize()
        assert eng.status() == 0
        outs[drv] = (g, free.cpu().numpy())
    gk, fk = outs[R.DOMINO_DRIVER_KERNELS]
    tol = TOL[dtype]
    for drv in persistent:
        gp, fp = outs[drv]
        np.testing.assert_allclose(gp["h"], gk["h"], rtol=0, atol=tol)
        np.testing.assert_allclose(gp["z"], gk["z"], rtol=0, atol=tol)
        # free-running chains agree wherever the oracle's decision is not a near tie
        for b in range(B):
            for j in range(15):
                if o["margin"][b, j] <= tol:
                    break
                assert fp[b, j] == fk[b, j] == o["tokens"][b, j]
    eng.close()


def test_persistent_repeat_runs_are_identical():
    """Same inputs twice through the persistent driver: bit-identical tokens."""
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    sc = _scales(sh)
    w = cached_weights(sh, 0, sc)
    r = inputs.make_requests(sh, [77])
    eng = make_engine(sh, max_B=1, max_K=100, dw=device_weights(w))
    dreq = device_requests(r)
    for drv in (R.DOMINO_DRIVER_PERSISTENT, R.DOMINO_DRIVER_PERSISTENT_GRID):
        eng.set_driver(drv)
        for K in (0, 100):
            a = eng.run(*dreq, K=K).cpu().numpy()
            b = eng.run(*dreq, K=K).cpu().numpy()
            assert (a == b).all()
    eng.close()


def test_persistent_driver_rejects_unsupported_batch():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    w = cached_weights(sh, 0, ())
    eng = make_engine(sh, max_B=4, max_K=0, dw=device_weights(w))
    eng.set_driver(R.DOMINO_DRIVER_PERSISTENT)
    r = inputs.make_requests(sh, [1, 2, 3, 4])
    hid, s, ver = device_requests(r)
    out = torch.empty((4, 15), dtype=torch.int32, device="cuda")
    # full vocabulary with B > 1 runs on the tensor-core kernels instead
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 4, 0, out) == R.DOMINO_ERR_UNSUPPORTED
    eng.set_driver(R.DOMINO_DRIVER_PERSISTENT_GRID)
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 4, 0, out) == R.DOMINO_ERR_UNSUPPORTED
    eng.close()
