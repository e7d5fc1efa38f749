"""A device-side wait that runs out reports DOMINO_ERR_TIMEOUT and leaves the
context usable (page "Add correctness-first Domino support to DFlash V2",
section "Supported and numerical scope": clear errors, no silent fallback).

The one-shot test hook withholds one CTA's arrival at a grid barrier of the
persistent driver, so every CTA's bounded wait there expires: nothing faults
or hangs, the kernel returns, and the host reads the timeout status."""
import time

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import TOL, cached_oracle_weights, cached_weights, check_free_run, device_requests, device_weights, \
    make_engine

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _scales(sh):
    return (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5), ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


# grid-barrier kernel: barrier 1 follows the seed update, 3 the first
# projector phase, 4 the first correction phase; tagged-exchange kernel:
# publication 1 is the CTA's GRU units after the seed, 3 the first step's
# best, 4 its units after update 2
@pytest.mark.parametrize("driver", [2, 3], ids=["tagged", "grid"])
@pytest.mark.parametrize("barrier", [1, 3, 4])
@pytest.mark.parametrize("B,K", [(1, 0), (3, 100)])
def test_withheld_barrier_arrival_times_out_and_recovers(barrier, B, K, driver):
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    sc = _scales(sh)
    w = cached_weights(sh, 0, sc)
    ow = cached_oracle_weights(sh, 0, sc)
    r = inputs.make_requests(sh, list(range(70, 70 + B)))
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    eng.set_driver(driver)
    dreq = device_requests(r)
    eng.run(*dreq, K=K)  # an ordinary run first
    assert eng.status() == R.DOMINO_OK

    assert R.domino_rollout_debug_drop_barrier_arrival(eng.ctx, barrier) == R.DOMINO_OK
    t0 = time.monotonic()
    eng.run(*dreq, K=K)
    st = eng.status()  # synchronises: the kernel has returned
    waited = time.monotonic() - t0
    assert st == R.DOMINO_ERR_TIMEOUT, R.domino_rollout_strerror(st)
    assert waited < 5.0, waited  # bounded waits (200 ms each), not a hang

    # the hook was one-shot and the context is still usable
    out = eng.run(*dreq, K=K)
    assert eng.status() == R.DOMINO_OK
    check_free_run(o, out.cpu().numpy(), TOL["bf16"])
    eng.close()


def test_hook_rejects_negative_barrier():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    eng = make_engine(sh, max_B=1, max_K=0, dw=device_weights(cached_weights(sh, 0, _scales(sh))))
    assert R.domino_rollout_debug_drop_barrier_arrival(eng.ctx, -1) == R.DOMINO_ERR_INVALID_ARG
    assert R.domino_rollout_debug_drop_barrier_arrival(None, 1) == R.DOMINO_ERR_INVALID_ARG
    assert R.domino_rollout_debug_drop_barrier_arrival(eng.ctx, 0) == R.DOMINO_OK
    eng.close()
