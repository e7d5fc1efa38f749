"""Per-step term s of projector layer 1 computed inside the library from the
backbone hidden rows (run with s = NULL after load_backbone_proj), against
the oracle's backbone_s on the same seeded inputs."""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import (TOL, cached_oracle_weights, cached_weights, check_against_oracle, check_free_run,
                     device_requests, device_weights, gpu_debug, make_engine)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _scales(sh):
    return (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5), ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


def _run(sh, B, K, scales=(), hid_scale=0.02, driver=None, seeds=None):
    from speculative_decoding_draft_lm_gb300.rollout import to_device
    w = cached_weights(sh, 0, scales)
    ow = cached_oracle_weights(sh, 0, scales)
    W_hid = inputs.make_fc1_hidden(sh, seed=5, scale=hid_scale)
    r = inputs.make_requests(sh, seeds or list(range(300, 300 + B)))
    o = oracle.rollout(ow, r["hidden"], None, r["verified"], K, W_hid=W_hid)
    eng = make_engine(sh, max_B=B, max_K=K if 0 < K < sh.V else 0, dw=device_weights(w))
    eng.load_backbone_proj(to_device(W_hid))
    if driver is not None:
        eng.set_driver(driver)
    hid, _, ver = device_requests(r)
    g = gpu_debug(eng, sh, (hid, None, ver), B, K, o["tokens"])
    check_against_oracle(ow, o, g, sh, K)
    free = eng.run(hid, None, ver, K=K)
    torch.cuda.synchronize()
    assert eng.status() == 0
    check_free_run(o, free.cpu().numpy(), TOL[sh.dtype])
    eng.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("B,K", [(1, 0), (1, 100), (3, 0), (3, 100), (16, 0), (16, 100)])
def test_small_in_library_s(dtype, B, K):
    sh = inputs.small_shape(dtype=dtype)
    _run(sh, B, K, scales=_scales(sh), hid_scale=0.1)


def test_small_in_library_s_both_drivers():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    for drv in (R.DOMINO_DRIVER_KERNELS, R.DOMINO_DRIVER_PERSISTENT, R.DOMINO_DRIVER_PERSISTENT_GRID):
        _run(sh, 1, 0, scales=_scales(sh), hid_scale=0.1, driver=drv)


@pytest.mark.parametrize("name", ["qwen3_8b_b1_k0", "qwen3_8b_b8_k2048"])
def test_full_size_in_library_s(name):
    wl = inputs.WORKLOADS[name]
    _run(wl.shape, wl.B, wl.K, seeds=list(wl.request_seeds))


def test_null_s_without_backbone_weight_is_rejected():
    from speculative_decoding_draft_lm_gb300 import rollout as R
    sh = inputs.small_shape(dtype="bf16")
    eng = make_engine(sh, max_B=2, max_K=0, dw=device_weights(cached_weights(sh, 0, _scales(sh))))
    r = inputs.make_requests(sh, [1, 2])
    hid, _, ver = device_requests(r)
    with pytest.raises(R.DominoError):
        eng.run(hid, None, ver, K=0)
    eng.close()
