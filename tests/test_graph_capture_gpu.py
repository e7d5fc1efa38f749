"""run() is asynchronous and makes no host synchronisation, so a whole block
rollout can be captured in a CUDA graph and replayed: the persistent drivers
(cooperative + programmatic dependent launch; the tagged-exchange one draws
its tags from a run counter in device memory, so replays do not reuse them),
the batched per-phase driver with the cluster pool selection, and the
tensor-core GRU path."""
import numpy as np
import pytest

from speculative_decoding_draft_lm_gb300 import inputs

from helpers import cached_weights, device_requests, device_weights, make_engine

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _scales(sh):
    return (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5), ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


@pytest.mark.parametrize("B,K,driver", [(1, 0, 0), (1, 100, 0), (3, 100, 0), (16, 0, 0), (1, 0, 3), (3, 100, 2)])
def test_captured_rollout_replays_like_eager(B, K, driver):
    sh = inputs.small_shape(dtype="bf16")
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(cached_weights(sh, 0, _scales(sh))))
    eng.set_driver(driver)
    r1 = inputs.make_requests(sh, list(range(500, 500 + B)))
    r2 = inputs.make_requests(sh, list(range(600, 600 + B)))
    hid, s, ver = device_requests(r1)
    out = torch.empty((B, 15), dtype=torch.int32, device="cuda")
    eager1 = eng.run(hid, s, ver, K=K).clone()
    eager2 = eng.run(*device_requests(r2), K=K).clone()
    torch.cuda.synchronize()
    assert eng.status() == 0

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        eng.run(hid, s, ver, K=K, out=out)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        eng.run(hid, s, ver, K=K, out=out)
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert eng.status() == 0
    np.testing.assert_array_equal(out.cpu().numpy(), eager1.cpu().numpy())
    # new inputs in the captured buffers: the replay follows them
    h2, s2, v2 = device_requests(r2)
    hid.copy_(h2)
    s.copy_(s2)
    ver.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert eng.status() == 0
    np.testing.assert_array_equal(out.cpu().numpy(), eager2.cpu().numpy())
    for _ in range(3):  # repeated replays of the same inputs
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert eng.status() == 0
        np.testing.assert_array_equal(out.cpu().numpy(), eager2.cpu().numpy())
    eng.close()
