"""Parity of the CUDA rollout (through the C ABI) with the CPU oracle.

Small cases compare every dump element by element; the full-size workloads
(Qwen3-8B-shaped and the larger target, B = 1/8/64, K0 and K2048) run in the
same launch configuration the benchmark times and compare base logits, GRU
states, projector pre-activations, the pool and every proposal.
"""
import json
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

from helpers import (TOL, cached_oracle_weights, cached_weights, check_against_oracle, check_free_run,
                     device_requests, device_weights, gpu_debug, make_engine)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FEEDBACK_SCALES = lambda sh: (("emb", 1.0), ("w_ih", sh.E ** -0.5), ("w_hh", sh.G ** -0.5),  # noqa: E731
                              ("fc1", 0.5 * sh.G ** -0.5), ("fc2", 0.2))


def _parity(shape, B, K, seeds=None, scales=(), scores=False, driver=None):
    seeds = seeds or list(range(1, B + 1))
    w = cached_weights(shape, 0, scales)
    ow = cached_oracle_weights(shape, 0, scales)
    r = inputs.make_requests(shape, seeds)
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    eng = make_engine(shape, max_B=B, max_K=K if 0 < K < shape.V else 0, dw=device_weights(w))
    if driver is not None:
        eng.set_driver(driver)
    dreq = device_requests(r)
    g = gpu_debug(eng, shape, dreq, B, K, o["tokens"], want_scores=scores)
    check_against_oracle(ow, o, g, shape, K)
    if scores:
        tol = TOL[shape.dtype]
        for b in range(B):
            want = np.stack([np.asarray(x) for x in oracle.rollout(
                ow, r["hidden"][b:b + 1], r["s"][b:b + 1], r["verified"][b:b + 1], K,
                keep_scores=True)["c"][0]])
            assert np.abs(g["scores"][b] - want).max() <= tol
    free = eng.run(*dreq, K=K)
    torch.cuda.synchronize()
    assert eng.status() == 0
    check_free_run(o, free.cpu().numpy(), TOL[shape.dtype])
    eng.close()
    return o, g


# ---- small cases: several tiles, ragged tails ------------------------------

def test_tiny_fp32_workload_full_dump():
    wl = inputs.WORKLOADS["tiny_fp32_b1_k0"]
    _parity(wl.shape, 1, 0, seeds=list(wl.request_seeds), scores=True)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("K", [0, 1, 100, 999, 1000, 5000])
def test_small_ragged_feedback(dtype, K):
    sh = inputs.small_shape(dtype=dtype)
    _parity(sh, 3, K, seeds=[11, 12, 13], scales=FEEDBACK_SCALES(sh), scores=True)


def test_hand_worked_golden_on_gpu():
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_rollout.json")
    g = json.load(open(path))
    sh = inputs.Shape(V=3, H=1, E=1, G=1, F=1, dtype="fp32")
    for case in g["cases"]:
        w = {k: np.asarray(v, dtype=np.float32) for k, v in g["weights_common"].items()}
        w["emb"] = np.asarray(case["emb"], dtype=np.float32)
        dw = device_weights(w)
        K = case["K"]
        eng = make_engine(sh, max_B=1, max_K=K, dw=dw)
        r = {"hidden": np.asarray(g["hidden"], np.float32).reshape(1, 16, 1),
             "s": np.asarray(g["s"], np.float32).reshape(1, 15, 1),
             "verified": np.asarray([case["verified"]], np.int32)}
        out = eng.run(*device_requests(r), K=K)
        torch.cuda.synchronize()
        assert out.cpu().numpy()[0].tolist() == case["expected"], case["name"]
        eng.close()


# ---- full-size workloads ---------------------------------------------------

@pytest.mark.parametrize("K", [0, 100])
@pytest.mark.parametrize("B", [16, 37])
def test_small_batches_on_the_tensor_core_gru(B, K):
    """B >= 12: GRU and projector layer 1 run as tcgen05 contractions."""
    sh = inputs.small_shape(dtype="bf16")
    _parity(sh, B, K, seeds=list(range(200, 200 + B)), scales=FEEDBACK_SCALES(sh))


@pytest.mark.parametrize("name", ["qwen3_8b_b1_k0", "qwen3_8b_b8_k0", "qwen3_8b_b64_k0",
                                  "qwen3_8b_b1_k2048", "qwen3_8b_b8_k2048", "qwen3_8b_b64_k2048",
                                  "large_b64_k0", "large_b64_k2048"])
def test_full_size_workloads(name):
    wl = inputs.WORKLOADS[name]
    _parity(wl.shape, wl.B, wl.K, seeds=list(wl.request_seeds))


# ---- edge cases --------------------------------------------------------------

def _small_engine(B=4, K=0, dtype="bf16", scales=None):
    sh = inputs.small_shape(dtype=dtype)
    sc = FEEDBACK_SCALES(sh) if scales is None else scales
    w = cached_weights(sh, 0, sc)
    eng = make_engine(sh, max_B=B, max_K=K, dw=device_weights(w))
    return sh, sc, w, eng


def test_empty_batch_is_a_no_op():
    sh, sc, w, eng = _small_engine()
    r = inputs.make_requests(sh, [1])
    hid, s, ver = device_requests(r)
    out = torch.full((1, 15), -5, dtype=torch.int32, device="cuda")
    from speculative_decoding_draft_lm_gb300 import rollout as R
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 0, 0, out) == 0
    torch.cuda.synchronize()
    assert (out == -5).all()
    assert eng.last_launch_count() == 0


def test_bad_verified_token_flags_request():
    sh, sc, w, eng = _small_engine()
    r = inputs.make_requests(sh, [1, 2, 3])
    r["verified"][1] = sh.V  # out of range
    hid, s, ver = device_requests(r)
    out = eng.run(hid, s, ver, K=0)
    from speculative_decoding_draft_lm_gb300 import rollout as R
    assert eng.status() == R.DOMINO_ERR_BAD_TOKEN
    got = out.cpu().numpy()
    assert (got[1] == -1).all()
    ow = cached_oracle_weights(sh, 0, sc)
    ok = {k: v[[0, 2]] for k, v in r.items()}
    o = oracle.rollout(ow, ok["hidden"], ok["s"], ok["verified"], 0)
    check_free_run(o, got[[0, 2]], TOL["bf16"])
    # the error word is cleared by reading it
    assert eng.status() == 0


def test_host_side_argument_errors():
    sh, sc, w, eng = _small_engine(B=2, K=10)
    from speculative_decoding_draft_lm_gb300 import rollout as R
    r = inputs.make_requests(sh, [1, 2])
    hid, s, ver = device_requests(r)
    out = torch.empty((2, 15), dtype=torch.int32, device="cuda")
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 3, 0, out) == R.DOMINO_ERR_INVALID_ARG  # B > max_B
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 2, -1, out) == R.DOMINO_ERR_INVALID_ARG
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 2, 11, out) == R.DOMINO_ERR_INVALID_ARG  # K > max_K
    assert R.domino_rollout_run(eng.ctx, None, s, ver, 2, 0, out) == R.DOMINO_ERR_INVALID_ARG
    # K >= V means the full vocabulary and needs no pool workspace
    assert R.domino_rollout_run(eng.ctx, hid, s, ver, 2, sh.V, out) == 0
    fresh = R.domino_rollout_init(R.domino_config(sh.V, sh.H, sh.E, sh.G, sh.F, 16, 2, 0, 1), 0)
    assert R.domino_rollout_run(fresh, hid, s, ver, 2, 0, out) == R.DOMINO_ERR_NOT_LOADED
    R.domino_rollout_destroy(fresh)
    with pytest.raises(R.DominoError):
        R.domino_rollout_init(R.domino_config(sh.V, sh.H, sh.E, sh.G, sh.F, 8, 2, 0, 1), 0)
    with pytest.raises(R.DominoError):  # bf16 needs multiples of 8
        R.domino_rollout_init(R.domino_config(sh.V, 20, sh.E, sh.G, sh.F, 16, 2, 0, 1), 0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("K", [0, 64])
def test_exact_ties_take_lowest_token_id(K):
    """Duplicate vocabulary rows tie exactly; the lower id must win."""
    sh = inputs.small_shape(dtype="bf16")
    sc = FEEDBACK_SCALES(sh)
    w = {k: v.copy() for k, v in cached_weights(sh, 0, sc).items()}
    r = inputs.make_requests(sh, [21, 22])
    ow0 = oracle.OracleWeights(w)
    o0 = oracle.rollout(ow0, r["hidden"], r["s"], r["verified"], K)
    # clone every chosen token's rows into a lower id so that each step ties
    dup = {}
    for t in np.unique(o0["tokens"]):
        lo = int(t) - 7 if t >= 7 else int(t) + 7
        dup[int(t)] = lo
    for t, lo in dup.items():
        for n in ("lm_head", "fc2", "emb"):
            w[n][lo] = w[n][t]
        w["b"][lo] = w["b"][t]
    ow = oracle.OracleWeights(w)
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    eng = make_engine(sh, max_B=2, max_K=K, dw=device_weights(w))
    dreq = device_requests(r)
    assert (o["margin"] == 0.0).any(), "the duplicated rows must create exact ties"
    # the oracle resolves every tie to the lower id; the GPU must agree
    g = gpu_debug(eng, sh, dreq, 2, K, o["tokens"])
    for b in range(2):
        for j in range(15):
            gt, ot = int(g["tokens"][b, j]), int(o["tokens"][b, j])
            if o["margin"][b, j] == 0.0:  # an exact duplicate tie
                assert gt == ot, (b, j, gt, ot)
    eng.close()


def test_batch_independence():
    sh = inputs.small_shape(dtype="bf16")
    sc = FEEDBACK_SCALES(sh)
    w = cached_weights(sh, 0, sc)
    r = inputs.make_requests(sh, list(range(30, 38)))
    dw = device_weights(w)
    for K in (0, 100):
        eng = make_engine(sh, max_B=8, max_K=K, dw=dw)
        whole = eng.run(*device_requests(r), K=K).cpu().numpy()
        for b in range(8):
            one = {k: v[b:b + 1] for k, v in r.items()}
            single = eng.run(*device_requests(one), K=K).cpu().numpy()
            assert (single[0] == whole[b]).all(), (K, b)
        eng.close()


@pytest.mark.parametrize("K", [1, 50, 300, 600])
def test_pool_cutoff_inside_a_large_tie_group(K):
    """Hundreds of vocabulary rows share one LM-head row, so the pool cutoff
    falls inside a group of exactly equal scores: the lowest ids must win."""
    sh = inputs.small_shape(V=2000, dtype="bf16")
    sc = FEEDBACK_SCALES(sh)
    w = {k: v.copy() for k, v in cached_weights(sh, 0, sc).items()}
    r = inputs.make_requests(sh, [5, 6])
    # make row 1234 score high, then clone it over 600 scattered ids
    w["lm_head"][1234] = inputs.to_bf16_bits((oracle.widen(w["lm_head"][1234]) * 6.0).astype(np.float32))
    ids = np.random.default_rng(3).choice(sh.V, size=600, replace=False)
    for v in ids:
        w["lm_head"][v] = w["lm_head"][1234]
    ow = oracle.OracleWeights(w)
    o = oracle.rollout(ow, r["hidden"], r["s"], r["verified"], K)
    score = o["L"][:, 1:16].max(axis=1)
    for b in range(2):  # the cutoff really sits inside the tie group
        kth = np.sort(score[b])[::-1][K - 1]
        assert (score[b] == kth).sum() > 1
    eng = make_engine(sh, max_B=2, max_K=K, dw=device_weights(w))
    g = gpu_debug(eng, sh, device_requests(r), 2, K, o["tokens"])
    for b in range(2):
        assert g["pool"][b].tolist() == o["pool"][b].tolist()
    check_against_oracle(ow, o, g, sh, K)
    eng.close()
