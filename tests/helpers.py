"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle
on the same seeded inputs and compare them under the tolerance rule.

Tolerance rule (floating point): base logits, GRU states, projector
pre-activations and corrected scores agree within TOL[dtype] (max abs).
Tokens: wherever the oracle's top-2 margin exceeds the tolerance the CUDA
token must equal the oracle's; where it does not, the CUDA token must score
within the tolerance of the oracle's best (several answers are correct).
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
from speculative_decoding_draft_lm_gb300 import inputs

TOL = {"fp32": 1e-4, "bf16": 2e-2}


@functools.lru_cache(maxsize=2)
def cached_weights(shape: inputs.Shape, seed: int = 0, scales: tuple = ()):
    return inputs.make_weights(shape, seed, dict(scales))


@functools.lru_cache(maxsize=2)
def cached_oracle_weights(shape: inputs.Shape, seed: int = 0, scales: tuple = ()):
    return oracle.OracleWeights(cached_weights(shape, seed, scales))


def device_weights(w: dict):
    from speculative_decoding_draft_lm_gb300.rollout import to_device
    return {k: to_device(v) for k, v in w.items()}


def device_requests(r: dict):
    import torch
    from speculative_decoding_draft_lm_gb300.rollout import to_device
    return (to_device(r["hidden"]), to_device(r["s"]),
            torch.from_numpy(np.ascontiguousarray(r["verified"], dtype=np.int32)).cuda())


def make_engine(shape: inputs.Shape, max_B: int, max_K: int, dw: dict):
    from speculative_decoding_draft_lm_gb300.rollout import DominoRollout
    eng = DominoRollout(shape.V, shape.H, shape.E, shape.G, shape.F, max_B=max_B, max_K=max_K,
                        dtype=shape.dtype)
    eng.load_weights(dw)
    return eng


def gpu_debug(eng, shape, dreq, B, K, forced_np, want_scores=False):
    """Teacher-forced debug run; returns numpy dumps."""
    import torch
    hid, s, ver = dreq
    Kc = shape.V if (K == 0 or K >= shape.V) else K
    f32 = dict(dtype=torch.float32, device="cuda")
    dbg = {
        "logits": torch.empty((B, 16, shape.V), **f32),
        "h": torch.empty((B, 15, shape.G), **f32),
        "z": torch.empty((B, 14, shape.F), **f32),
        "top1": torch.empty((B, 15), **f32),
    }
    if 0 < K < shape.V:
        dbg["pool"] = torch.empty((B, K), dtype=torch.int32, device="cuda")
    if want_scores:
        dbg["scores"] = torch.empty((B, 14, Kc), **f32)
    forced = None
    if forced_np is not None:
        forced = torch.from_numpy(np.ascontiguousarray(forced_np, dtype=np.int32)).cuda()
    out = eng.debug_run(hid, s, ver, K=K, forced=forced, dbg=dbg)
    torch.cuda.synchronize()
    st = eng.status()
    res = {k: v.cpu().numpy() for k, v in dbg.items()}
    res["tokens"] = out.cpu().numpy()
    res["status"] = st
    return res


def oracle_scores_at(ow: oracle.OracleWeights, o: dict, b: int, k: int, ids) -> np.ndarray:
    """Oracle corrected score of step k (1..14) of request b at token ids."""
    ids = np.asarray(ids, dtype=np.int64)
    a = oracle.silu(o["z"][b, k - 1])
    return ow.fc2[ids] @ a + ow.b[ids] + o["L"][b, oracle.ROW_OFFSET + k, ids]


def check_against_oracle(ow, o, g, shape, K, tol=None, check_scores=True):
    """Compare a teacher-forced CUDA debug run ``g`` with the oracle run ``o``."""
    tol = TOL[shape.dtype] if tol is None else tol
    B = o["tokens"].shape[0]
    assert g["status"] == 0, g["status"]
    # base logits
    errL = np.abs(g["logits"] - o["L"]).max()
    assert errL <= tol, f"base logits max abs err {errL}"
    # GRU states and projector pre-activations
    errh = np.abs(g["h"] - o["h"]).max()
    assert errh <= tol, f"h max abs err {errh}"
    errz = np.abs(g["z"] - o["z"]).max()
    assert errz <= tol, f"z max abs err {errz}"
    # pool: equal except ids whose score ties the cutoff within tol
    full = K == 0 or K >= shape.V
    if not full:
        for b in range(B):
            gp = g["pool"][b]
            assert (np.diff(gp) > 0).all(), "pool not ascending"
            score = o["L"][b, 1:16].max(axis=0)
            kth = np.sort(score)[::-1][K - 1]
            diff = set(gp.tolist()) ^ set(o["pool"][b].tolist())
            for v in diff:
                assert abs(score[v] - kth) <= tol, f"pool differs at id {v}: score {score[v]} vs cutoff {kth}"
    # tokens, teacher-forced
    for b in range(B):
        for j in range(15):
            gt, ot = int(g["tokens"][b, j]), int(o["tokens"][b, j])
            if j == 0:
                row = o["L"][b, oracle.ROW_OFFSET]
                gval, oval = row[gt], row[ot]
            else:
                if not full:
                    assert gt in set(g["pool"][b].tolist())
                gval, oval = oracle_scores_at(ow, o, b, j, [gt, ot])
            if o["margin"][b, j] > tol:
                assert gt == ot, f"request {b} proposal {j}: gpu {gt} oracle {ot} margin {o['margin'][b, j]}"
            else:
                assert gval >= oval - tol, f"request {b} proposal {j}: near-tie token {gt} scores {gval} < {oval}-tol"
            if check_scores:
                assert abs(g["top1"][b, j] - gval) <= tol, f"request {b} proposal {j}: top1 {g['top1'][b, j]} vs {gval}"


def check_free_run(o, gpu_tokens, tol):
    """Free-running chains agree up to each request's first near-tie step."""
    B = o["tokens"].shape[0]
    for b in range(B):
        for j in range(15):
            if o["margin"][b, j] <= tol:
                break
            assert gpu_tokens[b, j] == o["tokens"][b, j], f"free run: request {b} proposal {j}"
