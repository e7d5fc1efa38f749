"""CPU oracle of the Domino draft-block rollout (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
import this package; the CUDA library never does.
"""
from .domino_oracle import (  # noqa: F401
    BLOCK, N_PROPOSALS, N_CORRECTED, ROW_OFFSET, OracleWeights, argmax_lowest, backbone_s,
    candidate_pool, candidate_pool_compact, gru_cell, lm_head, rollout, run, silu, sigmoid, top2_margin,
    widen,
)
