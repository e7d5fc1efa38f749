"""Seeded synthetic inputs for the Domino draft-block rollout.

This module only draws random numbers and stores them in the dtypes the
workloads name.  It holds none of the rollout's arithmetic: both the CPU
oracle (``oracle/``) and the CUDA path read what it returns, and neither
imports the other.

Recipe (the shapes and distributions of the Domino rollout microbenchmark on
the page "Add correctness-first Domino support to DFlash V2", section
"Performance summary"; no dataset or trained checkpoint is involved):

* weights, drawn in this order from one PCG64 stream seeded with
  ``SeedSequence(weight_seed, spawn_key=(0,))``:
  ``lm_head [V,H]``, ``emb [V,E]``, ``w_ih [3G,E]`` (gate rows r|z|n),
  ``w_hh [3G,G]``, ``fc1 [F,G]``, ``fc2 [V,F]``, ``b [V]``; each is
  float32 ``standard_normal`` times its scale (0.02 unless overridden);
* per request ``r`` (seeded with ``SeedSequence(request_seeds[r],
  spawn_key=(1,))``): ``hidden [16,H]`` and ``s [15,F]`` standard normal,
  then ``verified_token`` uniform in ``[0, V)``;
* for bf16 workloads every float tensor is rounded from float32 to bf16
  with round-to-nearest-even and handed out as the raw uint16 bit pattern.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

BLOCK = 16          # draft block size (positions per request)
N_PROPOSALS = 15    # proposals produced per block


@dataclass(frozen=True)
class Shape:
    """Model dimensions of one workload."""
    V: int
    H: int
    E: int
    G: int
    F: int
    dtype: str  # "fp32" or "bf16"


TINY = Shape(V=4096, H=256, E=128, G=128, F=256, dtype="fp32")
QWEN3_8B = Shape(V=151936, H=4096, E=1024, G=1024, F=1024, dtype="bf16")
LARGE_TARGET = Shape(V=151936, H=5120, E=1536, G=1536, F=1536, dtype="bf16")
QWEN3_8B_V80K = Shape(V=80000, H=4096, E=1024, G=1024, F=1024, dtype="bf16")


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    B: int
    K: int
    request_seeds: tuple
    weight_seed: int = 0
    # per-tensor standard deviation overrides, e.g. {"emb": 1.0}
    scales: dict = field(default_factory=dict)


def _seeds(B: int, first: int) -> tuple:
    return tuple(range(first, first + B))


# The five workloads of the benchmark.  "qwen3_8b_*" use Qwen3-8B-shaped
# dimensions; "large_*" the larger target (H=5120, E=G=F=1536).
WORKLOADS = {
    "tiny_fp32_b1_k0": Workload("tiny_fp32_b1_k0", TINY, 1, 0, (0,)),
    "qwen3_8b_b1_k0": Workload("qwen3_8b_b1_k0", QWEN3_8B, 1, 0, (1,)),
    "qwen3_8b_b8_k0": Workload("qwen3_8b_b8_k0", QWEN3_8B, 8, 0, _seeds(8, 1)),
    "qwen3_8b_b64_k0": Workload("qwen3_8b_b64_k0", QWEN3_8B, 64, 0, _seeds(64, 1)),
    "qwen3_8b_b1_k2048": Workload("qwen3_8b_b1_k2048", QWEN3_8B, 1, 2048, (1,)),
    "qwen3_8b_b8_k2048": Workload("qwen3_8b_b8_k2048", QWEN3_8B, 8, 2048, _seeds(8, 1)),
    "qwen3_8b_b64_k2048": Workload("qwen3_8b_b64_k2048", QWEN3_8B, 64, 2048, _seeds(64, 1)),
    "large_b64_k0": Workload("large_b64_k0", LARGE_TARGET, 64, 0, _seeds(64, 1)),
    "large_b64_k2048": Workload("large_b64_k2048", LARGE_TARGET, 64, 2048, _seeds(64, 1)),
    # profiling cases: the Qwen3-8B hidden sizes with the vocabulary cut to
    # 80,000 rows, so fc2 (164 MB) still exceeds L2 while the whole case
    # holds about 2 GB of device memory
    "qwen3_8b_v80k_b1_k0": Workload("qwen3_8b_v80k_b1_k0", QWEN3_8B_V80K, 1, 0, (1,)),
    "qwen3_8b_v80k_b1_k2048": Workload("qwen3_8b_v80k_b1_k2048", QWEN3_8B_V80K, 1, 2048, (1,)),
    "qwen3_8b_v80k_b64_k0": Workload("qwen3_8b_v80k_b64_k0", QWEN3_8B_V80K, 64, 0, _seeds(64, 1)),
}

WEIGHT_NAMES = ("lm_head", "emb", "w_ih", "w_hh", "fc1", "fc2", "b")


def weight_shapes(sh: Shape) -> dict:
    return {
        "lm_head": (sh.V, sh.H),
        "emb": (sh.V, sh.E),
        "w_ih": (3 * sh.G, sh.E),
        "w_hh": (3 * sh.G, sh.G),
        "fc1": (sh.F, sh.G),
        "fc2": (sh.V, sh.F),
        "b": (sh.V,),
    }


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _normal(gen: np.random.Generator, shape, scale: float, dtype: str,
            chunk_rows: int = 8192) -> np.ndarray:
    """Draw N(0, scale^2) float32 values row-chunk by row-chunk (bounded RAM)."""
    shape = tuple(shape)
    if dtype == "fp32":
        out = gen.standard_normal(shape, dtype=np.float32)
        out *= np.float32(scale)
        return out
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        x = gen.standard_normal((r1 - r0, flat.shape[1]), dtype=np.float32)
        x *= np.float32(scale)
        flat[r0:r1] = to_bf16_bits(x)
    return out


def make_weights(sh: Shape, seed: int = 0, scales: dict | None = None) -> dict:
    """All Domino weights for shape ``sh`` (float32 or bf16 bit patterns)."""
    scales = scales or {}
    gen = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(0,))))
    shapes = weight_shapes(sh)
    return {n: _normal(gen, shapes[n], scales.get(n, 0.02), sh.dtype) for n in WEIGHT_NAMES}


def make_fc1_hidden(sh: Shape, seed: int = 0, scale: float = 0.02) -> np.ndarray:
    """Backbone-hidden half of projector layer 1, [F, H] (its own stream, so
    the other weights do not change when it is drawn)."""
    gen = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(2,))))
    return _normal(gen, (sh.F, sh.H), scale, sh.dtype)


def make_requests(sh: Shape, request_seeds) -> dict:
    """Per-request draft hidden states, per-step ``s`` rows and verified tokens."""
    B = len(request_seeds)
    dt = np.float32 if sh.dtype == "fp32" else np.uint16
    hidden = np.empty((B, BLOCK, sh.H), dtype=dt)
    s = np.empty((B, N_PROPOSALS, sh.F), dtype=dt)
    tok = np.empty((B,), dtype=np.int32)
    for r, sd in enumerate(request_seeds):
        gen = np.random.Generator(np.random.PCG64(np.random.SeedSequence(int(sd), spawn_key=(1,))))
        x = gen.standard_normal((BLOCK, sh.H), dtype=np.float32)
        y = gen.standard_normal((N_PROPOSALS, sh.F), dtype=np.float32)
        if sh.dtype == "fp32":
            hidden[r], s[r] = x, y
        else:
            hidden[r], s[r] = to_bf16_bits(x), to_bf16_bits(y)
        tok[r] = gen.integers(0, sh.V)
    return {"hidden": hidden, "s": s, "verified": tok}


def make(workload: Workload | str, B: int | None = None):
    """(weights, requests) for a named workload; ``B`` truncates the batch."""
    wl = WORKLOADS[workload] if isinstance(workload, str) else workload
    seeds = wl.request_seeds if B is None else wl.request_seeds[:B]
    return make_weights(wl.shape, wl.weight_seed, wl.scales), make_requests(wl.shape, seeds)


def small_shape(V=1000, H=96, E=40, G=48, F=80, dtype="bf16") -> Shape:
    """A small shape that still spans several tiles with ragged tails."""
    return Shape(V=V, H=H, E=E, G=G, F=F, dtype=dtype)


def with_scales(wl: Workload, **scales) -> Workload:
    d = dict(wl.scales)
    d.update(scales)
    return replace(wl, scales=d)
