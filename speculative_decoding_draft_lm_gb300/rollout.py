"""Python binding of the C ABI in ``include/domino_rollout.h`` (ctypes).

Argument marshalling only: every step of the rollout runs in the CUDA
library.  Device memory comes from torch tensors; the calls take their
``data_ptr()`` and the current torch stream.  There is no CPU fallback: if
the library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdomino_rollout.so")

DOMINO_OK = 0
DOMINO_ERR_INVALID_ARG = -1
DOMINO_ERR_UNSUPPORTED = -2
DOMINO_ERR_NOT_LOADED = -3
DOMINO_ERR_CUDA = -4
DOMINO_ERR_OOM = -5
DOMINO_ERR_TIMEOUT = -6
DOMINO_ERR_BAD_TOKEN = -7
DOMINO_ERR_SCRATCH_LIMIT = -8
DOMINO_STATIC_SCRATCH_FLOATS = 2 * 1024 * 1024

DOMINO_DTYPE_FP32 = 0
DOMINO_DTYPE_BF16 = 1
DOMINO_BLOCK = 16

DOMINO_DRIVER_AUTO = 0
DOMINO_DRIVER_KERNELS = 1
DOMINO_DRIVER_PERSISTENT = 2
DOMINO_DRIVER_PERSISTENT_GRID = 3

# every symbol the header declares
EXPORTED = (
    "domino_rollout_init", "domino_rollout_load_weights", "domino_rollout_run",
    "domino_rollout_debug_run", "domino_rollout_set_driver", "domino_rollout_status",
    "domino_rollout_last_launch_count", "domino_rollout_destroy", "domino_rollout_strerror",
    "domino_rollout_enable_timing", "domino_rollout_read_timing", "domino_candidate_pool_static",
    "domino_rollout_set_proposals", "domino_rollout_load_backbone_proj", "domino_rollout_set_vocab_partitions",
    "domino_rollout_debug_drop_barrier_arrival",
)

PHASES = ("lmhead", "argmax", "pool", "gru", "fc1", "correct", "steps", "other")


class domino_config(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int), ("G", ctypes.c_int),
                ("F", ctypes.c_int), ("block", ctypes.c_int), ("max_B", ctypes.c_int),
                ("max_K", ctypes.c_int), ("dtype", ctypes.c_int)]


class domino_debug_bufs(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("pool", ctypes.c_void_p), ("h", ctypes.c_void_p),
                ("z", ctypes.c_void_p), ("top1", ctypes.c_void_p), ("scores", ctypes.c_void_p),
                ("trace", ctypes.c_void_p)]


DOMINO_TRACE_SLOTS = 96


class DominoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run __graft_entry__.build() or python -m speculative_decoding_draft_lm_gb300.build)")
    lib = ctypes.CDLL(path)
    vp, ip, i = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    lib.domino_rollout_init.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(domino_config), i]
    lib.domino_rollout_load_weights.argtypes = [vp] * 8
    lib.domino_rollout_run.argtypes = [vp, vp, vp, vp, i, i, vp, vp]
    lib.domino_rollout_debug_run.argtypes = [vp, vp, vp, vp, i, i, vp, ctypes.POINTER(domino_debug_bufs), vp, vp]
    lib.domino_rollout_set_driver.argtypes = [vp, i]
    lib.domino_rollout_status.argtypes = [vp, vp]
    lib.domino_rollout_last_launch_count.argtypes = [vp]
    lib.domino_rollout_destroy.argtypes = [vp]
    lib.domino_rollout_destroy.restype = None
    lib.domino_rollout_enable_timing.argtypes = [vp, i]
    lib.domino_rollout_read_timing.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
    lib.domino_candidate_pool_static.argtypes = [vp, i, i, i, vp, vp]
    lib.domino_rollout_set_proposals.argtypes = [vp, i]
    lib.domino_rollout_load_backbone_proj.argtypes = [vp, vp]
    lib.domino_rollout_set_vocab_partitions.argtypes = [vp, i]
    lib.domino_rollout_debug_drop_barrier_arrival.argtypes = [vp, i]
    lib.domino_rollout_strerror.argtypes = [i]
    lib.domino_rollout_strerror.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name not in ("domino_rollout_destroy", "domino_rollout_strerror"):
            getattr(lib, name).restype = ip
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load_library().domino_rollout_strerror(status).decode()


def _check(status: int, where: str) -> int:
    if status != DOMINO_OK:
        raise DominoError(status, where)
    return status


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ---- the C entry points, same names ---------------------------------------

def domino_rollout_init(cfg: domino_config, device: int = 0) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    _check(load_library().domino_rollout_init(ctypes.byref(ctx), ctypes.byref(cfg), device), "domino_rollout_init")
    return ctx


def domino_rollout_load_weights(ctx, lm_head, emb, w_ih, w_hh, fc1, fc2, bias) -> int:
    return _check(load_library().domino_rollout_load_weights(
        ctx, _ptr(lm_head), _ptr(emb), _ptr(w_ih), _ptr(w_hh), _ptr(fc1), _ptr(fc2), _ptr(bias)),
        "domino_rollout_load_weights")


def domino_rollout_run(ctx, hidden, s, verified_tok, B: int, K: int, out_tokens, stream=None) -> int:
    return load_library().domino_rollout_run(ctx, _ptr(hidden), _ptr(s), _ptr(verified_tok), B, K,
                                             _ptr(out_tokens), _stream(stream))


def domino_rollout_debug_run(ctx, hidden, s, verified_tok, B: int, K: int, forced_tokens, dbg: dict,
                             out_tokens, stream=None) -> int:
    bufs = domino_debug_bufs(*[_ptr(dbg.get(n)) for n in ("logits", "pool", "h", "z", "top1", "scores", "trace")])
    return load_library().domino_rollout_debug_run(ctx, _ptr(hidden), _ptr(s), _ptr(verified_tok), B, K,
                                                   _ptr(forced_tokens), ctypes.byref(bufs), _ptr(out_tokens),
                                                   _stream(stream))


def domino_rollout_set_driver(ctx, driver: int) -> int:
    return _check(load_library().domino_rollout_set_driver(ctx, driver), "domino_rollout_set_driver")


def domino_rollout_load_backbone_proj(ctx, w_hid) -> int:
    return _check(load_library().domino_rollout_load_backbone_proj(ctx, _ptr(w_hid)),
                  "domino_rollout_load_backbone_proj")


def domino_rollout_set_vocab_partitions(ctx, P: int) -> int:
    return _check(load_library().domino_rollout_set_vocab_partitions(ctx, P), "domino_rollout_set_vocab_partitions")


def domino_rollout_set_proposals(ctx, n: int) -> int:
    return _check(load_library().domino_rollout_set_proposals(ctx, n), "domino_rollout_set_proposals")


def domino_rollout_debug_drop_barrier_arrival(ctx, n: int) -> int:
    """Test hook of the timeout path (see the header): returns the status."""
    return load_library().domino_rollout_debug_drop_barrier_arrival(ctx, n)


def domino_rollout_status(ctx, stream=None) -> int:
    return load_library().domino_rollout_status(ctx, _stream(stream))


def domino_rollout_last_launch_count(ctx) -> int:
    return load_library().domino_rollout_last_launch_count(ctx)


def domino_rollout_enable_timing(ctx, enable: bool) -> int:
    return _check(load_library().domino_rollout_enable_timing(ctx, int(bool(enable))),
                  "domino_rollout_enable_timing")


def domino_rollout_read_timing(ctx) -> dict:
    """{phase: (ms, launches)} accumulated since the last read."""
    ms = (ctypes.c_float * len(PHASES))()
    n = (ctypes.c_int * len(PHASES))()
    _check(load_library().domino_rollout_read_timing(ctx, ms, n), "domino_rollout_read_timing")
    return {p: (float(ms[i]), int(n[i])) for i, p in enumerate(PHASES)}


def domino_candidate_pool_static(base_logits, B: int, V: int, K: int, pool_out, stream=None) -> int:
    """Allocation-free pool selection (see the header): returns the status."""
    return load_library().domino_candidate_pool_static(_ptr(base_logits), B, V, K, _ptr(pool_out), _stream(stream))


def domino_rollout_destroy(ctx) -> None:
    load_library().domino_rollout_destroy(ctx)


def domino_rollout_strerror(status: int) -> str:
    return strerror(status)


# ---- convenience wrapper over torch tensors --------------------------------

class DominoRollout:
    """Owns one library context; weights are torch CUDA tensors (borrowed).

    ``weights`` maps lm_head, emb, w_ih, w_hh, fc1, fc2, b to device tensors
    (float32, or bfloat16 / 2-byte bit patterns for the bf16 dtype).
    """

    def __init__(self, V, H, E, G, F, max_B, max_K=0, dtype="bf16", device=0):
        self.dims = dict(V=V, H=H, E=E, G=G, F=F)
        self.dtype = dtype
        self.max_B, self.max_K = max_B, max_K
        self.device = device
        cfg = domino_config(V, H, E, G, F, DOMINO_BLOCK, max_B, max_K,
                            DOMINO_DTYPE_BF16 if dtype == "bf16" else DOMINO_DTYPE_FP32)
        self.ctx = domino_rollout_init(cfg, device)
        self._weights = None

    def _check_tensor(self, t, shape, name):
        esize = 2 if self.dtype == "bf16" else 4
        if tuple(t.shape) != tuple(shape) or t.element_size() != esize or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: want contiguous CUDA {shape} with {esize}-byte elements, "
                             f"got {tuple(t.shape)} {t.dtype} on {t.device}")

    def load_weights(self, weights: dict):
        d = self.dims
        shapes = {"lm_head": (d["V"], d["H"]), "emb": (d["V"], d["E"]), "w_ih": (3 * d["G"], d["E"]),
                  "w_hh": (3 * d["G"], d["G"]), "fc1": (d["F"], d["G"]), "fc2": (d["V"], d["F"]),
                  "b": (d["V"],)}
        for n, shp in shapes.items():
            self._check_tensor(weights[n], shp, n)
        self._weights = dict(weights)  # keep them alive while borrowed
        domino_rollout_load_weights(self.ctx, weights["lm_head"], weights["emb"], weights["w_ih"],
                                    weights["w_hh"], weights["fc1"], weights["fc2"], weights["b"])

    def load_backbone_proj(self, w_hid):
        """Register W_hid [F, H]; then run(hidden, None, verified) derives s."""
        if w_hid is not None:
            self._check_tensor(w_hid, (self.dims["F"], self.dims["H"]), "w_hid")
        self._w_hid = w_hid  # keep it alive while borrowed
        domino_rollout_load_backbone_proj(self.ctx, w_hid)

    def set_driver(self, driver: int):
        domino_rollout_set_driver(self.ctx, driver)

    def set_proposals(self, n: int):
        domino_rollout_set_proposals(self.ctx, n)

    def set_vocab_partitions(self, P: int):
        domino_rollout_set_vocab_partitions(self.ctx, P)

    def run(self, hidden, s, verified, K=0, out=None, stream=None):
        import torch
        B = hidden.shape[0]
        if out is None:
            out = torch.empty((B, 15), dtype=torch.int32, device=hidden.device)
        _check(domino_rollout_run(self.ctx, hidden, s, verified, B, K, out, stream), "domino_rollout_run")
        return out

    def debug_run(self, hidden, s, verified, K=0, forced=None, dbg=None, out=None, stream=None):
        import torch
        B = hidden.shape[0]
        if out is None:
            out = torch.empty((B, 15), dtype=torch.int32, device=hidden.device)
        _check(domino_rollout_debug_run(self.ctx, hidden, s, verified, B, K, forced, dbg or {}, out, stream),
               "domino_rollout_debug_run")
        return out

    def status(self, stream=None) -> int:
        return domino_rollout_status(self.ctx, stream)

    def enable_timing(self, enable=True):
        domino_rollout_enable_timing(self.ctx, enable)

    def read_timing(self) -> dict:
        return domino_rollout_read_timing(self.ctx)

    def last_launch_count(self) -> int:
        return domino_rollout_last_launch_count(self.ctx)

    def close(self):
        if getattr(self, "ctx", None) is not None and self.ctx.value:
            domino_rollout_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def to_device(arr, device="cuda"):
    """numpy float32 array or uint16 bf16 bit pattern -> torch CUDA tensor."""
    import numpy as np
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)
