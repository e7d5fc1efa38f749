"""CPU checks of the C ABI: the library builds, loads and exports every
symbol its header declares, and host-side argument checks answer without a
GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "domino_rollout.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DOMINO_API\s+[\w\s\*]+?\b(domino_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_lm_gb300 import build, rollout
    if not os.path.exists(rollout.LIB_PATH):
        build.build()
    return rollout.load_library()


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("domino_rollout_init", "domino_rollout_load_weights", "domino_rollout_run",
                 "domino_rollout_debug_run", "domino_rollout_status", "domino_rollout_destroy",
                 "domino_rollout_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from speculative_decoding_draft_lm_gb300 import rollout
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(rollout.EXPORTED) == _declared()


def test_strerror_and_null_handles(lib):
    from speculative_decoding_draft_lm_gb300 import rollout as R
    assert R.strerror(R.DOMINO_OK) == "ok"
    assert "token" in R.strerror(R.DOMINO_ERR_BAD_TOKEN)
    assert lib.domino_rollout_run(None, None, None, None, 1, 0, None, None) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_status(None, None) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_set_driver(None, 0) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_set_proposals(None, 7) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_set_vocab_partitions(None, 2) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_load_backbone_proj(None, None) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_enable_timing(None, 1) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_candidate_pool_static(None, 1, 10, 2, None, None) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_debug_drop_barrier_arrival(None, 1) == R.DOMINO_ERR_INVALID_ARG
    lib.domino_rollout_destroy(None)
    assert lib.domino_rollout_last_launch_count(None) == 0


def test_config_validation_precedes_device_access(lib):
    from speculative_decoding_draft_lm_gb300 import rollout as R
    ctx = ctypes.c_void_p()
    bad_block = R.domino_config(100, 64, 8, 8, 8, 8, 1, 0, 1)
    assert lib.domino_rollout_init(ctypes.byref(ctx), ctypes.byref(bad_block), 0) == R.DOMINO_ERR_UNSUPPORTED
    bad_dtype = R.domino_config(100, 64, 8, 8, 8, 16, 1, 0, 7)
    assert lib.domino_rollout_init(ctypes.byref(ctx), ctypes.byref(bad_dtype), 0) == R.DOMINO_ERR_UNSUPPORTED
    odd_bf16 = R.domino_config(100, 60, 8, 8, 8, 16, 1, 0, 1)
    assert lib.domino_rollout_init(ctypes.byref(ctx), ctypes.byref(odd_bf16), 0) == R.DOMINO_ERR_UNSUPPORTED
    neg = R.domino_config(100, 64, 8, 8, 8, 16, 0, 0, 1)
    assert lib.domino_rollout_init(ctypes.byref(ctx), ctypes.byref(neg), 0) == R.DOMINO_ERR_INVALID_ARG
    assert lib.domino_rollout_init(None, ctypes.byref(neg), 0) == R.DOMINO_ERR_INVALID_ARG
    assert not ctx.value
