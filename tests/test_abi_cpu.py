"""The C-ABI library on a machine without a GPU: it loads, exports exactly the
entry points include/qa.h declares, and rejects invalid arguments with status
codes before touching the device (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qa.h")


@pytest.fixture(scope="module")
def qa():
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    return set(re.findall(r"^\s*(?:qa_status|int|const char \*)\s*(qa_\w+)\s*\(", text, re.M))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("qa_cache_alloc", "qa_cache_free", "qa_cache_reset", "qa_prefill",
                     "qa_decode_step"):
        assert required in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(qa):
    names = declared_functions()
    for n in names:
        assert hasattr(qa.lib, n), n
    assert names == set(qa.SIGNATURES), "binding and header disagree"


def test_library_exports_nothing_else(qa):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", qa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert exported == declared_functions()


def test_abi_version_and_status_strings(qa):
    ver = int(re.search(r"#define QA_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert qa.qa_abi_version() == ver
    for code in range(9):
        assert qa.qa_status_str(code) and qa.qa_status_str(code) != "unknown status"
    assert qa.qa_status_str(99) == "unknown status"


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2), (dict(n_q_heads=6, n_kv_heads=4), 2), (dict(n_q_heads=32, n_kv_heads=2), 2),
    (dict(capacity=0), 1), (dict(max_batch=0), 1), (dict(num_layers=0), 1),
    (dict(rope_theta=0.0), 1), (dict(rms_eps=-1.0), 1)])
def test_alloc_rejects_bad_geometry(qa, kw, status):
    args = dict(num_layers=1, max_batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, capacity=64,
                rope_theta=1e6, rms_eps=1e-6)
    args.update(kw)
    with pytest.raises(qa.QaError) as e:
        qa.qa_cache_alloc(**args)
    assert e.value.status == status


def test_alloc_null_arguments(qa):
    assert qa.lib.qa_cache_alloc(None, None) == 1


def test_null_cache_is_rejected_everywhere(qa):
    lens = (ctypes.c_int32 * 1)(4)
    assert qa.lib.qa_cache_free(None) == 0
    assert qa.lib.qa_cache_reset(None, None) == 1
    assert qa.lib.qa_prefill(None, 0, 1, lens, 16, 16, 16, 16, 16, 16, None) == 1
    assert qa.lib.qa_prefill_transform(None, 0, 1, lens, 16, 16, 16, 16, 16, 16, None) == 1
    assert qa.lib.qa_decode_step(None, 0, 1, 16, 16, 16, 16, 16, 16, None) == 1
    assert qa.lib.qa_cache_set_lengths(None, 0, lens, None) == 1
    assert qa.lib.qa_cache_lengths(None, 0, lens) == 1
    assert qa.lib.qa_get_device_error(None, None) == 1
    assert qa.lib.qa_stats(None, None) == 1
    assert qa.lib.qa_memory_info(None, None, None) == 1
    assert qa.lib.qa_decode_splits(None, 0, 1) == 0
    assert qa.lib.qa_decode_step_device_lengths(None, 0, 1, 16, 16, 16, 16, 16, 16, None) == 1
    assert qa.lib.qa_cache_sync_lengths(None, 0, None) == 1
    assert qa.lib.qa_cache_set_window(None, 0, 16) == 1
    assert qa.lib.qa_cache_set_decode_overlap(None, 2) == 1
    assert qa.lib.qa_cache_view(None, 0, None, None, None, None) == 1
    pos = (ctypes.c_int32 * 1)(0)
    assert qa.lib.qa_decode_step_noalloc(None, 1, pos, 16, 16, 16, 16, 16, 16, 16, 16, None) == 1


def test_valid_alloc_without_a_device_reports_cuda_error(qa):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(qa.QaError) as e:
        qa.qa_cache_alloc(1, 1, 2, 1, 64, 72)
    assert e.value.status == 6


def test_new_hooks_validate_before_touching_the_device(qa):
    lens = (ctypes.c_int32 * 1)(4)
    assert qa.lib.qa_prefill_attend(None, 0, 1, lens, 16, 16, None) == 1
    # the failure-detection hook: only the two tiled kernels, a bounded limit
    for kernel, us in ((0, 100), (3, 100), (7, 100), (1, 0), (2, 2000001)):
        assert qa.lib.qa_debug_arm_wait_timeout(kernel, us) == 1
    assert qa.lib.qa_debug_arm_wait_timeout(2, 1000) == 0
    assert qa.lib.qa_debug_arm_wait_timeout(-1, 0) == 0   # disarm


def test_noalloc_error_read_without_a_device_reports_cuda_error(qa):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    w = ctypes.c_uint32(123)
    assert qa.lib.qa_noalloc_get_device_error(ctypes.byref(w), None) == 6
