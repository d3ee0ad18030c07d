"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every entry
point that include/qgemv.h declares, and its pure host functions and argument checks
behave as documented."""
import ctypes
import os
import re
import subprocess

import pytest

from quantized_weight_dequant_gb300 import qgemv, synth
from quantized_weight_dequant_gb300.build import LIB, build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_library()


def _declared():
    txt = open(os.path.join(ROOT, "include", "qgemv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemv_[a-z_]+)\s*\(", txt)))


def test_library_exports_every_declared_entry_point():
    declared = _declared()
    assert "qgemv_run" in declared and "qgemv_create" in declared
    out = subprocess.check_output(["nm", "-D", "--defined-only", LIB]).decode()
    exported = set(re.findall(r"\bT (qgemv_\w+)", out))
    missing = [d for d in declared if d not in exported]
    assert not missing, missing
    L = qgemv.lib()
    for d in declared:
        assert hasattr(L, d)
    assert set(qgemv.EXPORTS) == set(declared)


def test_build_marker_matches_the_sources():
    from quantized_weight_dequant_gb300.build import source_digest
    assert qgemv.build_marker() == "qgemv-build:" + source_digest()


@pytest.mark.parametrize("fmt", list(synth.FORMAT_NAMES))
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (4096, 14336), (3, 4096)])
def test_packed_bytes_matches_the_layouts(fmt, N, K):
    assert qgemv.packed_bytes(fmt, N, K) == synth.packed_bytes(fmt, N, K)


def test_packed_bytes_rejects_bad_shapes_and_formats():
    assert qgemv.packed_bytes(synth.Q4_K, 4, 100) == 0
    assert qgemv.packed_bytes(synth.Q8_0, 4, 48) == 0
    assert qgemv.packed_bytes(synth.Q8_0, 4, 64) == 4 * 2 * 34
    assert qgemv.packed_bytes(synth.NVFP4, 4, 48) == 4 * 24 + 4 * 3
    assert qgemv.packed_bytes(9, 4, 256) == 0
    assert qgemv.packed_bytes(synth.Q4_K, 0, 256) == 0


def test_group_sizes_and_status_strings():
    import oracle
    for f in synth.FORMAT_NAMES:
        assert qgemv.group_size(f) == oracle.group_size(f)
    assert qgemv.group_size(17) == 0
    for s in range(10):
        assert qgemv.status_string(s) and qgemv.status_string(s) != "unknown status"
    assert qgemv.status_string(99) == "unknown status"


def test_null_handle_and_pointer_arguments_are_rejected_without_a_launch():
    L = qgemv.lib()
    assert L.qgemv_run(None, 0, 16, 16, 4, 256, 16, None) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_unpack(None, 0, 16, 4, 256, 16, 16, None, None) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_check_error(None, None) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_set_option(None, 0, 0) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_create(None, 0) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_destroy(None) == qgemv.OK
    # the layer, batch and many-row entry points check the handle first as well
    assert L.qgemv_run_ex(None, 0, 16, 16, 4, 256, 1.0, 0.0, 16, 0, None) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_run_group(None, 16, 256, 1, None, None) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_run_batch(None, 0, 16, 2, 16, 4, 256, 16, None) == qgemv.ERR_INVALID_ARG
    assert L.qgemv_run_gemm(None, 1, 16, 32, 16, 4, 256, 16, None) == qgemv.ERR_INVALID_ARG


def test_create_reports_no_device_when_there_is_none():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert qgemv.lib().qgemv_create(ctypes.byref(h), 0) == qgemv.ERR_NO_DEVICE
    assert not h.value
