"""libfir_os.so on the host, no GPU compute: it loads, exports every entry point that
include/fir_os.h declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from frequency_domain_order_gb300 import build as fbuild
from frequency_domain_order_gb300 import fir_os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fir_os.h")


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fir_os.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fir_os_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fir_os_plan_create", "fir_os_execute", "fir_os_plan_destroy",
                     "fir_os_execute_host", "fir_os_plan_info", "fir_os_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in fir_os.SIGNATURES, f"binding lacks {name}"


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert L.fir_os_status_string(code)
    assert L.fir_os_status_string(-99) == b"unknown status"


def _create(L, M, N, data_kind=fir_os.COMPLEX, coef_kind=fir_os.COEF_TIME, coef_complex=0,
            coef=0x1000):
    h = ctypes.c_void_p()
    rc = L.fir_os_plan_create(ctypes.byref(h), M, N, data_kind, coef_kind, coef_complex, coef, None)
    return rc, h


@pytest.mark.parametrize("M,N", [(10, 100), (10, 32), (10, 1 << 17), (0, 256), (300, 256)])
def test_bad_sizes_rejected_on_host(L, M, N):
    rc, h = _create(L, M, N)
    assert rc == fir_os.E_UNSUPPORTED and not h.value
    assert L.fir_os_last_error()


def test_bad_kinds_and_pointers_rejected_on_host(L):
    assert _create(L, 8, 64, data_kind=7)[0] == fir_os.E_INVAL
    assert _create(L, 8, 64, coef_kind=5)[0] == fir_os.E_INVAL
    assert _create(L, 8, 64, coef=0)[0] == fir_os.E_INVAL
    # real data with a complex h
    assert _create(L, 8, 64, data_kind=fir_os.REAL, coef_complex=1)[0] == fir_os.E_UNSUPPORTED
    # a given H must be 16-byte aligned
    assert _create(L, 8, 64, coef_kind=fir_os.COEF_FREQ, coef=0x1008)[0] == fir_os.E_ALIGN
    assert L.fir_os_plan_create(None, 8, 64, 1, 0, 0, 0x1000, None) == fir_os.E_INVAL


def test_null_plan_rejected(L):
    assert L.fir_os_execute(None, 0x1000, 10, 0x2000, 0x3000, None) == fir_os.E_INVAL
    assert L.fir_os_execute_host(None, 0x1000, 10, 0x2000, 0x3000, None) == fir_os.E_INVAL
    assert L.fir_os_plan_info(None, None, None, None) == fir_os.E_INVAL
    assert L.fir_os_plan_kernel(None, None, None, None, None) == fir_os.E_INVAL
    assert L.fir_os_device_status(None, None) == fir_os.E_INVAL
    assert L.fir_os_plan_destroy(None) == fir_os.OK


def test_no_device_is_an_error_not_a_crash(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _create(L, 64, 256)
    assert rc == fir_os.E_CUDA and not h.value


def test_test_hooks_reject_bad_arguments(L):
    assert L.fir_os_plan_set_wait_limit(None, 0) == fir_os.E_INVAL
    assert L.fir_os_plan_set_dft_engine(None, fir_os.DFT_TENSOR) == fir_os.E_INVAL
    assert L.fir_os_debug_fail_alloc(-1) == fir_os.E_INVAL
    assert L.fir_os_debug_fail_alloc(0) == fir_os.OK


def test_injected_allocation_failure_is_nomem_and_leaks_nothing(L):
    """The first allocation of fir_os_plan_create is its host-side plan object, made before any
    device call: an injected failure there returns FIR_OS_E_NOMEM, no plan, and leaves the
    library's live-allocation count unchanged (GPU tests cover the device buffers)."""
    before = L.fir_os_debug_live_allocs()
    assert L.fir_os_debug_fail_alloc(1) == fir_os.OK
    rc, h = _create(L, 64, 256)
    assert rc == fir_os.E_NOMEM and not h.value
    assert b"plan allocation" in L.fir_os_last_error()
    assert L.fir_os_debug_live_allocs() == before
    # the hook fired once and is spent: the next call gets past the plan object
    rc, h = _create(L, 8, 64, data_kind=7)
    assert rc == fir_os.E_INVAL
    assert L.fir_os_debug_fail_alloc(0) == fir_os.OK
