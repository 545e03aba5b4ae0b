"""The allocation-free frequency-response entry point, through the C ABI, on a GPU.

fir_os_frequency_response_noalloc exists for callers that may not allocate device memory when
they build a filter's response (their device memory belongs to their own pool, they run on a
real-time thread, or the device is at its memory limit).  It computes the same float64 step-1
transform that fir_os_plan_create runs with allocated buffers, but in a fixed array inside the
library.  This file checks, on consecutive calls, that its response matches numpy's float64 FFT
of the taps, and that filtering with it matches both the float64 oracle (direct convolution)
and filtering with the plan that computes the response itself, under the same parity bar as
the other GPU tests.  It sits last in collection order so that a stop-at-first-failure run has
already run everything else.
"""
import ctypes

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fo():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build, fir_os
    build.build()
    return fir_os


def _noalloc_response(fo, h, N):
    import torch
    hd = torch.from_numpy(h).cuda()
    Hd = torch.empty(N, dtype=torch.complex64, device="cuda")
    rc = fo.lib().fir_os_frequency_response_noalloc(
        hd.data_ptr(), h.size, N, 1 if np.iscomplexobj(h) else 0, Hd.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == fo.OK, fo.lib().fir_os_last_error()
    torch.cuda.synchronize()
    return Hd


def _filter(plan, x, real):
    import torch
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    st = torch.zeros(plan.M - 1, dtype=xd.dtype, device="cuda")
    plan.execute(xd, yd, st)
    torch.cuda.synchronize()
    plan.device_status()
    return yd.cpu().numpy()


def test_consecutive_calls_match_the_allocating_path(fo):
    cases = [W.scaled(W.WORKLOADS["C2"], 7, 100), W.scaled(W.WORKLOADS["C3"], 2, 100),
             W.scaled(W.WORKLOADS["C4"], 9, 5)]
    outs = []
    for w in cases:  # consecutive calls reuse the same fixed array
        h = W.make_h_device(w)
        Hd = _noalloc_response(fo, h, w.N)
        hp = np.zeros(w.N, np.complex128)
        hp[: w.M] = h
        H64 = np.fft.fft(hp)
        H = Hd.cpu().numpy()
        assert np.abs(H - H64).max() <= 1e-6 * np.abs(H64).max()
        x = W.make_x(w)
        import torch
        plan_alloc = fo.Plan(w.M, w.N, torch.from_numpy(h).cuda(), real=w.real)
        plan_given = fo.Plan(w.M, w.N, Hd, real=w.real, coef_kind=fo.COEF_FREQ)
        y_alloc = _filter(plan_alloc, x, w.real)
        y_given = _filter(plan_given, x, w.real)
        rel_tol, abs_tol = W.tolerance(W.oracle_h(w), x)
        rel, mx = W.errors(y_given, y_alloc)
        assert rel <= rel_tol and mx <= abs_tol, (w.name, rel, mx)
        import oracle
        want, _ = oracle.direct(x, W.oracle_h(w))
        rel, mx = W.errors(y_given, want)
        assert rel <= rel_tol and mx <= abs_tol, (w.name, "against the oracle", rel, mx)
        outs.append(y_given)
    assert len(outs) == 3


def test_rejects_sizes_beyond_the_fixed_array(fo):
    import torch
    h = torch.zeros(16, dtype=torch.float32, device="cuda")
    H = torch.zeros(16, dtype=torch.complex64, device="cuda")
    L = fo.lib()
    assert L.fir_os_frequency_response_noalloc(h.data_ptr(), 16, 1 << 17, 0, H.data_ptr(), None) \
        == fo.E_UNSUPPORTED
    assert b"65536" in L.fir_os_last_error()
    assert L.fir_os_frequency_response_noalloc(None, 16, 64, 0, H.data_ptr(), None) == fo.E_INVAL
