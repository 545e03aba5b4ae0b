"""The FFT-size chooser (fir_os_choose_n / fir_os_predict_gsps): host-only, no GPU needed.

It must return the power of two N >= M (64 .. 65536) that maximises its own prediction, the
prediction must scale with the SM count, and for the workloads' filters it picks the sizes the
measured table favours (M = 1024 -> 4096 and M = 8192 -> 32768, the sizes C2 and C3 use).
"""
import pytest

from frequency_domain_order_gb300 import build, fir_os


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


@pytest.mark.parametrize("real", [False, True])
@pytest.mark.parametrize("M", [1, 2, 63, 64, 65, 255, 1000, 1024, 3000, 8192, 16385, 40000, 65536])
def test_choice_is_the_argmax_of_the_prediction(M, real):
    N, g = fir_os.choose_n(M, real)
    assert N >= max(64, M) and N <= 65536 and N & (N - 1) == 0
    cands = [n for n in (1 << k for k in range(6, 17)) if n >= M]
    preds = {n: fir_os.predict_gsps(M, n, real) for n in cands}
    assert g == pytest.approx(max(preds.values()))
    assert preds[N] == pytest.approx(g)
    assert all(p > 0 for p in preds.values())


def test_prediction_scales_with_sms_and_choice_does_not_change():
    for M in (100, 1024, 8192):
        n152, g152 = fir_os.choose_n(M, False, 152)
        n76, g76 = fir_os.choose_n(M, False, 76)
        assert n152 == n76
        assert g76 == pytest.approx(g152 / 2)
        assert fir_os.choose_n(M, False, 0) == (n152, pytest.approx(g152))


def test_workload_filters():
    assert fir_os.choose_n(1024)[0] == 4096
    assert fir_os.choose_n(8192)[0] == 32768
    # more outputs per block at the same transform size predict more throughput
    assert fir_os.predict_gsps(1025, 4096) > fir_os.predict_gsps(3073, 4096)


def test_errors():
    L = fir_os.lib()
    import ctypes
    n, g = ctypes.c_int(), ctypes.c_double()
    assert L.fir_os_choose_n(0, fir_os.COMPLEX, 0, ctypes.byref(n), ctypes.byref(g)) == fir_os.E_INVAL
    assert L.fir_os_choose_n(70000, fir_os.COMPLEX, 0, ctypes.byref(n), ctypes.byref(g)) == fir_os.E_UNSUPPORTED
    assert L.fir_os_choose_n(10, 7, 0, ctypes.byref(n), ctypes.byref(g)) == fir_os.E_INVAL
    assert L.fir_os_choose_n(10, fir_os.COMPLEX, -1, ctypes.byref(n), ctypes.byref(g)) == fir_os.E_INVAL
    assert L.fir_os_choose_n(10, fir_os.COMPLEX, 0, None, ctypes.byref(g)) == fir_os.E_INVAL
    assert L.fir_os_choose_n(10, fir_os.COMPLEX, 0, ctypes.byref(n), None) == 0  # gsps may be NULL
    assert L.fir_os_predict_gsps(5000, 4096, fir_os.COMPLEX, 0, ctypes.byref(g)) == fir_os.E_UNSUPPORTED
    assert L.fir_os_predict_gsps(10, 100, fir_os.COMPLEX, 0, ctypes.byref(g)) == fir_os.E_UNSUPPORTED
    assert L.fir_os_predict_gsps(10, 1024, fir_os.COMPLEX, 0, None) == fir_os.E_INVAL
