"""The polyphase DFT channelizer (fir_chan_*) against the float64 oracle's defining sum.

The bar is the filter's: relative L2 error <= 1e-5 and max abs error <= 1e-4 * ||h||_1 *
max|x| (every output is a sum of Nh products h[l] x, modulated by unit phasors).  Cases: the
page's two banks (128 and 1024 channels, D = K/2, 2^18 real samples; the 1024-channel one
sampled), every supported K with real and complex input, decimations other than K/2, prototypes
that are not a multiple of K, a nonzero initial state, a stream split over calls (equal to one
call, bit for bit), long real-input calls whose transforms carry two output vectors each
(sampled, including the full-length 2^26-sample stream, and a split that keeps the pairs),
and the argument checks.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build
    build.build()


def _bar(h, x):
    return 1e-5, 1e-4 * np.abs(h).sum() * np.abs(x).max()


def _check(got, want, h, x, label):
    rel_tol, abs_tol = _bar(h, x)
    d = np.asarray(got, dtype=np.complex128) - want
    rel = np.linalg.norm(d) / np.linalg.norm(want)
    mx = np.abs(d).max()
    assert np.all(np.isfinite(np.asarray(got).view(np.float32))), f"{label}: non-finite output"
    assert rel <= rel_tol and mx <= abs_tol, f"{label}: rel-L2 {rel:.3g} (bar {rel_tol:g}), max-abs {mx:.3g} (bar {abs_tol:.3g})"


def _run(K, D, h, x, s0, calls=None):
    torch = pytest.importorskip("torch")
    from frequency_domain_order_gb300 import fir_os
    real = not np.iscomplexobj(x)
    plan = fir_os.ChanPlan(K, D, to_dev(h.astype(np.float32)), real=real)
    xd = to_dev(x)
    yd = torch.full((x.size // D, K), float("nan"), dtype=torch.complex64, device="cuda")
    sd = to_dev(s0) if len(h) > 1 else None
    calls = calls or [x.size]
    off = 0
    for c in calls:
        plan.execute(xd[off: off + c], yd[off // D: (off + c) // D], sd)
        off += c
    torch.cuda.synchronize()
    y, s = yd.cpu().numpy(), (sd.cpu().numpy() if sd is not None else None)
    plan.close()
    return y, s


@pytest.mark.parametrize("name", ["P1"])
def test_page_bank_full(name):
    c = W.CHANNELIZERS[name]
    h, x = W.chan_prototype(c), W.chan_x(c)
    s0 = np.zeros(c.Nh - 1, dtype=x.dtype)
    y, s = _run(c.K, c.D, h, x, s0)
    want, s_want = oracle.channelize(x, h.astype(np.float32).astype(np.float64), c.K, c.D, s0)
    _check(y, want, h, x, name)
    assert np.array_equal(s, x[-(c.Nh - 1):])


def test_page_bank_1024_sampled():
    c = W.CHANNELIZERS["P2"]
    h, x = W.chan_prototype(c), W.chan_x(c)
    s0 = np.zeros(c.Nh - 1, dtype=x.dtype)
    y, _ = _run(c.K, c.D, h, x, s0)
    rng = np.random.Generator(np.random.PCG64(3))
    ms = np.unique(np.concatenate([[0, 1, 15, 16, 17, c.nout - 1], rng.integers(0, c.nout, 24)]))
    want = oracle.channelize_at(x, h.astype(np.float32).astype(np.float64), c.K, c.D, s0, ms)
    _check(y[ms], want, h, x, "P2 sampled")


@pytest.mark.parametrize("real", [True, False], ids=["real", "complex"])
@pytest.mark.parametrize("K,D,Nh", [
    (64, 32, 512), (64, 1, 100), (128, 128, 300), (256, 128, 2048), (512, 7, 1500),
    (1024, 512, 4096), (2048, 1024, 6000), (4096, 2048, 8192), (4096, 4096, 1),
])
def test_sizes_against_oracle(K, D, Nh, real):
    rng = np.random.Generator(np.random.PCG64(K * 7 + D + Nh))
    nout = max(3, min(41, (1 << 16) // D, int(3e8) // (K * Nh)))  # bounded oracle work; 41 is odd
    n = nout * D
    h = rng.standard_normal(Nh) / np.sqrt(Nh)
    if real:
        x = rng.standard_normal(n).astype(np.float32)
        s0 = rng.standard_normal(Nh - 1).astype(np.float32)
    else:
        x = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
        s0 = (rng.standard_normal(Nh - 1) + 1j * rng.standard_normal(Nh - 1)).astype(np.complex64)
    y, s = _run(K, D, h, x, s0)
    want, s_want = oracle.channelize(x, h.astype(np.float32).astype(np.float64), K, D, s0)
    _check(y, want, h, x, f"K={K} D={D} Nh={Nh} {'real' if real else 'complex'}")
    if Nh > 1:
        s_want = np.asarray(s_want)
        assert np.array_equal(s, (s_want.real if real else s_want).astype(x.dtype))


@pytest.mark.parametrize("real", [True, False], ids=["real", "complex"])
def test_split_calls_equal_one_call(real):
    rng = np.random.Generator(np.random.PCG64(77))
    K, D, Nh = 256, 128, 2048
    n = 64 * D
    h = rng.standard_normal(Nh) / np.sqrt(Nh)
    if real:
        x = rng.standard_normal(n).astype(np.float32)
        s0 = rng.standard_normal(Nh - 1).astype(np.float32)
    else:
        x = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
        s0 = (rng.standard_normal(Nh - 1) + 1j * rng.standard_normal(Nh - 1)).astype(np.complex64)
    y1, s1 = _run(K, D, h, x, s0)
    y2, s2 = _run(K, D, h, x, s0, calls=[5 * D, 20 * D, 39 * D])
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(s1, s2)


def _pack_threshold(K):
    """Output vectors from which a real-input call shares each transform between two vectors:
    twice one wave of transforms (SMs x 512 threads / (K / 16) threads per transform)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 2 * sms * 512 // (K // 16)


def _sampled_vectors(nout, hist_vectors, seed, n_random=24):
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, 2, 3, hist_vectors - 1, hist_vectors, hist_vectors + 1, nout - 3, nout - 2, nout - 1]
    return np.unique(np.clip(np.concatenate([fixed, rng.integers(0, nout, n_random)]), 0, nout - 1))


def test_packed_real_calls():
    """Real input, calls long enough to pair output vectors in one transform: an odd vector
    count (the last vector unpaired), a nonzero state, sampled vectors against the oracle
    (first vectors reading the state, the boundary where the branches leave it, the end), and
    a split into two calls that keep the pairs, equal to one call bit for bit."""
    K, D, Nh = 1024, 512, 8192
    thr = _pack_threshold(K)
    nout = 2 * thr + 1
    rng = np.random.Generator(np.random.PCG64(91))
    h = W.chan_prototype(W.CHANNELIZERS["P2"]).astype(np.float64)
    x = rng.uniform(-1, 1, nout * D).astype(np.float32)
    s0 = rng.uniform(-1, 1, Nh - 1).astype(np.float32)
    y1, st1 = _run(K, D, h, x, s0)
    ms = _sampled_vectors(nout, Nh // D, seed=5)
    want = oracle.channelize_at(x, h.astype(np.float32).astype(np.float64), K, D, s0, ms)
    _check(y1[ms], want, h, x, "packed real, sampled")
    assert np.array_equal(st1, x[-(Nh - 1):])
    y2, st2 = _run(K, D, h, x, s0, calls=[thr * D, (nout - thr) * D])
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(st1, st2)


@pytest.mark.parametrize("K,D,taps_per_branch", [
    (64, 32, 8), (256, 128, 8), (4096, 2048, 3),   # K = 2D: four vectors per thread
    (256, 64, 6), (128, 128, 8), (1024, 300, 5),   # other hops: two vectors per transform
])
def test_packed_modes_other_banks(K, D, taps_per_branch):
    """Long real-input calls of other banks (every thread-group shape from 4 to 256 threads per
    transform): sampled vectors against the oracle, and a split into two calls of the pair
    mode equal to the single call bit for bit."""
    Nh = taps_per_branch * K - K // 3  # not a multiple of K
    thr = _pack_threshold(K)
    nout = 2 * thr + 3
    rng = np.random.Generator(np.random.PCG64(K + D))
    h = rng.standard_normal(Nh) / np.sqrt(Nh)
    x = rng.uniform(-1, 1, nout * D).astype(np.float32)
    s0 = rng.uniform(-1, 1, Nh - 1).astype(np.float32)
    y1, st1 = _run(K, D, h, x, s0)
    ms = _sampled_vectors(nout, -(-Nh // D), seed=K + 3 * D)
    want = oracle.channelize_at(x, h.astype(np.float32).astype(np.float64), K, D, s0, ms)
    _check(y1[ms], want, h, x, f"K={K} D={D} packed, sampled")
    assert np.array_equal(st1, x[-(Nh - 1):])
    y2, st2 = _run(K, D, h, x, s0, calls=[thr * D, (nout - thr) * D])
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(st1, st2)


def test_page_bank_1024_long_stream_sampled():
    """The 1024-channel bank over the benchmark's 2^26-sample stream (packed transforms, the
    benchmark's launch): sampled vectors against the oracle."""
    c = W.CHANNELIZERS["P2big"]
    h, x = W.chan_prototype(c), W.chan_x(c)
    s0 = np.zeros(c.Nh - 1, dtype=x.dtype)
    assert c.nout >= _pack_threshold(c.K)
    y, s = _run(c.K, c.D, h, x, s0)
    ms = _sampled_vectors(c.nout, c.Nh // c.D, seed=6)
    want = oracle.channelize_at(x, h.astype(np.float32).astype(np.float64), c.K, c.D, s0, ms)
    _check(y[ms], want, h, x, "P2big sampled")
    assert np.array_equal(s, x[-(c.Nh - 1):])


def test_argument_checks():
    torch = pytest.importorskip("torch")
    from frequency_domain_order_gb300 import fir_os
    L = fir_os.lib()
    import ctypes
    h = torch.ones(1024, device="cuda")
    p = ctypes.c_void_p()
    assert L.fir_chan_plan_create(ctypes.byref(p), 100, 50, 1024, fir_os.REAL, h.data_ptr(), None) == fir_os.E_UNSUPPORTED
    assert L.fir_chan_plan_create(ctypes.byref(p), 128, 129, 1024, fir_os.REAL, h.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_plan_create(ctypes.byref(p), 128, 0, 1024, fir_os.REAL, h.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_plan_create(ctypes.byref(p), 128, 64, 0, fir_os.REAL, h.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_plan_create(ctypes.byref(p), 128, 64, 1024, 9, h.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_plan_create(ctypes.byref(p), 128, 64, 1024, fir_os.REAL, None, None) == fir_os.E_INVAL
    assert L.fir_chan_plan_create(ctypes.byref(p), 128, 64, 1024, fir_os.REAL, h.data_ptr() + 2, None) == fir_os.E_ALIGN
    big = torch.ones(4096 * 16, device="cuda")
    assert L.fir_chan_plan_create(ctypes.byref(p), 4096, 2048, 4096 * 16, fir_os.REAL, big.data_ptr(), None) == fir_os.E_UNSUPPORTED
    plan = fir_os.ChanPlan(128, 64, h)
    x = torch.zeros(64 * 10, device="cuda")
    y = torch.zeros((10, 128), dtype=torch.complex64, device="cuda")
    s = torch.zeros(1023, device="cuda")
    hp = plan._h
    assert L.fir_chan_execute(hp, x.data_ptr(), 64 * 10 - 1, y.data_ptr(), s.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_execute(hp, x.data_ptr(), 640, y.data_ptr(), None, None) == fir_os.E_INVAL
    assert L.fir_chan_execute(hp, x.data_ptr(), 640, x.data_ptr() + 64, s.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_execute(hp, x.data_ptr(), 640, y.data_ptr(), x.data_ptr(), None) == fir_os.E_INVAL
    assert L.fir_chan_execute(hp, x.data_ptr(), 0, y.data_ptr(), s.data_ptr(), None) == 0
    assert L.fir_chan_execute(hp, x.data_ptr(), 640, y.data_ptr(), s.data_ptr(), None) == 0
    torch.cuda.synchronize()
    plan.close()
