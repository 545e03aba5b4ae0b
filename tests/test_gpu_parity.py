"""CUDA path against the float64 oracle, element by element, through the C ABI.

Small sizes compare every output; the full workload sizes (single call, the launch
configuration the benchmark times) compare a seeded sample of outputs that the oracle
evaluates one by one.  The bar is the one the method's target states: relative L2 error
<= 1e-5 and max abs error <= 1e-4 * ||h||_1 * max|x| (float64 error measurement).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_parity, make_plan, run_calls, run_device, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build
    build.build()


def _oracle_full(w, x, calls_state0=None):
    y, s = oracle.direct(x, W.oracle_h(w), calls_state0)
    return y, s


# ----------------------------------------------------------------------------- C1


def test_c1_full_and_state():
    w = W.WORKLOADS["C1"]
    x = W.make_x(w)
    plan = make_plan(w)
    y, st = run_calls(plan, x, w.calls)
    want, s_want = _oracle_full(w, x)
    assert_parity(y, want, W.oracle_h(w), x, "C1")
    assert np.array_equal(st, x[-(w.M - 1):])


def test_c1_split_is_bitwise_identical_to_single_call():
    w = W.WORKLOADS["C1split"]
    x = W.make_x(w)
    plan = make_plan(w)
    y1, s1 = run_calls(plan, x, (x.size,))
    y2, s2 = run_calls(plan, x, w.calls)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(s1, s2)
    want, _ = _oracle_full(w, x)
    assert_parity(y2, want, W.oracle_h(w), x, "C1 split")


# ----------------------------------------------------------------------------- scaled workloads


@pytest.mark.parametrize("name,blocks,tail,calls", [
    ("C2", 37, 1001, 1), ("C2", 37, 1001, 3), ("C3", 5, 12345, 2), ("C4", 41, 123, 5),
    ("C5", 3, 777, 2),
])
def test_scaled_workload(name, blocks, tail, calls):
    w = W.scaled(W.WORKLOADS[name], blocks, tail, calls)
    x = W.make_x(w)
    plan = make_plan(w)
    y, st = run_calls(plan, x, w.calls)
    h = W.oracle_h(w)
    if w.n * w.M <= 3e8:
        want, _ = oracle.direct(x, h)
        assert_parity(y, want, h, x, w.name)
    else:
        idx = W.sample_indices(w.n, w.L, seed=7, n_random=1 << 13)
        want = oracle.direct_at(x, h, None, idx)
        assert_parity(y[idx], want, h, x, w.name + " sampled")
    assert np.array_equal(st, x[-(w.M - 1):])


# ----------------------------------------------------------------------------- shards


@pytest.mark.parametrize("name,blocks,tail,parts", [
    ("C2", 37, 1001, 4), ("C3", 9, 12345, 3), ("C4", 41, 123, 5), ("C5", 5, 777, 2),
])
def test_shards_with_halos_equal_one_call(name, blocks, tail, parts):
    """Each shard filtered by its own call, its halo (the M-1 samples before it) as the state:
    the outputs concatenate to one call's bit for bit, and the last shard's state is S0'."""
    from frequency_domain_order_gb300.shard import shard_ranges, shard_states
    torch = pytest.importorskip("torch")
    w = W.scaled(W.WORKLOADS[name], blocks, tail)
    x = W.make_x(w)
    s0 = W.make_x(W.scaled(w, 1))[: w.M - 1]
    plan = make_plan(w)
    xd = to_dev(x)
    y1, st1 = run_device(plan, xd, (w.n,), to_dev(s0))
    ranges = shard_ranges(w.n, w.L, parts, real=w.real)
    states = shard_states(xd, to_dev(s0), ranges, w.M)
    y2 = torch.empty_like(xd)
    for (a, b), st in zip(ranges, states):
        st = st.clone()
        plan.execute(xd[a:b], y2[a:b], st)
        last = st
    torch.cuda.synchronize()
    plan.device_status()
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert np.array_equal(st1.cpu().numpy(), last.cpu().numpy())


@pytest.mark.parametrize("name", ["C4", "C1"])
def test_short_call_variant_equals_full_wave(name):
    """Calls of less than one wave (N <= 1024) run the kernel variant that keeps H and the
    twiddles in shared memory; longer calls keep them in Tensor Memory.  The same stream filtered
    in one call of about 2.5 waves and in calls of under one wave each (split on whole
    transforms) gives the same output and state bit for bit."""
    torch = pytest.importorskip("torch")
    base = W.WORKLOADS[name]
    plan = make_plan(base)
    groups = 512 // max(64, base.N // 16)
    per_unit = max(1, 64 // (base.N // 16)) * (2 if base.real else 1)  # blocks per work unit
    wave = plan.kernel()["grid"] * groups * per_unit  # blocks in one wave of units
    span = base.L * (2 if base.real else 1)
    w = W.scaled(base, (5 * wave) // 2, 0)
    x = W.make_x(w)
    s0 = W.make_x(W.scaled(base, 1))[: base.M - 1]
    xd = to_dev(x)
    y1, st1 = run_device(plan, xd, (w.n,), to_dev(s0))
    chunk = (wave * base.L * 2 // 3) // span * span  # two thirds of a wave, whole transforms
    calls = [chunk] * (w.n // chunk) + ([w.n % chunk] if w.n % chunk else [])
    y2, st2 = run_device(plan, xd, calls, to_dev(s0))
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert np.array_equal(st1.cpu().numpy(), st2.cpu().numpy())
    plan.close()


# ----------------------------------------------------------------------------- full size, sampled


@pytest.mark.parametrize("name", ["C2", "C3", "C5"])
def test_full_size_sampled(name):
    torch = pytest.importorskip("torch")
    w = W.WORKLOADS[name]
    x = W.make_x(w)
    plan = make_plan(w)
    xd = to_dev(x)
    yd, st = run_device(plan, xd, w.calls)
    k = w.blocks()
    idx = W.sample_indices(w.n, w.L, seed=11, whole_blocks=[0, k // 3, k - 1],
                           n_random=1 << 13 if w.M > 4096 else 1 << 15)
    got = yd[torch.from_numpy(idx).cuda()].cpu().numpy()
    h = W.oracle_h(w)
    want = oracle.direct_at(x, h, None, idx)
    assert_parity(got, want, h, x, name + " full-size sampled")
    assert np.array_equal(st.cpu().numpy(), x[-(w.M - 1):])
    del xd, yd


def test_c4_stream_of_64_calls_sampled():
    torch = pytest.importorskip("torch")
    w = W.WORKLOADS["C4"]
    x = W.make_x(w)
    plan = make_plan(w)
    xd = to_dev(x)
    yd, st = run_device(plan, xd, w.calls)
    idx = W.sample_indices(w.n, w.L, seed=13, n_random=1 << 16)
    # call boundaries too
    cb = np.cumsum(w.calls)[:-1]
    idx = np.unique(np.concatenate([idx, cb - 1, cb, cb + 1]))
    got = yd[torch.from_numpy(idx).cuda()].cpu().numpy()
    h = W.oracle_h(w)
    want = oracle.direct_at(x, h, None, idx)
    assert_parity(got, want.real, h, x, "C4 64 calls sampled")
    assert np.abs(want.imag).max() == 0
    assert np.array_equal(st.cpu().numpy(), x[-(w.M - 1):])


# ----------------------------------------------------------------------------- every N, both kinds


def _random_case(N, real, seed, M=None, n=None, hcomplex=None):
    rng = np.random.Generator(np.random.PCG64(seed))
    if M is None:
        M = int(rng.integers(1, N + 1))
    if hcomplex is None:
        hcomplex = (not real) and bool(rng.integers(0, 2))
    L = N - M + 1
    if n is None:
        n = int(min(3 * L + int(rng.integers(0, L + 1)), 200000))
    if real:
        x = rng.uniform(-1, 1, n).astype(np.float32)
        s0 = rng.uniform(-1, 1, M - 1).astype(np.float32)
    else:
        x = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
        s0 = (rng.standard_normal(M - 1) + 1j * rng.standard_normal(M - 1)).astype(np.complex64)
    if hcomplex:
        h = ((rng.standard_normal(M) + 1j * rng.standard_normal(M)) / np.sqrt(M)).astype(np.complex64)
    else:
        h = (rng.standard_normal(M) / np.sqrt(M)).astype(np.float32)
    return M, x, s0, h


def _plan(M, N, h, real, freq=False):
    from frequency_domain_order_gb300 import fir_os
    if freq:
        hp = np.zeros(N, np.complex128)
        hp[:M] = h
        H = np.fft.fft(hp).astype(np.complex64)
        return fir_os.Plan(M, N, to_dev(H), real=real, coef_kind=fir_os.COEF_FREQ)
    return fir_os.Plan(M, N, to_dev(h), real=real)


def _check_case(M, N, x, s0, h, real, calls, label, freq=False):
    plan = _plan(M, N, h, real, freq)
    y, st = run_calls(plan, x, calls, s0 if M > 1 else None)
    h64 = h.astype(np.complex128)
    if x.size * M <= 5e7:
        want, s_want = oracle.direct(x, h64, s0)
        assert_parity(y, want.real if real else want, h64, x, label)
    else:
        idx = W.sample_indices(x.size, N - M + 1, seed=3, n_random=4096)
        want = oracle.direct_at(x, h64, s0, idx)
        assert_parity(y[idx], want.real if real else want, h64, x, label + " sampled")
        s_want = oracle.state_next(x, s0, M)
    if M > 1:
        assert np.array_equal(st, s_want.real.astype(st.dtype) if real else s_want.astype(st.dtype))


@pytest.mark.parametrize("real", [False, True], ids=["complex", "real"])
@pytest.mark.parametrize("logn", list(range(6, 17)))
def test_every_size(logn, real):
    N = 1 << logn
    M, x, s0, h = _random_case(N, real, seed=100 * logn + real)
    cut = x.size // 3
    _check_case(M, N, x, s0, h, real, (cut, x.size - cut), f"N={N} M={M} real={real}")


# ----------------------------------------------------------------------------- edge cases


@pytest.mark.parametrize("real", [False, True], ids=["complex", "real"])
def test_edges(real):
    torch = pytest.importorskip("torch")
    N = 256
    # M = 1 (no state), M = N (L = 1), L < M - 1 (state written by its own kernel),
    # n < M - 1 (state shifts), a single sample
    for M, n in ((1, 1000), (N, 50), (200, 700), (100, 7), (64, 1)):
        M_, x, s0, h = _random_case(N, real, seed=M * 7 + n, M=M, n=n, hcomplex=False)
        _check_case(M, N, x, s0, h, real, (n,), f"edge M={M} n={n}")
    # n = 0 is a no-op: nothing written
    M, x, s0, h = _random_case(N, real, seed=5, M=40, n=10, hcomplex=False)
    plan = _plan(M, N, h, real)
    xd, st = to_dev(x), to_dev(s0)
    yd = torch.full_like(xd, 7)
    plan.execute(xd[:0], yd[:0], st)
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), s0)
    assert bool((yd == 7).all())


@pytest.mark.parametrize("real", [False, True], ids=["complex", "real"])
def test_misaligned_input_and_output(real):
    """x and y views starting one sample past a 16-byte boundary (bulk copies round out)."""
    torch = pytest.importorskip("torch")
    N = 4096
    M, x, s0, h = _random_case(N, real, seed=77, M=1000, n=40 * (N - 999) + 5, hcomplex=False)
    plan = _plan(M, N, h, real)
    xd = to_dev(np.concatenate([x[:1], x]))[1:]
    yfull = torch.empty(x.size + 1, dtype=xd.dtype, device="cuda")
    yd = yfull[1:]
    st = to_dev(s0)
    plan.execute(xd, yd, st)
    torch.cuda.synchronize()
    want, _ = oracle.direct(x, h.astype(np.complex128), s0)
    assert_parity(yd.cpu().numpy(), want.real if real else want, h.astype(np.complex128), x,
                  "misaligned")


def test_many_calls_random_lengths():
    N, real = 1024, True
    M, x, s0, h = _random_case(N, real, seed=9, M=255, n=60000, hcomplex=False)
    rng = np.random.Generator(np.random.PCG64(10))
    cuts = np.sort(rng.choice(np.arange(1, x.size), 25, replace=False))
    calls = np.diff(np.concatenate([[0], cuts, [x.size]]))
    _check_case(M, N, x, s0, h, real, tuple(int(c) for c in calls), "random calls")


# ----------------------------------------------------------------------------- step 1 variants


@pytest.mark.parametrize("N,M,real", [(4096, 1024, False), (1024, 255, True), (32768, 8192, False),
                                      (65536, 16385, False)])
def test_given_response_matches_taps(N, M, real):
    _, x, s0, h = _random_case(N, real, seed=N + M, M=M, n=3 * (N - M + 1) + 11, hcomplex=False)
    plan_t = _plan(M, N, h, real, freq=False)
    plan_f = _plan(M, N, h, real, freq=True)
    yt, _ = run_calls(plan_t, x, (x.size,), s0)
    yf, _ = run_calls(plan_f, x, (x.size,), s0)
    h64 = h.astype(np.complex128)
    idx = W.sample_indices(x.size, N - M + 1, seed=5, n_random=4096)
    want = oracle.direct_at(x, h64, s0, idx)
    assert_parity(yt[idx], want.real if real else want, h64, x, "taps")
    assert_parity(yf[idx], want.real if real else want, h64, x, "given H")


@pytest.mark.parametrize("N,real", [(256, False), (1024, True), (4096, False), (4096, True), (32768, False),
                                    (65536, False)])
def test_given_response_without_taps(N, real):
    """A given response that is not the transform of an M-tap filter (random bins, Hermitian
    for real data): every block is then a circular convolution with h_eff = IDFT(H), of which
    step 5 keeps R_i[M-1 .. M-1+L).  The oracle runs steps 2-5 block by block with the same
    H; the bar takes ||h_eff||_1 in place of ||h||_1.  Unlike a linear convolution, the result
    now depends on where the blocks start, so the stream is cut into calls at a multiple of L
    (a call's blocks start at its first sample)."""
    from frequency_domain_order_gb300 import fir_os
    rng = np.random.default_rng(7000 + N + real)
    M = N // 4 + 3
    L = N - M + 1
    n = 3 * L + L // 2 + 5
    G = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    if real:
        G = 0.5 * (G + np.conj(G[(-np.arange(N)) % N]))  # Hermitian: h_eff is real
        x = rng.uniform(-1, 1, n).astype(np.float32)
        s0 = rng.uniform(-1, 1, M - 1).astype(np.float32)
    else:
        x = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
        s0 = (rng.standard_normal(M - 1) + 1j * rng.standard_normal(M - 1)).astype(np.complex64)
    H = G.astype(np.complex64)
    plan = fir_os.Plan(M, N, to_dev(H), real=real, coef_kind=fir_os.COEF_FREQ)
    cut = 2 * L
    y, st = run_calls(plan, x, (cut, n - cut), s0)
    want, s_want = oracle.overlap_save(x, H, M, s0)
    h_eff = np.fft.ifft(H.astype(np.complex128))
    assert_parity(y, want.real if real else want, h_eff, x, f"N={N} real={real} given H")
    assert np.array_equal(st, s_want.real.astype(st.dtype) if real else s_want.astype(st.dtype))


# ----------------------------------------------------------------------------- host buffers


@pytest.mark.parametrize("pinned", [True, False], ids=["page-locked", "pageable"])
@pytest.mark.parametrize("name", ["C2", "C4", "C3"])
def test_host_path_equals_device_path(name, pinned):
    """Host buffers: page-locked ones are filtered in place over the host link, pageable ones
    through the chunked copy pipeline; both give the device path's output bit for bit."""
    torch = pytest.importorskip("torch")
    w = W.scaled(W.WORKLOADS[name], 1500 if name != "C3" else 40, 333)
    x = W.make_x(w)
    plan = make_plan(w)
    y_dev, s_dev = run_calls(plan, x, (x.size,))
    xh = torch.from_numpy(x.copy())
    yh = torch.empty_like(xh)
    sh = torch.zeros(w.M - 1, dtype=xh.dtype)
    if pinned:
        xh, yh, sh = xh.pin_memory(), yh.pin_memory(), sh.pin_memory()
    for _ in range(2):  # a second call continues from the carried state
        sh.zero_()
        plan.execute_host(xh, yh, sh)
        assert np.array_equal(yh.numpy().view(np.uint32), y_dev.view(np.uint32))
        assert np.array_equal(sh.numpy(), s_dev)


# ----------------------------------------------------------------------------- argument checks


def test_runtime_argument_checks():
    torch = pytest.importorskip("torch")
    from frequency_domain_order_gb300 import fir_os
    M, N = 64, 256
    h = np.ones(M, np.float32) / M
    plan = _plan(M, N, h, False)
    x = torch.zeros(1000, dtype=torch.complex64, device="cuda")
    st = torch.zeros(M - 1, dtype=torch.complex64, device="cuda")
    with pytest.raises(fir_os.FirOsError) as e:
        plan.execute(x[:600], x[400:], st)  # x and y overlap
    assert e.value.status == fir_os.E_INVAL
    with pytest.raises(fir_os.FirOsError) as e:
        plan.execute(x[:500], x[500:], x[:10])  # state overlaps x
    assert e.value.status == fir_os.E_INVAL
    raw = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    L = fir_os.lib()
    rc = L.fir_os_execute(plan.handle, raw.data_ptr() + 2, 10, raw.data_ptr() + 1024, st.data_ptr(), None)
    assert rc == fir_os.E_ALIGN
    # a given H off a 16-byte boundary
    Hbuf = torch.zeros(N + 1, dtype=torch.complex64, device="cuda")
    with pytest.raises(fir_os.FirOsError) as e:
        fir_os.Plan(M, N, Hbuf[1:], coef_kind=fir_os.COEF_FREQ)
    assert e.value.status == fir_os.E_ALIGN
    # real data needs a Hermitian H
    Hc = torch.zeros(N, dtype=torch.complex64, device="cuda")
    Hc[3] = 1.0
    with pytest.raises(fir_os.FirOsError) as e:
        fir_os.Plan(M, N, Hc, real=True, coef_kind=fir_os.COEF_FREQ)
    assert e.value.status == fir_os.E_UNSUPPORTED
    plan.device_status()


# ----------------------------------------------------------------------------- measurement aid


def test_fp32_probe_measures_a_plausible_peak():
    """fir_os_fp32_probe: the flops it reports over its event-timed duration give a peak between
    a tenth of and twice the nominal SMs x 128 lanes x 2 x max clock; bad arguments are rejected."""
    torch = pytest.importorskip("torch")
    from frequency_domain_order_gb300 import fir_os
    import ctypes
    stream = torch.cuda.current_stream()
    fir_os.fp32_probe(256, stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    flops = fir_os.fp32_probe(8192, stream)
    b.record(stream)
    b.synchronize()
    tflops = flops / (a.elapsed_time(b) * 1e-3) / 1e12
    props = torch.cuda.get_device_properties(0)
    nominal = props.multi_processor_count * 128 * 2 * 2.2e9 / 1e12
    assert flops > 0 and 0.1 * nominal < tflops < 2 * nominal, (tflops, nominal)
    L = fir_os.lib()
    f = ctypes.c_double()
    assert L.fir_os_fp32_probe(0, None, ctypes.byref(f)) == fir_os.E_INVAL
    assert L.fir_os_fp32_probe(16, None, None) == fir_os.E_INVAL
