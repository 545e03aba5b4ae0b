"""Randomised cases against the float64 oracle, fixed seed: every FFT size from 64 to 65536,
real and complex data (real or complex taps), degenerate and random filter lengths, stream
lengths from empty to many waves of the GPU, streams cut into several calls, banks of channels,
channelizer banks of every supported K with hops that divide K or not, and the optional
tensor-core DFT engine on half of the plans that have it (N = 4096 and N >= 16384).

Each case checks the parity bar (rel-L2 <= 1e-5, max-abs <= 1e-4 ||h||_1 max|x|; sampled outputs
when the full oracle would be slow; for fewer than 16 outputs the relative bar's denominator is
floored, see _rel) and the carried state exactly.
"""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build
    build.build()


def _bar(h, x):
    return 1e-5, 1e-4 * np.abs(h).sum() * (np.abs(x).max() if x.size else 0.0)


def _rel(d, want, h, window):
    """Relative L2 error of d against want.  The relative bar is a property of an output vector:
    the rounding error of an FFT convolution is absolute, about eps log2(N) ||h||_2 rms(window)
    per sample, so a call of one or two outputs whose values happen to lie near zero would be
    held to more than float32 holds.  Below 16 outputs the denominator is floored at the size
    such outputs have for these inputs, sqrt(n) ||h||_2 rms(window)."""
    den = np.linalg.norm(want)
    if want.size < 16 and window.size:
        rms = np.sqrt(np.mean(np.abs(window.astype(np.complex128)) ** 2))
        den = max(den, np.sqrt(want.size) * np.linalg.norm(h) * rms)
    return np.linalg.norm(d) / max(den, 1e-30)


def _filter_case(rng):
    import torch
    from frequency_domain_order_gb300 import fir_os
    N = 1 << int(rng.integers(6, 17))
    real = bool(rng.integers(0, 2))
    M = int(rng.choice([1, 2, N // 4 + 1, N // 2, N - 1, N, int(rng.integers(1, N + 1))]))
    L = N - M + 1
    nmax = int(min(4e6, 2e7 / M))
    n = int(rng.integers(0, max(2, min(nmax, L * int(rng.choice([1, 3, 50, 2000, 20000])) + 1))))
    channels = int(rng.choice([1, 1, 1, 3]))
    hc = (not real) and bool(rng.integers(0, 2))
    h = (rng.standard_normal(M) + (1j * rng.standard_normal(M) if hc else 0)) / np.sqrt(M)
    h32 = h.astype(np.complex64 if hc else np.float32)
    dt = np.float32 if real else np.complex64

    def sig(k):
        return (rng.standard_normal(k) + (0 if real else 1j * rng.standard_normal(k))).astype(dt)
    x = np.stack([sig(n) for _ in range(channels)])
    s0 = np.stack([sig(M - 1) for _ in range(channels)])
    plan = fir_os.Plan(M, N, torch.from_numpy(h32).cuda(), real=real)
    tensor = (N == 4096 or N >= 16384) and bool(rng.integers(0, 2))  # the optional tensor-core DFT engine
    if tensor:
        plan.set_dft_engine(fir_os.DFT_TENSOR)
    xd = torch.from_numpy(x).cuda()
    yd = torch.full_like(xd, float("nan"))
    sd = torch.from_numpy(s0.copy()).cuda()
    cuts = sorted({0, n, *[int(c) for c in rng.integers(0, n + 1, int(rng.choice([0, 0, 1, 4])))]})
    for a, b in zip(cuts, cuts[1:]):
        if channels == 1:
            plan.execute(xd[0, a:b], yd[0, a:b], sd[0] if M > 1 else None)
        else:
            plan.execute_batched(xd[:, a:b], yd[:, a:b], sd if M > 1 else None)
    torch.cuda.synchronize()
    plan.device_status()
    y, s = yd.cpu().numpy(), sd.cpu().numpy()
    plan.close()
    label = (f"N={N} M={M} n={n} real={real} complex-h={hc} channels={channels} cuts={cuts[:6]}"
             f"{' tensor-core DFTs' if tensor else ''}")
    h64 = h32.astype(np.complex128)
    for c in range(channels):
        if n:
            if n * M <= 3e7:
                want, _ = oracle.direct(x[c], h64, s0[c] if M > 1 else None)
                got = y[c]
            else:
                idx = W.sample_indices(n, L, seed=c, n_random=2048)
                want = oracle.direct_at(x[c], h64, s0[c] if M > 1 else None, idx)
                got = y[c][idx]
            if real:
                want = want.real
            d = got.astype(np.complex128) - want
            rel = _rel(d, want, h64, np.concatenate([s0[c], x[c]]) if M > 1 else x[c])
            rt, at = _bar(h64, x[c])
            assert np.all(np.isfinite(got)) and rel <= rt and np.abs(d).max() <= at, (
                f"{label} channel {c}: finite {np.all(np.isfinite(got))}, rel-L2 {rel:.3g}, "
                f"max-abs {np.abs(d).max():.3g} (bar {at:.3g})")
        if M > 1:
            assert np.array_equal(s[c], np.concatenate([s0[c], x[c]])[-(M - 1):]), label


def _host_case(rng):
    """One fir_os_execute_host call on CPU tensors (page-locked buffers: the block kernel filters
    them in place, the other kernels through the chunked copy pipeline; pageable buffers: the
    pipeline), lengths from empty to several pipeline chunks with a ragged last one, two calls
    in a row so that the second starts from the carried state."""
    import torch
    from frequency_domain_order_gb300 import fir_os
    N = 1 << int(rng.integers(6, 17))
    real = bool(rng.integers(0, 2))
    M = int(rng.choice([1, 2, N // 4 + 1, N - 1, int(rng.integers(1, N + 1))]))
    L = N - M + 1
    span = L * (2 if real else 1)
    chunk = max(span, (1 << 21) // span * span)  # the pipeline's chunk: whole transforms
    n = int(rng.choice([0, 1, int(rng.integers(1, 5000)), chunk, chunk + int(rng.integers(1, chunk + 1)),
                        2 * chunk + 1]))
    n = min(n, 5_000_000)
    pinned = bool(rng.integers(0, 2))
    hc = (not real) and bool(rng.integers(0, 2))
    h = (rng.standard_normal(M) + (1j * rng.standard_normal(M) if hc else 0)) / np.sqrt(M)
    h32 = h.astype(np.complex64 if hc else np.float32)
    dt = np.float32 if real else np.complex64

    def sig(k):
        return (rng.standard_normal(k) + (0 if real else 1j * rng.standard_normal(k))).astype(dt)
    xs = [sig(n), sig(int(rng.integers(0, 3 * span)))]
    s0 = sig(M - 1)
    plan = fir_os.Plan(M, N, torch.from_numpy(h32).cuda(), real=real)
    tensor = (N == 4096 or N >= 16384) and bool(rng.integers(0, 2))  # the optional tensor-core DFT engine
    if tensor:
        plan.set_dft_engine(fir_os.DFT_TENSOR)
    sh = torch.from_numpy(s0.copy())
    if pinned:
        sh = sh.pin_memory()
    ys = []
    for x in xs:
        xh = torch.from_numpy(x)
        yh = torch.full_like(xh, float("nan"))
        if pinned:
            xh, yh = xh.pin_memory(), yh.pin_memory()
        plan.execute_host(xh, yh, sh if M > 1 else None)
        ys.append(yh.numpy().copy())
    plan.device_status()
    plan.close()
    label = (f"host N={N} M={M} n={[x.size for x in xs]} real={real} complex-h={hc} "
             f"{'page-locked' if pinned else 'pageable'}{' tensor-core DFTs' if tensor else ''}")
    # the two calls are one stream: the oracle filters their concatenation
    x = np.concatenate(xs)
    y = np.concatenate(ys)
    h64 = h32.astype(np.complex128)
    if x.size:
        nt = x.size
        ends = np.arange(0, nt + 1, chunk, dtype=np.int64)
        idx = np.concatenate([np.arange(0, min(nt, 64)), np.arange(max(0, nt - 64), nt), xs[0].size + np.arange(-3, 4),
                              (ends[:, None] + np.arange(-3, 4)[None, :]).ravel(), rng.integers(0, nt, 4096)])
        idx = np.unique(idx[(idx >= 0) & (idx < nt)])
        want = oracle.direct_at(x, h64, s0 if M > 1 else None, idx)
        if real:
            want = want.real
        got = y[idx]
        d = got.astype(np.complex128) - want
        rel = _rel(d, want, h64, np.concatenate([s0, x]) if M > 1 else x)
        rt, at = _bar(h64, x)
        assert np.all(np.isfinite(got)) and rel <= rt and np.abs(d).max() <= at, (
            f"{label}: finite {np.all(np.isfinite(got))}, rel-L2 {rel:.3g}, max-abs {np.abs(d).max():.3g} "
            f"(bar {at:.3g})")
    if M > 1:
        assert np.array_equal(sh.numpy(), np.concatenate([s0, x])[-(M - 1):]), label


def _chan_case(rng):
    import torch
    from frequency_domain_order_gb300 import fir_os
    K = 1 << int(rng.integers(6, 13))
    D = int(rng.choice([K, K // 2, K // 4, int(rng.integers(1, K + 1))]))
    Nh = max(1, int(rng.integers(1, 9)) * K - int(rng.integers(0, K)))
    real = bool(rng.integers(0, 2))
    nout = int(rng.choice([0, 1, 7, int(rng.integers(1, 3000)), 5000]))
    nout = min(nout, max(1, int(3e9 // (K * Nh))))
    n = nout * D
    h = (rng.standard_normal(Nh) / np.sqrt(Nh)).astype(np.float32)
    dt = np.float32 if real else np.complex64
    x = (rng.standard_normal(n) + (0 if real else 1j * rng.standard_normal(n))).astype(dt)
    s0 = (rng.standard_normal(Nh - 1) + (0 if real else 1j * rng.standard_normal(Nh - 1))).astype(dt)
    try:
        plan = fir_os.ChanPlan(K, D, torch.from_numpy(h).cuda(), real=real)
    except fir_os.FirOsError as e:  # more taps than shared memory holds at this K
        assert e.status == fir_os.E_UNSUPPORTED
        return
    yd = torch.full((nout, K), float("nan"), dtype=torch.complex64, device="cuda")
    sd = torch.from_numpy(s0.copy()).cuda() if Nh > 1 else None
    plan.execute(torch.from_numpy(x).cuda(), yd, sd)
    torch.cuda.synchronize()
    y = yd.cpu().numpy()
    plan.close()
    label = f"K={K} D={D} Nh={Nh} real={real} nout={nout}"
    if nout:
        ms = np.unique(np.concatenate([[0, nout - 1], rng.integers(0, nout, 12)]))
        want = oracle.channelize_at(x, h.astype(np.float64), K, D, s0 if Nh > 1 else None, ms)
        d = y[ms].astype(np.complex128) - want
        rel = np.linalg.norm(d) / max(np.linalg.norm(want), 1e-30)
        rt, at = _bar(h.astype(np.float64), x)
        assert np.all(np.isfinite(y[ms])) and rel <= rt and np.abs(d).max() <= at, label
    if Nh > 1:
        assert np.array_equal(sd.cpu().numpy(), np.concatenate([s0, x])[-(Nh - 1):]), label


@pytest.mark.parametrize("seed", range(12))
def test_random_cases(seed):
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    for _ in range(50):
        if rng.integers(0, 4) == 3:
            _chan_case(rng)
        else:
            _filter_case(rng)


@pytest.mark.parametrize("seed", range(4))
def test_random_host_buffer_cases(seed):
    rng = np.random.Generator(np.random.PCG64(2000 + seed))
    for _ in range(10):
        _host_case(rng)
