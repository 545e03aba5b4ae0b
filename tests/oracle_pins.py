"""Pins for the float64 oracle: facts fixed by the overlap-save claim and by mathematics,
none of them a re-typing of the oracle's own formulas.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle disagrees.
The same pins run against the real oracle (test_oracle_pins.py) and against copies with
planted mistakes (test_oracle_mutants.py), which must each fail at least one pin.

Method: "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法" (zl.czvv.com/42398539.html),
主权项 steps 1-6.
"""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _pairs(a):
    a = np.asarray(a, dtype=np.float64).reshape(-1, 2) if len(a) else np.zeros((0, 2))
    return a[:, 0] + 1j * a[:, 1]


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _cn(rng, n):
    return rng.standard_normal(n) + 1j * rng.standard_normal(n)


def pin_golden_tiny(o):
    """Hand-worked tiny cases (tests/golden/direct_tiny.json): outputs and carried state."""
    with open(os.path.join(GOLDEN, "direct_tiny.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        h, x, s = _pairs(c["h"]), _pairs(c["x"]), _pairs(c["state"])
        y, s1 = o.direct(x, h, s)
        assert np.array_equal(y, _pairs(c["y"])), (c["name"], y)
        assert np.array_equal(s1, _pairs(c["state_out"])), (c["name"], s1)


def pin_impulse(o):
    """x = delta with zero state reproduces h, then zeros (exact)."""
    rng = _rng(11)
    for M, n in ((1, 5), (7, 20), (64, 100)):
        h = _cn(rng, M)
        x = np.zeros(n, dtype=complex)
        x[0] = 1.0
        y, _ = o.direct(x, h)
        want = np.zeros(n, dtype=complex)
        want[:M] = h[:n]
        assert np.array_equal(y, want), M


def pin_step(o):
    """x = 1 with zero state gives the running sum of h (numpy.cumsum)."""
    rng = _rng(12)
    M, n = 33, 80
    h = _cn(rng, M)
    y, _ = o.direct(np.ones(n), h)
    cs = np.cumsum(h)
    want = np.concatenate([cs, np.full(n - M, cs[-1])])
    assert np.allclose(y, want, rtol=0, atol=1e-12 * np.sum(np.abs(h)))


def pin_numpy_convolve(o):
    """With state, y equals numpy.convolve(concat(S0, x), h) from index M-1 on."""
    rng = _rng(13)
    for M, n in ((5, 40), (31, 200), (128, 333)):
        h, x, s = _cn(rng, M), _cn(rng, n), _cn(rng, M - 1)
        y, _ = o.direct(x, h, s)
        want = np.convolve(np.concatenate([s, x]), h)[M - 1: M - 1 + n]
        assert np.allclose(y, want, rtol=0, atol=1e-12 * np.abs(want).max()), M


def pin_exponential_eigen(o):
    """A complex exponential at DFT bin f is an eigenvector: y[t] = H[f] x[t], with H the
    numpy FFT of h zero-padded to N (the convolution/correlation and sign pin)."""
    rng = _rng(14)
    M, N, n = 20, 64, 150
    h = _cn(rng, M)
    H = np.fft.fft(np.concatenate([h, np.zeros(N - M)]))
    for f in (1, 5, 37):
        t = np.arange(-(M - 1), n)
        e = np.exp(2j * np.pi * f * t / N)
        y, _ = o.direct(e[M - 1:], h, e[: M - 1])
        assert np.allclose(y, H[f] * e[M - 1:], rtol=0, atol=1e-11), f


def pin_linearity_and_shift(o):
    """Linearity in x, and a delay of d samples (zero state) delays the output by d."""
    rng = _rng(15)
    M, n, d = 17, 90, 7
    h, x1, x2 = _cn(rng, M), _cn(rng, n), _cn(rng, n)
    a, b = 0.5 - 2j, 1.5 + 0.25j
    y1, _ = o.direct(x1, h)
    y2, _ = o.direct(x2, h)
    y12, _ = o.direct(a * x1 + b * x2, h)
    assert np.allclose(y12, a * y1 + b * y2, rtol=0, atol=1e-12 * np.abs(y12).max())
    ys, _ = o.direct(np.concatenate([np.zeros(d), x1]), h)
    assert np.allclose(ys[d:], y1, rtol=0, atol=1e-13 * np.abs(y1).max())
    assert np.all(ys[:d] == 0)


def pin_split_stream(o):
    """Cutting the stream into calls with the state carried equals one call, bit for bit
    (step 6: repeat from step 2 while data remains)."""
    rng = _rng(16)
    M = 9
    h, x, s = _cn(rng, M), _cn(rng, 100), _cn(rng, M - 1)
    y, s_end = o.direct(x, h, s)
    parts, st = [], s
    for lo, hi in ((0, 3), (3, 40), (40, 41), (41, 100)):
        yp, st = o.direct(x[lo:hi], h, st)
        parts.append(yp)
    assert np.array_equal(np.concatenate(parts), y)
    assert np.array_equal(st, s_end)
    assert np.array_equal(s_end, x[-(M - 1):])


def pin_direct_at(o):
    """The sampled evaluator agrees with numpy.convolve at arbitrary indices."""
    rng = _rng(17)
    M, n = 12, 300
    h, x, s = _cn(rng, M), _cn(rng, n), _cn(rng, M - 1)
    idx = np.array([0, 1, 10, 11, 12, 150, 298, 299])
    want = np.convolve(np.concatenate([s, x]), h)[M - 1: M - 1 + n][idx]
    got = o.direct_at(x, h, s, idx)
    assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())


def pin_dft_textbook(o):
    """DFT: the hand-worked N=4 case (tests/golden/dft4.json), delta -> ones,
    bin exponential -> N delta_f, numpy.fft agreement, inverse round trip."""
    with open(os.path.join(GOLDEN, "dft4.json")) as f:
        g = json.load(f)
    X = o.dft(_pairs(g["x"]))
    assert np.allclose(X, _pairs(g["X"]), rtol=0, atol=1e-14)
    N = 16
    d = np.zeros(N, complex)
    d[0] = 1
    assert np.allclose(o.dft(d), np.ones(N), rtol=0, atol=1e-14)
    f = 3
    e = np.exp(2j * np.pi * f * np.arange(N) / N)
    want = np.zeros(N, complex)
    want[f] = N
    assert np.allclose(o.dft(e), want, rtol=0, atol=1e-12)
    z = _cn(_rng(18), 48)
    assert np.allclose(o.dft(z), np.fft.fft(z), rtol=0, atol=1e-11)
    assert np.allclose(o.dft(o.dft(z), inverse=True), z, rtol=0, atol=1e-12)


def pin_fft_library(o):
    """The oracle's FFT equals numpy.fft (forward) and numpy.fft.ifft (inverse, 1/N)."""
    rng = _rng(19)
    for N in (1, 2, 4, 8, 64, 1024, 1 << 15):
        z = _cn(rng, N)
        F = o.fft(z)
        assert np.allclose(F, np.fft.fft(z), rtol=0, atol=1e-12 * max(1.0, np.abs(F).max())), N
        Fi = o.fft(z, inverse=True)
        assert np.allclose(Fi, np.fft.ifft(z), rtol=0, atol=1e-13 * max(1.0, np.abs(Fi).max())), N


def pin_freq_response(o):
    """Step 1: H equals numpy.fft.fft of h zero-padded at the tail."""
    rng = _rng(20)
    for M, N in ((1, 8), (64, 256), (255, 1024)):
        h = _cn(rng, M)
        H = o.freq_response(h, N)
        want = np.fft.fft(np.concatenate([h, np.zeros(N - M)]))
        assert np.allclose(H, want, rtol=0, atol=1e-12 * np.abs(want).max()), (M, N)


def pin_overlap_save_matches_definition(o):
    """Steps 2-5 (block FFT, multiply, inverse FFT, discard M-1) reach the linear
    convolution: ragged last block, L < M-1, n < M-1, n = 0, real and complex."""
    rng = _rng(21)
    cases = [(64, 256, 12352 // 4 + 17), (5, 16, 100), (9, 16, 50), (16, 16, 33),
             (100, 128, 7), (3, 4, 0), (1, 8, 21), (255, 1024, 2 * 770 + 606)]
    for M, N, n in cases:
        h, x, s = _cn(rng, M), _cn(rng, n), _cn(rng, M - 1)
        if M == 255:
            h, x, s = h.real + 0j, x.real + 0j, s.real + 0j
        H = np.fft.fft(np.concatenate([h, np.zeros(N - M)]))
        y_os, s_os = o.overlap_save(x, H, M, s)
        want = np.convolve(np.concatenate([s, x]), h)[M - 1: M - 1 + n]
        scale = max(1.0, np.abs(want).max()) if n else 1.0
        assert np.allclose(y_os, want, rtol=0, atol=1e-12 * scale), (M, N, n)
        assert np.array_equal(s_os, np.concatenate([s, x])[-(M - 1):] if M > 1 else s_os)


def pin_given_response_is_causal(o):
    """A response given as complex64 (the FFT of an M-tap h, rounded) inverts, through the
    oracle's own inverse FFT, to h below M and to ~0 from M on."""
    rng = _rng(22)
    M, N = 300, 2048
    h = _cn(rng, M) / np.sqrt(M)
    H = np.fft.fft(np.concatenate([h, np.zeros(N - M)])).astype(np.complex64)
    he = o.fft(H, inverse=True)
    assert np.abs(he[:M] - h).max() < 1e-6 * np.abs(h).max()
    assert np.abs(he[M:]).max() < 1e-6 * np.abs(h).max()


ALL_PINS = [
    pin_golden_tiny, pin_impulse, pin_step, pin_numpy_convolve, pin_exponential_eigen,
    pin_linearity_and_shift, pin_split_stream, pin_direct_at, pin_dft_textbook,
    pin_fft_library, pin_freq_response, pin_overlap_save_matches_definition,
    pin_given_response_is_causal,
]
