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


def pin_overlap_save_with_any_response(o):
    """With a response that is not the transform of an M-tap h (random bins), steps 2-5
    give, block by block, the kept part of a circular convolution: R_i[M-1 .. M-1+L) with
    R_i = IDFT(DFT(E_i) H), E_i = xt[i L - (M-1) .. i L - (M-1) + N), computed here with
    numpy's FFT on the extended input (state in front, zeros past x)."""
    rng = _rng(23)
    for M, N, n in [(7, 16, 45), (67, 256, 3 * 190 + 31), (1, 8, 13), (16, 16, 5)]:
        H = _cn(rng, N)
        x, s = _cn(rng, n), _cn(rng, M - 1)
        L = N - M + 1
        k = (n + L - 1) // L
        xt = np.concatenate([s, x, np.zeros(k * L + N)])
        want = np.concatenate([np.fft.ifft(np.fft.fft(xt[i * L: i * L + N]) * H)[M - 1: M - 1 + L]
                               for i in range(k)])[:n] if n else np.zeros(0, complex)
        y_os, _ = o.overlap_save(x, H, M, s)
        assert np.allclose(y_os, want, rtol=0, atol=1e-12 * max(1.0, np.abs(want).max())), (M, N, n)


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


# ----------------------------------------------------------------------------- channelizer
# The polyphase channelizer of "GPU加速短波信道化：多相滤波器组的并行重构与CUDA实现", read as
# the K-channel DFT analysis filter bank decimated by D: output vector m follows the m-th hop of
# D new samples, t_m = m D + D - 1, and channel q is x filtered by h(l) e^{-2 pi i q l / K}.


def _folded_response(h, K):
    """sum_l h[l] e^{-2 pi i r l / K} for r = 0..K-1, through numpy's FFT of the prototype
    folded modulo K (zero-padded to a multiple of K)."""
    pad = (-len(h)) % K
    return np.fft.fft(np.concatenate([h, np.zeros(pad)]).reshape(-1, K).sum(axis=0))


def pin_chan_tone(o):
    """A complex tone at frequency -p0/K that has been running forever (state included) gives
    every channel q the closed form e^{-2 pi i p0 t_m / K} * Hfold[(q - p0) mod K]."""
    rng = _rng(31)
    for K, D, Nh, p0 in [(8, 4, 24, 3), (16, 8, 64, 0), (16, 16, 48, 11), (6, 3, 18, 5)]:
        h = rng.standard_normal(Nh)
        n = 10 * D
        t = np.arange(-(Nh - 1), n)
        tone = np.exp(-2j * np.pi * p0 * t / K)
        y, _ = o.channelize(tone[Nh - 1:], h, K, D, tone[:Nh - 1])
        hf = _folded_response(h, K)
        tm = np.arange(n // D) * D + D - 1
        want = np.exp(-2j * np.pi * p0 * tm / K)[:, None] * hf[(np.arange(K) - p0) % K][None, :]
        assert np.abs(y - want).max() < 1e-11 * np.abs(h).sum(), (K, D, p0)


def pin_chan_impulse(o):
    """x = delta at t0 with zero state: y[m, q] = h[t_m - t0] e^{-2 pi i q (t_m - t0) / K} while
    0 <= t_m - t0 < Nh, else 0."""
    rng = _rng(32)
    K, D, Nh = 8, 2, 40
    h = rng.standard_normal(Nh)
    for t0 in (0, 3, 7):
        n = 40
        x = np.zeros(n)
        x[t0] = 1.0
        y, _ = o.channelize(x, h, K, D)
        for m in range(n // D):
            d = m * D + D - 1 - t0
            want = np.zeros(K, complex)
            if 0 <= d < Nh:
                want = h[d] * np.exp(-2j * np.pi * np.arange(K) * d / K)
            assert np.abs(y[m] - want).max() < 1e-13, (t0, m)


def pin_chan_single_channel_is_convolution(o):
    """K = 1, D = 1 is plain linear convolution with the state in front (numpy.convolve)."""
    rng = _rng(33)
    h, x, s0 = _cn(rng, 13), _cn(rng, 50), _cn(rng, 12)
    y, s1 = o.channelize(x, h, 1, 1, s0)
    want = np.convolve(np.concatenate([s0, x]), h)[12:12 + 50]
    assert np.abs(y[:, 0] - want).max() < 1e-12 * np.abs(h).sum()
    assert np.array_equal(s1, np.concatenate([s0, x])[-12:])


def pin_chan_hop_invariant(o):
    """Decimating by K keeps exactly the odd output vectors of decimating by K/2 (same times)."""
    rng = _rng(34)
    K, Nh = 8, 32
    h, x, s0 = rng.standard_normal(Nh), _cn(rng, 96), _cn(rng, Nh - 1)
    y1, _ = o.channelize(x, h, K, K, s0)
    y2, _ = o.channelize(x, h, K, K // 2, s0)
    assert np.array_equal(y1, y2[1::2])


def pin_chan_split_stream(o):
    """Two calls with the state carried equal one call, exactly; channelize_at picks rows."""
    rng = _rng(35)
    K, D, Nh = 16, 8, 48
    h, x, s0 = rng.standard_normal(Nh), _cn(rng, 160), _cn(rng, Nh - 1)
    y, s = o.channelize(x, h, K, D, s0)
    ya, sa = o.channelize(x[:64], h, K, D, s0)
    yb, sb = o.channelize(x[64:], h, K, D, sa)
    assert np.array_equal(np.concatenate([ya, yb]), y)
    assert np.array_equal(sb, s)
    ms = np.array([0, 5, 19, 3])
    assert np.array_equal(o.channelize_at(x, h, K, D, s0, ms), y[ms])


ALL_PINS = [
    pin_golden_tiny, pin_impulse, pin_step, pin_numpy_convolve, pin_exponential_eigen,
    pin_linearity_and_shift, pin_split_stream, pin_direct_at, pin_dft_textbook,
    pin_fft_library, pin_freq_response, pin_overlap_save_matches_definition,
    pin_overlap_save_with_any_response, pin_given_response_is_causal,
    pin_chan_tone, pin_chan_impulse, pin_chan_single_channel_is_convolution, pin_chan_hop_invariant,
    pin_chan_split_stream,
]
