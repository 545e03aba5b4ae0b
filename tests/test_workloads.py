"""The seeded input recipes (CPU only): windows and filters against numpy's own routines,
the workload table against the stated sizes, determinism, and the sampled index sets."""
import numpy as np
import pytest

import workloads as W


def test_hamming_matches_numpy():
    for M in (1, 2, 64, 1024):
        assert np.allclose(W.hamming(M), np.hamming(M), rtol=0, atol=1e-15)


def test_bessel_i0_and_kaiser_match_numpy():
    x = np.linspace(0, 30, 61)
    assert np.allclose(W.bessel_i0(x), np.i0(x), rtol=1e-13, atol=0)
    for M in (1, 2, 255):
        assert np.allclose(W.kaiser(M, 8.0), np.kaiser(M, 8.0), rtol=0, atol=1e-13)


def test_lowpass_normalised_and_symmetric():
    h = W.lowpass(64, 0.25, W.hamming(64))
    assert abs(h.sum() - 1.0) < 1e-14
    assert np.allclose(h, h[::-1], rtol=0, atol=1e-16)
    # windowed sinc: proportional to numpy.sinc * window
    t = np.arange(64) - 31.5
    ref = np.sinc(0.25 * t) * np.hamming(64)
    assert np.allclose(h, ref / ref.sum(), rtol=0, atol=1e-15)


def test_bandpass_unit_gain_at_centre():
    h = W.bandpass(255, 0.2, 0.3, W.kaiser(255, 8.0))
    w0 = np.pi * 0.25
    g = np.sum(h * np.exp(-1j * w0 * np.arange(255)))
    assert abs(abs(g) - 1.0) < 1e-12
    # stop bands are well below the pass band
    H = np.abs(np.fft.rfft(h, 8192))
    f = np.linspace(0, 1, H.size)
    assert H[f < 0.1].max() < 1e-3 and H[f > 0.4].max() < 1e-3


@pytest.mark.parametrize("name,n,k,L", [("C1", 12352, 64, 193), ("C2", 12587008, 4096, 3073),
                                        ("C3", 25166848, 1024, 24577),
                                        ("C4", 64 << 20, 87155, 770),
                                        ("C5", 100663296, 2048, 49152)])
def test_workload_sizes(name, n, k, L):
    w = W.WORKLOADS[name]
    assert w.n == n and w.L == L and w.blocks() == k
    assert w.N == w.L + w.M - 1


def test_c4_calls_and_partial_block():
    w = W.WORKLOADS["C4"]
    assert len(w.calls) == 64 and all(c == 1 << 20 for c in w.calls)
    assert (1 << 20) == 1361 * 770 + 606


def test_inputs_deterministic_and_typed():
    w = W.scaled(W.WORKLOADS["C2"], 3, 5)
    a, b = W.make_x(w), W.make_x(w)
    assert a.dtype == np.complex64 and np.array_equal(a, b)
    w4 = W.scaled(W.WORKLOADS["C4"], 3, 5)
    assert W.make_x(w4).dtype == np.float32
    assert W.make_h_device(W.WORKLOADS["C3"]).dtype == np.complex64
    assert W.make_h_device(W.WORKLOADS["C2"]).dtype == np.float32


def test_given_response_recipe():
    w = W.WORKLOADS["C5"]
    H = W.make_H_given(w)
    assert H.dtype == np.complex64 and H.size == w.N
    h = W.make_h64(w)
    he = np.fft.ifft(H.astype(np.complex128))
    assert np.abs(he[: w.M] - h).max() < 1e-6 * np.abs(h).max()
    assert np.abs(he[w.M:]).max() < 1e-6 * np.abs(h).max()


def test_sample_indices():
    n, L = 100 * 77 + 13, 77
    idx = W.sample_indices(n, L, n_random=500)
    assert idx.dtype == np.int64 and np.all(np.diff(idx) > 0)
    assert idx[0] == 0 and idx[-1] == n - 1
    for b in (0, 1, 50, 100):
        lo, hi = b * L, min(n, (b + 1) * L)
        assert np.isin(np.arange(lo, hi), idx).all()
    assert np.isin(np.array([77 * 30 - 2, 77 * 30 + 2]), idx).all()


def test_scaled_calls():
    w = W.scaled(W.WORKLOADS["C1"], 64, 0, calls=2)
    assert w.calls == (6176, 6176)
