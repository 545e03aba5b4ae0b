"""Plant typical mistakes into a copy of the oracle's C source and check that the pins
catch every one (CPU only; nothing here touches a GPU).  This is what makes the pins worth
trusting: a dropped term, a wrong sign or index, a transposed operand each fails a pin."""
import os
import shutil
import tempfile

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "correlation instead of convolution": (
        "fo_xt(x, n, s0, M, j - m, &xr, &xi);", "fo_xt(x, n, s0, M, j + m - (M - 1), &xr, &xi);"),
    "conjugated complex product": (
        "ar += hr * xr - hi * xi;", "ar += hr * xr + hi * xi;"),
    "state read newest-first": (
        "*re = s0 ? s0[2 * s] : 0.0;", "*re = s0 ? s0[2 * ((M - 2) - s)] : 0.0;"),
    "last tap dropped": (
        "for (int m = 0; m < M; ++m) {", "for (int m = 0; m < M - 1; ++m) {"),
    "fft twiddle sign flipped": (
        "double ang = sign * 2.0 * FO_PI * (double)q / (double)len;",
        "double ang = -sign * 2.0 * FO_PI * (double)q / (double)len;"),
    "fft inverse not scaled": (
        "for (int64_t i = 0; i < 2 * N; ++i) z[i] /= (double)N;",
        "for (int64_t i = 0; i < 2 * N; ++i) z[i] /= 1.0;"),
    "fft butterfly operands swapped": (
        "z[2 * b] = ar - br;", "z[2 * b] = br - ar;"),
    "dft sign fixed to +": (
        "double ang = sign * 2.0 * FO_PI * (double)e / (double)N;",
        "double ang = 2.0 * FO_PI * (double)e / (double)N;"),
    "overlap-save keeps the wrong window": (
        "y[2 * o] = E[2 * (M - 1 + j)];", "y[2 * o] = E[2 * ((M + j) % N)];"),
    "overlap-save block starts one sample early": (
        "fo_xt(x, n, s0, M, i * L - (M - 1) + t, &E[2 * t], &E[2 * t + 1]);",
        "fo_xt(x, n, s0, M, i * L - M + t, &E[2 * t], &E[2 * t + 1]);"),
    "overlap-save multiplies by conj(H)": (
        "E[2 * t + 1] = fr * hi + fi * hr;", "E[2 * t + 1] = -fr * hi + fi * hr;"),
    "frequency response padded at the head": (
        "memcpy(H, h, sizeof(double) * 2 * (size_t)M);",
        "memcpy(H + 2 * (N - M), h, sizeof(double) * 2 * (size_t)M);"),
    "state carry off by one": (
        "fo_xt(x, n, s0, M, n - (int64_t)(M - 1) + t, &re, &im);",
        "fo_xt(x, n, s0, M, n - (int64_t)M + t, &re, &im);"),
    "channelizer twiddle sign flipped": (
        "const double ang = -2.0 * FO_PI * (double)e / (double)K;",
        "const double ang = 2.0 * FO_PI * (double)e / (double)K;"),
    "channelizer output at the start of the hop": (
        "const int64_t t0 = m * D + D - 1;", "const int64_t t0 = m * D;"),
    "channelizer prototype reversed": (
        "const double hr = h[2 * l] * wr - h[2 * l + 1] * wi, hi = h[2 * l] * wi + h[2 * l + 1] * wr;",
        "const double hr = h[2 * (Nh - 1 - l)] * wr - h[2 * (Nh - 1 - l) + 1] * wi, "
        "hi = h[2 * (Nh - 1 - l)] * wi + h[2 * (Nh - 1 - l) + 1] * wr;"),
    "channelizer modulation period D instead of K": (
        "const int64_t e = ((int64_t)q * l) % K;", "const int64_t e = ((int64_t)q * l) % D;"),
    "channelizer conjugated product": (
        "im += hr * a[1] + hi * a[0];", "im += hr * a[1] - hi * a[0];"),
    "sampled evaluator shifted": (
        "fo_one(x, n, h, M, s0, idx[q], &y_at[2 * q], &y_at[2 * q + 1]);",
        "fo_one(x, n, h, M, s0, idx[q] + 1, &y_at[2 * q], &y_at[2 * q + 1]);"),
}


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(workdir, name):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    tag = "".join(c if c.isalnum() else "_" for c in name)
    csrc = os.path.join(workdir, tag + ".c")
    with open(csrc, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_library(csrc, os.path.join(workdir, tag + ".so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake '{name}'"
