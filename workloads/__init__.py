"""Seeded synthetic inputs for overlap-save FIR filtering.

This module is shared by the tests, the benchmark and the smoke check.  It holds the
input recipes only -- filter design, seeded signals, the five workload definitions and the
sampled index sets used for parity at full size -- and none of the filtering arithmetic
(no convolution, no block transform).  Both the CUDA path and the float64 oracle receive
the arrays it returns.

Workloads (the overlap-save method of "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法",
claim steps 1-6: an M-tap h, FFT size N, block length L = N - M + 1):

  C1  complex64 x, N(0,1) re/im, seed 0; k=64 blocks of L=193; M=64 real Hamming lowpass
      (cutoff 0.25 of Nyquist); N=256; S0=0; also split 32+32 blocks over two calls
  C2  complex64 x, seed 1; k=4096 blocks of L=3073; M=1024 real Hamming lowpass (0.1); N=4096
  C3  complex64 x, seed 2; k=1024 blocks of L=24577; M=8192 complex h, re/im N(0,1)/sqrt(M),
      seed 3; N=32768
  C4  real float32 x, uniform [-1,1), seed 4; 64 consecutive calls of 2^20 samples with the
      state carried; M=255 real Kaiser(beta=8) bandpass 0.2-0.3 of Nyquist; N=1024, L=770
  C5  complex64 x, seed 5; k=2048 blocks of L=49152; the frequency response H is given:
      complex64, N=65536, the float64 FFT of an M=16385-tap complex h (re/im N(0,1)/sqrt(M),
      seed 6) zero-padded to N

Random numbers: numpy Generator(PCG64(seed)).  A complex signal draws all real parts,
then all imaginary parts, in float64, then is rounded to complex64; the oracle is fed
the rounded values, so both sides see bit-identical inputs.  Streams past 2^31 samples are
drawn on the device by torch's seeded generator instead (device_signal); the oracle gets
copies of the windows it needs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

# ----------------------------------------------------------------------------- windows


def hamming(M: int) -> np.ndarray:
    """Hamming window w[n] = 0.54 - 0.46 cos(2 pi n / (M-1)), n = 0..M-1 (float64)."""
    if M == 1:
        return np.ones(1)
    n = np.arange(M, dtype=np.float64)
    return 0.54 - 0.46 * np.cos(2.0 * np.pi * n / (M - 1))


def bessel_i0(x: np.ndarray) -> np.ndarray:
    """Modified Bessel function of the first kind, order 0, by its power series
    I0(x) = sum_k ((x/2)^k / k!)^2, summed until the terms stop changing the sum."""
    x = np.asarray(x, dtype=np.float64)
    q = (x / 2.0) ** 2
    term = np.ones_like(x)
    total = np.ones_like(x)
    for k in range(1, 500):
        term = term * q / (k * k)
        total = total + term
        if np.all(term <= 1e-17 * total):
            break
    return total


def kaiser(M: int, beta: float) -> np.ndarray:
    """Kaiser window w[n] = I0(beta sqrt(1 - (2n/(M-1) - 1)^2)) / I0(beta) (float64)."""
    if M == 1:
        return np.ones(1)
    n = np.arange(M, dtype=np.float64)
    r = 2.0 * n / (M - 1) - 1.0
    return bessel_i0(beta * np.sqrt(np.maximum(0.0, 1.0 - r * r))) / bessel_i0(np.array(beta))


def _sinc(t: np.ndarray) -> np.ndarray:
    """sin(pi t) / (pi t), 1 at t = 0."""
    t = np.asarray(t, dtype=np.float64)
    out = np.ones_like(t)
    nz = t != 0
    out[nz] = np.sin(np.pi * t[nz]) / (np.pi * t[nz])
    return out


def lowpass(M: int, cutoff: float, window: np.ndarray) -> np.ndarray:
    """Windowed-sinc lowpass with cutoff `cutoff` as a fraction of Nyquist (fs = 2),
    normalised to unit DC gain (sum h = 1).  float64."""
    t = np.arange(M, dtype=np.float64) - (M - 1) / 2.0
    h = cutoff * _sinc(cutoff * t) * window
    return h / h.sum()


def bandpass(M: int, c1: float, c2: float, window: np.ndarray) -> np.ndarray:
    """Windowed-sinc bandpass between c1 and c2 (fractions of Nyquist), normalised to unit
    gain magnitude at the band centre (c1 + c2) / 2.  float64."""
    t = np.arange(M, dtype=np.float64) - (M - 1) / 2.0
    h = (c2 * _sinc(c2 * t) - c1 * _sinc(c1 * t)) * window
    w0 = np.pi * (c1 + c2) / 2.0
    g = abs(np.sum(h * np.exp(-1j * w0 * np.arange(M))))
    return h / g


# ----------------------------------------------------------------------------- signals


def complex_normal(n: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """n complex samples, re then im drawn as N(0,1)*scale in float64 (complex128)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    re = rng.standard_normal(n)
    im = rng.standard_normal(n)
    out = np.empty(n, dtype=np.complex128)
    out.real = re * scale
    out.imag = im * scale
    return out


def uniform_real(n: int, seed: int) -> np.ndarray:
    """n real samples uniform in [-1, 1), float64."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.uniform(-1.0, 1.0, n)


def device_signal(n: int, real: bool, seed: int, device: str = "cuda"):
    """n input samples drawn on the device by torch's seeded generator, for streams too long to
    draw on the host (past 2^31 samples): float32 uniform in [-1, 1), or complex64 whose re
    and im are each N(0, 1/2).  Returns a torch tensor; windows of it are copied to the host
    for the oracle."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if real:
        return torch.rand(n, generator=g, device=device, dtype=torch.float32).mul_(2.0).sub_(1.0)
    return torch.randn(n, generator=g, device=device, dtype=torch.complex64)


# ----------------------------------------------------------------------------- workloads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    real: bool            # real float32 samples (else complex64)
    M: int                # filter taps
    N: int                # FFT size
    calls: tuple          # samples per execute call, in order (state carried between)
    x_seed: int
    coef: str             # "time": h is passed; "freq": H is passed
    h_kind: str           # "hamming_lowpass" | "kaiser_bandpass" | "complex_normal"
    h_args: tuple = ()
    h_seed: Optional[int] = None
    description: str = ""
    channels: int = 1     # independent streams filtered together (each `calls` long)

    @property
    def L(self) -> int:
        return self.N - self.M + 1

    @property
    def n(self) -> int:
        return int(sum(self.calls))

    @property
    def sample_bytes(self) -> int:
        return 4 if self.real else 8

    @property
    def h_complex(self) -> bool:
        return self.h_kind == "complex_normal"

    def with_calls(self, calls) -> "Workload":
        return dataclasses.replace(self, calls=tuple(int(c) for c in calls))

    def blocks(self) -> int:
        """Blocks of L outputs over the whole stream (a single call's count when the
        calls are block-aligned)."""
        return -(-self.n // self.L)


WORKLOADS = {
    "C1": Workload("C1", False, 64, 256, (64 * 193,), 0, "time", "hamming_lowpass", (0.25,),
                   description="complex64, M=64 Hamming lowpass 0.25, N=256, L=193, k=64"),
    "C1split": Workload("C1split", False, 64, 256, (32 * 193, 32 * 193), 0, "time",
                        "hamming_lowpass", (0.25,),
                        description="C1 split 32+32 blocks over two calls with state carry"),
    "C2": Workload("C2", False, 1024, 4096, (4096 * 3073,), 1, "time", "hamming_lowpass", (0.1,),
                   description="complex64, M=1024 Hamming lowpass 0.1, N=4096, L=3073, k=4096"),
    "C3": Workload("C3", False, 8192, 32768, (1024 * 24577,), 2, "time", "complex_normal", (),
                   h_seed=3,
                   description="complex64, M=8192 complex h, N=32768, L=24577, k=1024"),
    "C4": Workload("C4", True, 255, 1024, tuple([1 << 20] * 64), 4, "time", "kaiser_bandpass",
                   (8.0, 0.2, 0.3),
                   description="real f32, 64 calls of 2^20, M=255 Kaiser(8) bandpass 0.2-0.3, "
                               "N=1024, L=770"),
    "C5": Workload("C5", False, 16385, 65536, (2048 * 49152,), 5, "freq", "complex_normal", (),
                   h_seed=6,
                   description="complex64, H given (N=65536, FFT of M=16385 complex h), "
                               "L=49152, k=2048"),
    # banks of channels sharing one filter, filtered in one batched call per step
    "C2x16": Workload("C2x16", False, 1024, 4096, (256 * 3073,), 1, "time", "hamming_lowpass", (0.1,),
                      description="16 channels of complex64, C2's filter (M=1024, N=4096, L=3073), "
                                  "k=256 blocks per channel, one batched call",
                      channels=16),
    "C4x64": Workload("C4x64", True, 255, 1024, (1 << 20,), 4, "time", "kaiser_bandpass", (8.0, 0.2, 0.3),
                      description="64 channels of real f32, C4's filter (M=255, N=1024, L=770), "
                                  "2^20 samples per channel, one batched call",
                      channels=64),
}


def make_h64(w: Workload) -> np.ndarray:
    """The filter taps in float64 (real workloads: float64 array; complex: complex128)."""
    if w.h_kind == "hamming_lowpass":
        (c,) = w.h_args
        return lowpass(w.M, c, hamming(w.M))
    if w.h_kind == "kaiser_bandpass":
        beta, c1, c2 = w.h_args
        return bandpass(w.M, c1, c2, kaiser(w.M, beta))
    if w.h_kind == "complex_normal":
        return complex_normal(w.M, w.h_seed, 1.0 / math.sqrt(w.M))
    raise ValueError(w.h_kind)


def make_h_device(w: Workload) -> np.ndarray:
    """The taps as handed to the GPU: float32 for real h, complex64 for complex h."""
    h = make_h64(w)
    return h.astype(np.complex64 if np.iscomplexobj(h) else np.float32)


def make_H_given(w: Workload) -> np.ndarray:
    """For coef == "freq": H = float64 FFT of h zero-padded to N, rounded to complex64."""
    h = make_h64(w)
    hp = np.zeros(w.N, dtype=np.complex128)
    hp[: w.M] = h
    return np.fft.fft(hp).astype(np.complex64)


def oracle_h(w: Workload) -> np.ndarray:
    """The taps the oracle filters with, as complex128: the float32/complex64 taps the GPU
    received (promoted exactly), or for a given H the float64 taps it was made from."""
    if w.coef == "freq":
        return make_h64(w).astype(np.complex128)
    return make_h_device(w).astype(np.complex128)


def make_x(w: Workload) -> np.ndarray:
    """The whole input stream (all calls concatenated): complex64 or float32."""
    if w.real:
        return uniform_real(w.n, w.x_seed).astype(np.float32)
    return complex_normal(w.n, w.x_seed).astype(np.complex64)


def make_x_shard(w: Workload, g: int) -> np.ndarray:
    """Shard g of a stream of several workload-sized shards (one per GPU of a multi-GPU run):
    shard 0 is make_x(w); shard g > 0 draws the same distribution from seed x_seed + 1000 g."""
    if g == 0:
        return make_x(w)
    seed = w.x_seed + 1000 * g
    if w.real:
        return uniform_real(w.n, seed).astype(np.float32)
    return complex_normal(w.n, seed).astype(np.complex64)


def make_x_channels(w: Workload) -> np.ndarray:
    """The inputs of all channels, shape (channels, n): channel c is make_x_shard(w, c)."""
    return np.stack([make_x_shard(w, c) for c in range(w.channels)])


def make_state0(w: Workload) -> np.ndarray:
    """Initial state S0 = 0 (M-1 samples)."""
    return np.zeros(w.M - 1, dtype=np.float32 if w.real else np.complex64)


def scaled(w: Workload, blocks: int, tail: int = 0, calls: int = 1) -> Workload:
    """The same filter and FFT size on a shorter stream: `blocks` whole blocks plus
    `tail` extra samples (a ragged last block), split into `calls` nearly equal calls."""
    total = blocks * w.L + tail
    base = total // calls
    sizes = [base] * calls
    sizes[-1] += total - base * calls
    return dataclasses.replace(w, name=f"{w.name}[{blocks}b+{tail}]", calls=tuple(sizes))


def sample_indices(n: int, L: int, seed: int = 1234, whole_blocks=None, n_random: int = 1 << 16,
                   boundary: int = 2) -> np.ndarray:
    """A seeded set of output indices for parity checks at sizes where the oracle cannot
    evaluate every output: every output of the listed blocks (default: 0, 1, k/2, k-1),
    the outputs within `boundary` of every block boundary, and `n_random` uniform draws.
    Sorted, unique, int64."""
    k = -(-n // L)
    if whole_blocks is None:
        whole_blocks = sorted({0, min(1, k - 1), k // 2, k - 1})
    parts: List[np.ndarray] = []
    for b in whole_blocks:
        lo, hi = b * L, min(n, (b + 1) * L)
        parts.append(np.arange(lo, hi, dtype=np.int64))
    starts = np.arange(0, k, dtype=np.int64) * L
    for d in range(-boundary, boundary + 1):
        parts.append(starts + d)
    rng = np.random.Generator(np.random.PCG64(seed))
    parts.append(rng.integers(0, n, n_random, dtype=np.int64))
    idx = np.unique(np.concatenate(parts))
    return idx[(idx >= 0) & (idx < n)]


def tolerance(h: np.ndarray, x: np.ndarray):
    """The parity bar: relative L2 error <= 1e-5 and max abs error <=
    1e-4 * ||h||_1 * max|x| (complex modulus), both measured in float64."""
    h1 = float(np.sum(np.abs(np.asarray(h, dtype=np.complex128))))
    xm = float(np.max(np.abs(x))) if x.size else 0.0
    return 1e-5, 1e-4 * h1 * xm


def errors(got: np.ndarray, want: np.ndarray):
    """(relative L2 error, max abs error) of got against want, in float64."""
    g = np.asarray(got).astype(np.complex128)
    w = np.asarray(want).astype(np.complex128)
    d = g - w
    den = float(np.linalg.norm(w))
    rel = float(np.linalg.norm(d)) / den if den > 0 else float(np.linalg.norm(d))
    mx = float(np.max(np.abs(d))) if d.size else 0.0
    return rel, mx


# ----------------------------------------------------------------------------- channelizer
# The polyphase channelizer of "GPU加速短波信道化：多相滤波器组的并行重构与CUDA实现": input of
# 262144 = 2^18 float32 samples (40 ms at 6.5536 MHz); K = 128 or 1024 channels decimated by
# D = K/2 (50% overlapping channels); a Hamming-windowed lowpass prototype with cutoff 1/D of
# Nyquist (the page's firwin(Nh, 1/D, fs=2) design).  The page's prototype lengths (100 and 50
# taps) are shorter than K, which its own text flags as an error; the reading here is 8 taps per
# branch, Nh = 8 K.  Input: real N(0,1), seeded.


@dataclasses.dataclass(frozen=True)
class Channelizer:
    name: str
    K: int                # channels
    D: int                # decimation
    Nh: int               # prototype taps
    n: int                # input samples (a multiple of D)
    real: bool
    x_seed: int
    description: str = ""

    @property
    def nout(self) -> int:
        return self.n // self.D

    @property
    def sample_bytes(self) -> int:
        return 4 if self.real else 8


CHANNELIZERS = {
    "P1": Channelizer("P1", 128, 64, 1024, 1 << 18, True, 40,
                      "128 channels, D=64, Nh=1024 Hamming lowpass 1/64, 2^18 real samples"),
    "P2": Channelizer("P2", 1024, 512, 8192, 1 << 18, True, 41,
                      "1024 channels, D=512, Nh=8192 Hamming lowpass 1/512, 2^18 real samples"),
    "P2big": Channelizer("P2big", 1024, 512, 8192, 1 << 26, True, 42,
                         "1024 channels, D=512, Nh=8192 Hamming lowpass 1/512, 2^26 real samples"),
}


def chan_prototype(c: Channelizer) -> np.ndarray:
    """The prototype lowpass (float64): Hamming-windowed sinc, cutoff 1/D of Nyquist, unit DC gain."""
    return lowpass(c.Nh, 1.0 / c.D, hamming(c.Nh))


def chan_x(c: Channelizer) -> np.ndarray:
    """The input stream: real N(0,1) (float32) or complex N(0,1) (complex64)."""
    if c.real:
        rng = np.random.Generator(np.random.PCG64(c.x_seed))
        return rng.standard_normal(c.n).astype(np.float32)
    return complex_normal(c.n, c.x_seed).astype(np.complex64)
