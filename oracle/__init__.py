"""float64 CPU oracle for frequency-domain overlap-save FIR filtering -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package.  The CUDA library never calls it and shares no code with it: the arithmetic
lives in ``fir_oracle.c`` (plain C, float64), compiled here with gcc into
``liboracle_fir.so`` and called through ctypes.

Functions follow "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法" (zl.czvv.com/42398539.html),
claim (主权项):

* :func:`direct`          -- linear convolution with carried state, the plain definition
                             that overlap-save reaches exactly (steps 3 and 5 together)
* :func:`direct_at`       -- the same sum at chosen output indices (full-size parity)
* :func:`state_next`      -- step 3's carry of the newest M-1 samples into the next call
* :func:`dft` / :func:`fft` -- textbook DFT and the oracle's own radix-2 FFT
* :func:`freq_response`   -- step 1, H = FFT_N(h zero-padded)
* :func:`overlap_save`    -- steps 2-5 written out block by block (a second, independent
                             CPU formulation used to cross-check :func:`direct`)
* :func:`channelize`      -- the polyphase channelizer of "GPU加速短波信道化：多相滤波器组的
                             并行重构与CUDA实现" (a later row built on the same library), as
                             the defining sum of a K-channel DFT filter bank decimated by D

Pins (tests/test_oracle_pins.py): hand-worked tiny cases, impulse and step responses,
numpy.convolve and numpy.fft special cases, the complex-exponential eigen-relation,
linearity, time shift, split streams, and overlap_save == direct.  tests/test_oracle_mutants.py
plants typical mistakes into a copy of the C source and checks that a pin catches each.
No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fir_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_fir.so")
_lock = threading.Lock()
_default = None


def compile_library(src: str, out: str) -> str:
    """gcc -O2 -fopenmp shared library from a C source (portable flags only)."""
    d = os.path.dirname(os.path.abspath(out))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=d)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-Wall", "-Wextra",
           "-o", tmp, src, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, out)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError("oracle build failed:\n" + e.stderr) from e
    return out


def build(force: bool = False) -> str:
    """Compile fir_oracle.c into liboracle_fir.so next to it (skipped when up to date)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE):
        return _LIB
    return compile_library(SOURCE, _LIB)


def _c128(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a).astype(np.complex128))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes front end over one compiled copy of fir_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.fo_direct.argtypes = [P, I64, P, I, P, P]
        lib.fo_direct_at.argtypes = [P, I64, P, I, P, P, I64, P]
        lib.fo_state_next.argtypes = [P, I64, P, I, P]
        lib.fo_dft.argtypes = [P, I64, I, P]
        lib.fo_fft.argtypes = [P, I64, I]
        lib.fo_freq_response.argtypes = [P, I, I64, P]
        lib.fo_overlap_save.argtypes = [P, I64, P, I, I64, P, P]
        lib.fo_channelize.argtypes = [P, I64, P, I, I, I, P, P]
        lib.fo_channelize_at.argtypes = [P, I64, P, I, I, I, P, P, I64, P]
        for f in ("fo_direct", "fo_direct_at", "fo_state_next", "fo_dft", "fo_fft",
                  "fo_freq_response", "fo_overlap_save", "fo_channelize", "fo_channelize_at",
                  "fo_num_threads"):
            getattr(lib, f).restype = I
        self.lib = lib
        self.path = path

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise ValueError(f"oracle {what} rejected its arguments (code {rc})")

    def num_threads(self) -> int:
        """OpenMP threads the oracle runs on."""
        return int(self.lib.fo_num_threads())

    def state_next(self, x, state, M: int):
        """Last M-1 samples of concat(state, x) (complex128)."""
        x = _c128(x)
        s0 = _c128(np.zeros(M - 1) if state is None else state)
        out = np.empty(M - 1, dtype=np.complex128)
        self._check(self.lib.fo_state_next(_ptr(x), x.size, _ptr(s0), M, _ptr(out)),
                    "state_next")
        return out

    def direct(self, x, h, state=None):
        """y[j] = sum_{m<M} h[m] * xt[j-m], j = 0..n-1, with xt[t<0] = state[M-1+t].
        Returns (y, new_state), complex128."""
        x = _c128(x)
        h = _c128(h)
        M = h.size
        s0 = _c128(np.zeros(M - 1) if state is None else state)
        if s0.size != M - 1:
            raise ValueError("state must hold M-1 samples")
        y = np.empty(x.size, dtype=np.complex128)
        self._check(self.lib.fo_direct(_ptr(x), x.size, _ptr(h), M, _ptr(s0), _ptr(y)),
                    "direct")
        return y, self.state_next(x, s0, M)

    def direct_at(self, x, h, state, idx):
        """The definition at output indices idx only (complex128)."""
        x = _c128(x)
        h = _c128(h)
        M = h.size
        s0 = _c128(np.zeros(M - 1) if state is None else state)
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
        out = np.empty(idx.size, dtype=np.complex128)
        self._check(self.lib.fo_direct_at(_ptr(x), x.size, _ptr(h), M, _ptr(s0), _ptr(idx),
                                          idx.size, _ptr(out)), "direct_at")
        return out

    def dft(self, z, inverse: bool = False):
        """Textbook O(N^2) DFT; forward unscaled e^{-2 pi i nk/N}, inverse scaled 1/N."""
        z = _c128(z)
        out = np.empty_like(z)
        self._check(self.lib.fo_dft(_ptr(z), z.size, 1 if inverse else -1, _ptr(out)), "dft")
        return out

    def fft(self, z, inverse: bool = False):
        """The oracle's radix-2 FFT (power-of-two sizes), same convention as dft."""
        z = _c128(z).copy()
        self._check(self.lib.fo_fft(_ptr(z), z.size, 1 if inverse else -1), "fft")
        return z

    def freq_response(self, h, N: int):
        """Step 1: H = FFT_N(h zero-padded at the tail to N)."""
        h = _c128(h)
        H = np.empty(N, dtype=np.complex128)
        self._check(self.lib.fo_freq_response(_ptr(h), h.size, N, _ptr(H)), "freq_response")
        return H

    def overlap_save(self, x, H, M: int, state=None):
        """Steps 2-5 with a given N-point response H (N = H.size) and M-1 samples of
        state.  Returns (y, new_state)."""
        x = _c128(x)
        H = _c128(H)
        s0 = _c128(np.zeros(M - 1) if state is None else state)
        y = np.empty(x.size, dtype=np.complex128)
        self._check(self.lib.fo_overlap_save(_ptr(x), x.size, _ptr(H), M, H.size, _ptr(s0),
                                             _ptr(y)), "overlap_save")
        return y, self.state_next(x, s0, M)

    def channelize(self, x, h, K: int, D: int, state=None):
        """The K-channel DFT analysis filter bank decimated by D (the channelizer of
        "GPU加速短波信道化：多相滤波器组的并行重构与CUDA实现"), as its defining sum:
        y[m, q] = sum_l h[l] e^{-2 pi i q l / K} xt[m D + D - 1 - l].  len(x) must be a
        multiple of D; state holds len(h) - 1 samples (zeros if None).  Returns
        (y of shape (len(x) / D, K), complex128; the next state)."""
        x = _c128(x)
        h = _c128(h)
        Nh = h.size
        s0 = _c128(np.zeros(Nh - 1) if state is None else state)
        if s0.size != Nh - 1:
            raise ValueError("state must hold len(h) - 1 samples")
        if x.size % D:
            raise ValueError("len(x) must be a multiple of D")
        y = np.empty((x.size // D, K), dtype=np.complex128)
        self._check(self.lib.fo_channelize(_ptr(x), x.size, _ptr(h), Nh, K, D, _ptr(s0), _ptr(y)),
                    "channelize")
        return y, self.state_next(x, s0, Nh)

    def channelize_at(self, x, h, K: int, D: int, state, ms):
        """Rows ms of channelize(x, h, K, D, state)[0]."""
        x = _c128(x)
        h = _c128(h)
        Nh = h.size
        s0 = _c128(np.zeros(Nh - 1) if state is None else state)
        ms = np.ascontiguousarray(np.asarray(ms, dtype=np.int64))
        y = np.empty((ms.size, K), dtype=np.complex128)
        self._check(self.lib.fo_channelize_at(_ptr(x), x.size, _ptr(h), Nh, K, D, _ptr(s0), _ptr(ms),
                                              ms.size, _ptr(y)), "channelize_at")
        return y


def default() -> Oracle:
    """The oracle built from fir_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def num_threads() -> int:
    return default().num_threads()


def direct(x, h, state=None):
    return default().direct(x, h, state)


def direct_at(x, h, state, idx):
    return default().direct_at(x, h, state, idx)


def state_next(x, state, M: int):
    return default().state_next(x, state, M)


def dft(z, inverse: bool = False):
    return default().dft(z, inverse)


def fft(z, inverse: bool = False):
    return default().fft(z, inverse)


def freq_response(h, N: int):
    return default().freq_response(h, N)


def overlap_save(x, H, M: int, state=None):
    return default().overlap_save(x, H, M, state)


def channelize(x, h, K: int, D: int, state=None):
    return default().channelize(x, h, K, D, state)


def channelize_at(x, h, K: int, D: int, state, ms):
    return default().channelize_at(x, h, K, D, state, ms)
