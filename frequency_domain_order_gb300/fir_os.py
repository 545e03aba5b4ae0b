"""ctypes binding of libfir_os.so (include/fir_os.h) -- argument marshalling only.

Every step of the filtering runs in the library's CUDA kernels; this module converts torch
tensors to pointers and sizes, passes the current CUDA stream, and turns status codes into
exceptions.  There is no fallback: if the library is missing, :func:`lib` raises.

The method is frequency-domain overlap-save FIR filtering as claimed in
"一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法" (zl.czvv.com/42398539.html, 主权项 steps 1-6).
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfir_os.so")

OK = 0
E_INVAL = -1
E_UNSUPPORTED = -2
E_ALIGN = -3
E_NOMEM = -4
E_CUDA = -5
E_DEVICE = -6

REAL = 0
COMPLEX = 1
COEF_TIME = 0
COEF_FREQ = 1
DFT_FP32 = 0
DFT_TENSOR = 1

# every entry point include/fir_os.h declares, with its ctypes signature
_P, _I, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
SIGNATURES = {
    "fir_os_plan_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _I, _P, _P]),
    "fir_os_execute": (_I, [_P, _P, _I64, _P, _P, _P]),
    "fir_os_execute_host": (_I, [_P, _P, _I64, _P, _P, _P]),
    "fir_os_execute_batched": (_I, [_P, _P, _I64, _P, _I64, _P, _I64, _I64, _I, _P]),
    "fir_os_plan_destroy": (_I, [_P]),
    "fir_os_plan_info": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "fir_os_plan_kernel": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I),
                                ctypes.POINTER(_I)]),
    "fir_os_device_status": (_I, [_P, _P]),
    "fir_os_plan_set_wait_limit": (_I, [_P, _I64]),
    "fir_os_plan_set_dft_engine": (_I, [_P, _I]),
    "fir_os_debug_fail_alloc": (_I, [_I]),
    "fir_os_debug_live_allocs": (_I64, []),
    "fir_os_launches": (_I, [_P, _I64]),
    "fir_os_frequency_response_noalloc": (_I, [_P, _I, _I, _I, _P, _P]),
    "fir_os_choose_n": (_I, [_I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_double)]),
    "fir_os_predict_gsps": (_I, [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_double)]),
    "fir_os_fp32_probe": (_I, [_I, _P, ctypes.POINTER(ctypes.c_double)]),
    "fir_chan_plan_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _P, _P]),
    "fir_chan_execute": (_I, [_P, _P, _I64, _P, _P, _P]),
    "fir_chan_plan_info": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "fir_chan_plan_destroy": (_I, [_P]),
    "fir_os_status_string": (ctypes.c_char_p, [_I]),
    "fir_os_last_error": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def choose_n(M: int, real: bool = False, sms: int = 0):
    """fir_os_choose_n: (N, predicted GS/s) for an M-tap filter (host-only, no GPU needed)."""
    n, g = _I(), ctypes.c_double()
    _check(lib().fir_os_choose_n(int(M), REAL if real else COMPLEX, int(sms), ctypes.byref(n), ctypes.byref(g)))
    return n.value, g.value


def predict_gsps(M: int, N: int, real: bool = False, sms: int = 0) -> float:
    """fir_os_predict_gsps: predicted GS/s of an (M, N) plan (host-only)."""
    g = ctypes.c_double()
    _check(lib().fir_os_predict_gsps(int(M), int(N), REAL if real else COMPLEX, int(sms), ctypes.byref(g)))
    return g.value


def fp32_probe(iters: int, stream=None) -> float:
    """fir_os_fp32_probe: enqueue the FP32 multiply-add probe on `stream`; returns its flops."""
    f = ctypes.c_double()
    _check(lib().fir_os_fp32_probe(int(iters), _stream_handle(stream), ctypes.byref(f)))
    return f.value


def debug_fail_alloc(k: int):
    """fir_os_debug_fail_alloc: the k-th next allocation of the library fails (0 disarms)."""
    _check(lib().fir_os_debug_fail_alloc(int(k)))


def debug_live_allocs() -> int:
    """fir_os_debug_live_allocs: the library's live allocations (plan objects, device buffers)."""
    return int(lib().fir_os_debug_live_allocs())


class FirOsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def lib():
    """The loaded libfir_os.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m frequency_domain_order_gb300.build` "
                    "(or __graft_entry__.build()); there is no non-CUDA fallback")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _check(rc: int):
    if rc != OK:
        L = lib()
        msg = L.fir_os_last_error().decode() or L.fir_os_status_string(rc).decode()
        raise FirOsError(rc, msg)


def status_string(status: int) -> str:
    return lib().fir_os_status_string(status).decode()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


class Plan:
    """An overlap-save plan (fir_os_plan_create).

    coef: a CUDA tensor holding h (float32 or complex64, M taps; coef_kind COEF_TIME) or H
    (complex64, N bins, 16-byte aligned; COEF_FREQ).  real: x/y/state are float32 (else
    complex64)."""

    def __init__(self, M: int, N: int, coef, real: bool = False, coef_kind: int = COEF_TIME,
                 stream=None):
        import torch
        L = lib()
        if not coef.is_cuda or not coef.is_contiguous():
            raise ValueError("coef must be a contiguous CUDA tensor")
        coef_complex = 1 if coef.dtype == torch.complex64 else 0
        if coef.dtype not in (torch.float32, torch.complex64):
            raise ValueError("coef must be float32 or complex64")
        h = ctypes.c_void_p()
        _check(L.fir_os_plan_create(ctypes.byref(h), int(M), int(N), REAL if real else COMPLEX,
                                    int(coef_kind), coef_complex, coef.data_ptr(),
                                    _stream_handle(stream)))
        self._h = h
        self.M, self.N, self.real = int(M), int(N), bool(real)
        self.L = self.N - self.M + 1

    @property
    def handle(self):
        return self._h

    def execute(self, x, y, state, stream=None):
        """fir_os_execute on CUDA tensors (asynchronous on the stream)."""
        _check(lib().fir_os_execute(self._h, x.data_ptr(), int(x.numel()), y.data_ptr(),
                                    _ptr(state), _stream_handle(stream)))
        return y

    def execute_batched(self, x, y, state, stream=None):
        """fir_os_execute_batched on 2-D CUDA tensors (channels, n_samples) whose rows may be
        strided (contiguous within a row); state is (channels, M-1) or None when M == 1."""
        if x.dim() != 2 or y.shape != x.shape:
            raise ValueError("x and y must be 2-D tensors of the same shape (channels, n)")
        for t in (x, y) + ((state,) if state is not None else ()):
            if t.stride(1) != 1:
                raise ValueError("rows must be contiguous")
        channels, n = x.shape
        ss = state.stride(0) if state is not None else 0
        _check(lib().fir_os_execute_batched(self._h, x.data_ptr(), int(x.stride(0)), y.data_ptr(),
                                            int(y.stride(0)), _ptr(state), int(ss), int(n),
                                            int(channels), _stream_handle(stream)))
        return y

    def execute_host(self, x, y, state, stream=None):
        """fir_os_execute_host on CPU tensors (synchronous)."""
        _check(lib().fir_os_execute_host(self._h, x.data_ptr(), int(x.numel()), y.data_ptr(),
                                         _ptr(state), _stream_handle(stream)))
        return y

    def info(self):
        M, N, L = _I(), _I(), _I()
        _check(lib().fir_os_plan_info(self._h, ctypes.byref(M), ctypes.byref(N), ctypes.byref(L)))
        return M.value, N.value, L.value

    def kernel(self):
        k, c, g, s = _I(), _I(), _I(), _I()
        _check(lib().fir_os_plan_kernel(self._h, ctypes.byref(k), ctypes.byref(c), ctypes.byref(g),
                                        ctypes.byref(s)))
        kind = {0: "cta", 1: "cluster", 2: "tmem-resident"}.get(k.value, str(k.value))
        return {"kind": kind, "cluster": c.value, "grid": g.value,
                "smem_bytes": s.value}

    def launches(self, n: int) -> int:
        """Kernels one execute() of n samples launches."""
        rc = lib().fir_os_launches(self._h, int(n))
        if rc < 0:
            _check(rc)
        return rc

    def device_status(self, stream=None):
        _check(lib().fir_os_device_status(self._h, _stream_handle(stream)))

    def set_dft_engine(self, engine: int):
        """fir_os_plan_set_dft_engine: DFT_FP32 (default) or DFT_TENSOR (N = 4096 and N >= 16384)."""
        _check(lib().fir_os_plan_set_dft_engine(self._h, int(engine)))

    def set_wait_limit(self, limit_ns: int):
        """fir_os_plan_set_wait_limit: the kernels' limit for one bulk-copy wait (0: every wait
        runs out at once and the fallback gather runs)."""
        _check(lib().fir_os_plan_set_wait_limit(self._h, int(limit_ns)))

    def close(self):
        if getattr(self, "_h", None):
            lib().fir_os_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class ChanPlan:
    """A polyphase DFT channelizer (fir_chan_plan_*): K channels of the prototype h, decimated
    by D.  h is a CUDA float32 tensor of Nh taps."""

    def __init__(self, K: int, D: int, h, real: bool = True, stream=None):
        hp = _P()
        _check(lib().fir_chan_plan_create(ctypes.byref(hp), int(K), int(D), int(h.numel()),
                                          REAL if real else COMPLEX, h.data_ptr(), _stream_handle(stream)))
        self._h = hp
        self.K, self.D, self.Nh, self.real = int(K), int(D), int(h.numel()), real

    def execute(self, x, y, state, stream=None):
        """fir_chan_execute on CUDA tensors: x (n,), y (n / D, K) complex64, state (Nh - 1,)."""
        _check(lib().fir_chan_execute(self._h, x.data_ptr(), int(x.numel()), y.data_ptr(), _ptr(state),
                                      _stream_handle(stream)))
        return y

    def close(self):
        if self._h:
            lib().fir_chan_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
