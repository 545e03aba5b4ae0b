"""Calls past 2^31 samples: sample indices, byte offsets and channel offsets are 64-bit.

The filter (overlap-save, steps 2-6 of "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法") and
the polyphase channelizer run once each over a stream of a little more than 2^31 samples,
drawn on the device by a seeded generator.  Outputs are compared with the float64 oracle in
windows: every 32-bit boundary of the sample index and of the byte offset (2^28 .. 2^32 bytes,
2^31 samples), the block that spans sample 2^31, the first outputs (which read the initial
state), the last outputs, and seeded random windows.  The oracle evaluates each window from a
host copy of the input samples it needs (the output at t depends on x[t - M + 1 .. t] only).
The new state must equal the last M - 1 input samples bit for bit.

Each case holds 17-43 GB on the device and runs for well under a second on the GPU.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_parity, make_plan

pytestmark = pytest.mark.gpu

R = 48  # outputs per checked window


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build
    build.build()
    yield
    torch.cuda.empty_cache()


def _window_starts(n, L, M, seed, n_random=24):
    """First output index of every checked window (each R outputs long)."""
    starts = {0, max(0, M - 1 - R // 2), n - R}
    for thr in (1 << 28, 1 << 29, 1 << 30, 1 << 31, 1 << 32):
        if thr + R // 2 < n:
            starts.add(thr - R // 2)
    starts.add(((1 << 31) // L) * L - R // 2)  # the block that spans sample 2^31
    rng = np.random.Generator(np.random.PCG64(seed))
    starts.update(int(a) for a in rng.integers(M, n - R, n_random))
    return sorted(a for a in starts if 0 <= a <= n - R)


def _check_windows(xd, yd, h64, s0, M, real, starts, label):
    got, want, xs = [], [], []
    for a in starts:
        lo = max(0, a - (M - 1))
        xw = xd[lo: a + R].cpu().numpy()
        idx = np.arange(a - lo, a - lo + R)
        w = oracle.direct_at(xw, h64, s0 if lo == 0 else None, idx)
        want.append(w.real if real else w)
        got.append(yd[a: a + R].cpu().numpy())
        xs.append(xw)
    assert_parity(np.concatenate(got), np.concatenate(want), h64, np.concatenate(xs), label)


CASES = [  # workload (its filter and sample type), stream length
    ("C2", (1 << 31) + 3001),   # block kernel, complex, N = 4096
    ("C4", (1 << 31) + 1001),   # block kernel, real, N = 1024
    ("C3", (1 << 31) + 7),      # Tensor-Memory-resident kernel, N = 32768
    ("C5", (1 << 31) + 5),      # two-CTA kernel, N = 65536, H given
]


@pytest.mark.parametrize("name,n", CASES, ids=[c[0] for c in CASES])
def test_one_call_past_2_31_samples(name, n):
    import torch
    w = W.WORKLOADS[name]
    M, real = w.M, w.real
    plan = make_plan(w)
    h64 = W.oracle_h(w)
    s0 = (W.uniform_real(M - 1, 90).astype(np.float32) if real
          else W.complex_normal(M - 1, 90).astype(np.complex64))
    xd = W.device_signal(n, real, seed=91)
    yd = torch.empty_like(xd)
    st = torch.from_numpy(s0).cuda()
    plan.execute(xd, yd, st)
    torch.cuda.synchronize()
    plan.device_status()
    _check_windows(xd, yd, h64, s0, M, real, _window_starts(n, w.L, M, seed=92), f"{name} n={n}")
    assert torch.equal(st, xd[n - (M - 1):])
    plan.close()
    del xd, yd, st
    torch.cuda.empty_cache()


def test_batched_channels_past_2_31_samples():
    """Three channels of 2^30 + 77 real samples in one (channels, n) tensor: the last channel
    starts past sample 2^31 of the buffer."""
    import torch
    w = W.WORKLOADS["C4"]
    M, channels, n = w.M, 3, (1 << 30) + 77
    plan = make_plan(w)
    h64 = W.oracle_h(w)
    s0 = np.stack([W.uniform_real(M - 1, 100 + c).astype(np.float32) for c in range(channels)])
    xd = W.device_signal(channels * n, True, seed=93).view(channels, n)
    yd = torch.empty_like(xd)
    st = torch.from_numpy(s0).cuda()
    plan.execute_batched(xd, yd, st)
    torch.cuda.synchronize()
    plan.device_status()
    for c in range(channels):
        _check_windows(xd[c], yd[c], h64, s0[c], M, True, _window_starts(n, w.L, M, seed=94 + c, n_random=8),
                       f"channel {c}")
        assert torch.equal(st[c], xd[c, n - (M - 1):])
    plan.close()
    del xd, yd, st
    torch.cuda.empty_cache()


def test_channelizer_past_2_31_samples():
    """The 1024-channel bank (D = 512, Nh = 8192) over 2^31 + 3 D real samples: output vector
    m depends on x[m D + D - Nh .. m D + D - 1] only, so each checked vector is evaluated from
    a window that starts at a multiple of D."""
    import torch
    from frequency_domain_order_gb300 import fir_os
    c = W.CHANNELIZERS["P2big"]
    K, D, Nh = c.K, c.D, c.Nh
    n = (1 << 31) + 3 * D
    nout = n // D
    h = W.chan_prototype(c)
    h64 = h.astype(np.float32).astype(np.float64)
    s0 = W.uniform_real(Nh - 1, 95).astype(np.float32)
    plan = fir_os.ChanPlan(K, D, torch.from_numpy(h.astype(np.float32)).cuda(), real=True)
    xd = W.device_signal(n, True, seed=96)
    yd = torch.empty((nout, K), dtype=torch.complex64, device="cuda")
    st = torch.from_numpy(s0).cuda()
    plan.execute(xd, yd, st)
    torch.cuda.synchronize()
    ms = {0, 1, Nh // D - 1, Nh // D, nout - 2, nout - 1}
    for b in (1 << 19, 1 << 20, 1 << 21, 1 << 22):  # y element 2^31 .. 2^34 bytes, x index 2^31
        ms.update(m for m in (b - 2, b - 1, b, b + 1) if 0 <= m < nout)
    rng = np.random.Generator(np.random.PCG64(97))
    ms.update(int(m) for m in rng.integers(0, nout, 16))
    got, want, xs = [], [], []
    for m in sorted(ms):
        t_m = m * D + D - 1
        lo = max(0, (t_m - Nh + 1) // D * D)
        xw = xd[lo: t_m + 1].cpu().numpy()
        mw = (t_m - lo - (D - 1)) // D
        want.append(oracle.channelize_at(xw, h64, K, D, s0 if lo == 0 else np.zeros(Nh - 1, np.float32),
                                         np.array([mw]))[0])
        got.append(yd[m].cpu().numpy())
        xs.append(xw)
    got, want, xs = np.stack(got), np.stack(want), np.concatenate(xs)
    rel_tol, abs_tol = 1e-5, 1e-4 * np.abs(h64).sum() * np.abs(xs).max()
    d = got.astype(np.complex128) - want
    rel, mx = np.linalg.norm(d) / np.linalg.norm(want), np.abs(d).max()
    assert np.all(np.isfinite(got.view(np.float32)))
    assert rel <= rel_tol and mx <= abs_tol, f"rel-L2 {rel:.3g}, max-abs {mx:.3g} (bar {abs_tol:.3g})"
    assert torch.equal(st, xd[n - (Nh - 1):])
    plan.close()
    del xd, yd, st
    torch.cuda.empty_cache()
