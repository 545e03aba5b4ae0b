"""The tensor-core DFT engine (fir_os_plan_set_dft_engine, FIR_OS_DFT_TENSOR) against the oracle.

With it every radix-16 pass of the 4096-point transforms (step 4 of the claim in
"一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法", 主权项) computes its 16-point DFTs as
tcgen05.mma matrix products on split TF32 operands: the whole block transform at N = 4096, and
the 4096-point sub-transforms of the N = 16384 / 32768 (one SM) and N = 65536 (two-CTA cluster)
kernels.  The outputs must meet the same parity bar as the float32 engine (relative L2 error
<= 1e-5, max abs error <= 1e-4 * ||h||_1 * max|x|, measured in float64): whole streams with
ragged tails, several calls with the state carried, complex and packed real data, banks of
channels, the full C2, C3 and C5 workloads sampled, and M = 1 and M = N.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_parity, make_plan, run_calls, run_device, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fo():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build, fir_os
    build.build()
    return fir_os


def _tensor_plan(fo, w):
    plan = make_plan(w)
    plan.set_dft_engine(fo.DFT_TENSOR)
    return plan


@pytest.mark.parametrize("real", [False, True])
@pytest.mark.parametrize("blocks,tail,calls", [(1, 0, 1), (7, 1000, 1), (600, 333, 3), (3000, 5, 1)])
def test_tensor_engine_against_oracle(fo, real, blocks, tail, calls):
    base = W.WORKLOADS["C2"]
    if real:  # C2's filter on real data
        base = W.Workload("C2real", True, base.M, base.N, base.calls, 11, "time", base.h_kind, base.h_args)
    w = W.scaled(base, blocks, tail, calls)
    x = W.make_x(w)
    h = W.oracle_h(w)
    plan = _tensor_plan(fo, w)
    y, st = run_calls(plan, x, w.calls)
    if w.n <= 400_000:
        want, s_want = oracle.direct(x, h)
        assert_parity(y, want, h, x, f"{w.name} tensor engine")
    else:
        idx = W.sample_indices(w.n, w.L, seed=blocks, n_random=1 << 14)
        want = oracle.direct_at(x, h, None, idx)
        assert_parity(y[idx], want, h, x, f"{w.name} tensor engine, sampled")
        s_want = oracle.state_next(x, None, w.M)
    assert np.array_equal(st, (s_want.real if real else s_want).astype(st.dtype))
    plan.close()


@pytest.mark.parametrize("M", [1, 4096, 2049])
def test_tensor_engine_extreme_taps(fo, M):
    rng = np.random.Generator(np.random.PCG64(M))
    N = 4096
    n = 5 * (N - M + 1) + 77
    x = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
    h = ((rng.standard_normal(M) + 1j * rng.standard_normal(M)) / np.sqrt(M)).astype(np.complex64)
    s0 = (rng.standard_normal(M - 1) + 1j * rng.standard_normal(M - 1)).astype(np.complex64)
    plan = fo.Plan(M, N, to_dev(h))
    plan.set_dft_engine(fo.DFT_TENSOR)
    y, st = run_calls(plan, x, (n,), s0 if M > 1 else None)
    want, s_want = oracle.direct(x, h.astype(np.complex128), s0 if M > 1 else None)
    assert_parity(y, want, h, x, f"M={M} tensor engine")
    if M > 1:
        assert np.array_equal(st, s_want.astype(np.complex64))
    plan.close()


def test_tensor_engine_full_c2_sampled_and_close_to_fp32(fo):
    import torch
    w = W.WORKLOADS["C2"]
    x = W.make_x(w)
    h = W.oracle_h(w)
    xd = to_dev(x)
    plan = make_plan(w)
    y32, _ = run_device(plan, xd, w.calls)
    plan.set_dft_engine(fo.DFT_TENSOR)
    ytc, _ = run_device(plan, xd, w.calls)
    idx = W.sample_indices(w.n, w.L, seed=5, n_random=1 << 15)
    want = oracle.direct_at(x, h, None, idx)
    got = ytc.cpu().numpy()
    assert_parity(got[idx], want, h, x, "C2 tensor engine, sampled")
    # the two engines agree to the parity bar with each other over every output
    assert_parity(got, y32.cpu().numpy(), h, x, "tensor vs float32 engine")
    # and switching back gives the float32 engine's outputs bit for bit
    plan.set_dft_engine(fo.DFT_FP32)
    yb, _ = run_device(plan, xd, w.calls)
    assert torch.equal(yb.view(torch.int32), y32.view(torch.int32))
    plan.close()


def test_tensor_engine_sizes(fo):
    """Only N = 4096 and N >= 16384 have a tensor-core variant; the others refuse it."""
    for name in ("C1", "C4"):
        plan = make_plan(W.scaled(W.WORKLOADS[name], 2))
        with pytest.raises(fo.FirOsError) as err:
            plan.set_dft_engine(fo.DFT_TENSOR)
        assert err.value.status == fo.E_UNSUPPORTED
        with pytest.raises(fo.FirOsError) as err:
            plan.set_dft_engine(7)
        assert err.value.status == fo.E_INVAL
        plan.close()


def test_tensor_engine_with_the_wait_fallback(fo):
    """The zero wait limit (every bulk-copy wait runs out) with the tensor engine: the plain-load
    fallback gathers into the window the tiles overlap; outputs still meet the bar."""
    w = W.scaled(W.WORKLOADS["C2"], 300, 17)
    x = W.make_x(w)
    h = W.oracle_h(w)
    plan = _tensor_plan(fo, w)
    plan.set_wait_limit(0)
    xd = to_dev(x)
    import torch
    yd = torch.empty_like(xd)
    st = torch.zeros(w.M - 1, dtype=xd.dtype, device="cuda")
    plan.execute(xd, yd, st)
    torch.cuda.synchronize()
    with pytest.raises(fo.FirOsError) as err:
        plan.device_status()
    assert err.value.status == fo.E_DEVICE
    want, _ = oracle.direct(x, h)
    assert_parity(yd.cpu().numpy(), want, h, x, "tensor engine, fallback gathers")
    plan.close()


def test_tensor_engine_batched_channels(fo):
    """A bank of channels in one batched call with the tensor engine: every channel meets the bar
    against the oracle, with its own state carried over two calls."""
    import torch
    base = W.WORKLOADS["C2"]
    w = W.scaled(base, 9, 123)
    channels = 5
    xs = [W.make_x(W.dataclasses.replace(w, x_seed=w.x_seed + 1000 * c)) for c in range(channels)]
    h = W.oracle_h(w)
    plan = _tensor_plan(fo, w)
    xd = torch.stack([to_dev(x) for x in xs])
    yd = torch.empty_like(xd)
    st = torch.zeros((channels, w.M - 1), dtype=xd.dtype, device="cuda")
    half = (w.n // 2) // w.L * w.L
    plan.execute_batched(xd[:, :half], yd[:, :half], st)
    plan.execute_batched(xd[:, half:], yd[:, half:], st)
    torch.cuda.synchronize()
    plan.device_status()
    y = yd.cpu().numpy()
    for c in range(channels):
        want, s_want = oracle.direct(xs[c], h)
        assert_parity(y[c], want, h, xs[c], f"tensor engine, channel {c}")
        assert np.array_equal(st[c].cpu().numpy(), s_want.astype(np.complex64))
    plan.close()


@pytest.mark.parametrize("name,blocks", [("C2", 40), ("C3", 3), ("C5", 3)])
def test_tensor_engine_host_buffers(fo, name, blocks):
    """The host-buffer entry point with the tensor engine (N = 4096: the kernel reads and writes
    page-locked memory in place, gathering every window with plain loads; N >= 16384: the chunked
    copy pipeline) equals the device-buffer call bit for bit and meets the bar."""
    import torch
    w = W.scaled(W.WORKLOADS[name], blocks, 999)
    x = W.make_x(w)
    plan = _tensor_plan(fo, w)
    y_dev, s_dev = run_calls(plan, x, w.calls)
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    sh = torch.zeros(w.M - 1, dtype=xh.dtype).pin_memory()
    plan.execute_host(xh, yh, sh)
    plan.device_status()
    assert np.array_equal(yh.numpy().view(np.uint32), y_dev.view(np.uint32))
    assert np.array_equal(sh.numpy(), s_dev)
    h = W.oracle_h(w)
    if w.n * w.M <= 3e8:
        want, _ = oracle.direct(x, h)
        assert_parity(yh.numpy(), want, h, x, f"{name} tensor engine, host buffers")
    else:
        idx = W.sample_indices(w.n, w.L, seed=3, n_random=1 << 12, whole_blocks=[0])
        want = oracle.direct_at(x, h, None, idx)
        assert_parity(yh.numpy()[idx], want, h, x, f"{name} tensor engine, host buffers, sampled")
    plan.close()


# the resident (N = 16384, 32768) and two-CTA (N = 65536) kernels: C3's and C5's filters, and the
# same sizes with real data and with other tap counts
LARGE = [("C3", False, None, None), ("C5", False, None, None), ("C3", True, None, None), ("C5", True, None, None),
         ("N16384", False, 16384, 4097), ("N16384", True, 16384, 8193), ("N65536", False, 65536, 1)]


def _large_workload(name, real, N, M):
    if N is None:
        base = W.WORKLOADS[name]
        if real:  # the workload's sizes on real data, with real taps
            base = W.Workload(name + "real", True, base.M, base.N, base.calls, 13, "time", "hamming_lowpass", (0.2,))
        return base
    if M == 1:
        return W.Workload(name, real, M, N, (1,), 17, "time", "complex_normal", (), h_seed=21)
    return W.Workload(name, real, M, N, (1,), 17, "time", "hamming_lowpass", (0.25,))


@pytest.mark.parametrize("name,real,N,M", LARGE)
@pytest.mark.parametrize("blocks,tail,calls", [(1, 0, 1), (5, 777, 3)])
def test_tensor_engine_large_transforms(fo, name, real, N, M, blocks, tail, calls):
    w = W.scaled(_large_workload(name, real, N, M), blocks, tail, calls)
    x = W.make_x(w)
    h = W.oracle_h(w)
    plan = _tensor_plan(fo, w)
    y, st = run_calls(plan, x, w.calls)
    plan.device_status()
    if w.n * w.M <= 3e8:
        want, s_want = oracle.direct(x, h)
        assert_parity(y, want, h, x, f"{w.name} tensor engine")
    else:
        idx = W.sample_indices(w.n, w.L, seed=blocks, n_random=1 << 12, whole_blocks=[0])
        want = oracle.direct_at(x, h, None, idx)
        assert_parity(y[idx], want, h, x, f"{w.name} tensor engine, sampled")
        s_want = oracle.state_next(x, None, w.M)
    if w.M > 1:
        assert np.array_equal(st, (s_want.real if real else s_want).astype(st.dtype))
    plan.close()


@pytest.mark.parametrize("name", ["C3", "C5"])
def test_tensor_engine_full_size_sampled(fo, name):
    """The full C3 / C5 call with the tensor engine, sampled against the oracle, and within the
    bar of the float32 engine over every output."""
    w = W.WORKLOADS[name]
    x = W.make_x(w)
    h = W.oracle_h(w)
    xd = to_dev(x)
    plan = make_plan(w)
    y32, _ = run_device(plan, xd, w.calls)
    plan.set_dft_engine(fo.DFT_TENSOR)
    ytc, _ = run_device(plan, xd, w.calls)
    plan.device_status()
    idx = W.sample_indices(w.n, w.L, seed=7, n_random=1 << 13, whole_blocks=[0, w.n // w.L - 1])
    want = oracle.direct_at(x, h, None, idx)
    got = ytc.cpu().numpy()
    assert_parity(got[idx], want, h, x, f"{name} tensor engine, sampled")
    assert_parity(got, y32.cpu().numpy(), h, x, f"{name}: tensor vs float32 engine")
    plan.close()


@pytest.mark.parametrize("name", ["C3", "C5"])
def test_tensor_engine_large_batched(fo, name):
    """A bank of three channels through the multi-channel tensor-core variants, two calls."""
    import torch
    w = W.scaled(W.WORKLOADS[name], 3, 4321)
    channels = 3
    xs = [W.make_x(W.dataclasses.replace(w, x_seed=w.x_seed + 1000 * c)) for c in range(channels)]
    h = W.oracle_h(w)
    plan = _tensor_plan(fo, w)
    xd = torch.stack([to_dev(x) for x in xs])
    yd = torch.empty_like(xd)
    st = torch.zeros((channels, w.M - 1), dtype=xd.dtype, device="cuda")
    half = w.L + 1000
    plan.execute_batched(xd[:, :half], yd[:, :half], st)
    plan.execute_batched(xd[:, half:], yd[:, half:], st)
    torch.cuda.synchronize()
    plan.device_status()
    y = yd.cpu().numpy()
    for c in range(channels):
        idx = W.sample_indices(w.n, w.L, seed=c, n_random=1 << 12, whole_blocks=[0])
        want = oracle.direct_at(xs[c], h, None, idx)
        assert_parity(y[c][idx], want, h, xs[c], f"{name} tensor engine, channel {c}")
        s_want = oracle.state_next(xs[c], None, w.M)
        assert np.array_equal(st[c].cpu().numpy(), s_want.astype(np.complex64))
    plan.close()
