"""Multi-channel filtering (fir_os_execute_batched) through the C ABI.

Every channel of a batched call must equal fir_os_execute on that channel alone, bit for bit
(the same kernel filters the same blocks), for every kernel family: the block kernel (small
and 4096-point transforms, complex and real), the Tensor-Memory-resident kernel (32768) and
the two-CTA kernel (65536).  One channel of each case is also checked against the float64
oracle under the parity bar.  Rows are strided (padded) to check the stride arithmetic, and
each channel starts from its own nonzero state.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_parity, make_plan, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build
    build.build()


def _bank(w, channels, pad=37):
    """(x, state) for `channels` channels in padded rows: x (channels, n + pad) and
    state (channels, M - 1 + pad), each channel its own seeded data and nonzero S0."""
    xs = np.stack([W.make_x_shard(w, c) for c in range(channels)])
    src = W.scaled(w, (w.M - 1) // w.L + 1)  # a stream of at least M-1 samples
    s0 = np.stack([W.make_x_shard(src, 100 + c)[: w.M - 1] for c in range(channels)])
    xp = np.zeros((channels, w.n + pad), dtype=xs.dtype)
    xp[:, : w.n] = xs
    sp = np.zeros((channels, w.M - 1 + pad), dtype=xs.dtype)
    sp[:, : w.M - 1] = s0
    return xp, sp


@pytest.mark.parametrize("name,blocks,tail,channels", [
    ("C1", 9, 17, 5),        # N = 256: eight-group block kernel
    ("C2", 11, 1001, 4),     # N = 4096 complex
    ("C4", 13, 123, 6),      # N = 1024 real pairs
    ("C3", 3, 12345, 3),     # N = 32768: Tensor-Memory-resident kernel
    ("C5", 2, 777, 2),       # N = 65536: two-CTA kernel
])
def test_batched_equals_single_channel_calls(name, blocks, tail, channels):
    torch = pytest.importorskip("torch")
    w = W.scaled(W.WORKLOADS[name], blocks, tail)
    plan = make_plan(w)
    xp, sp = _bank(w, channels)
    xd = to_dev(xp)
    yd = torch.full_like(xd, float("nan"))
    sd = to_dev(sp)
    n = w.n
    for _ in range(2):  # the second call continues every channel from its carried state
        plan.execute_batched(xd[:, :n], yd[:, :n], sd[:, : w.M - 1])
        torch.cuda.synchronize()
        plan.device_status()
        y_b = yd[:, :n].cpu().numpy()
        s_b = sd[:, : w.M - 1].cpu().numpy()
        assert np.isnan(yd[:, n:].cpu().numpy()).all()  # padding untouched
        for c in range(channels):
            x1 = to_dev(xp[c, :n])
            y1 = torch.empty_like(x1)
            s1 = to_dev(sp[c, : w.M - 1])
            plan.execute(x1, y1, s1)
            torch.cuda.synchronize()
            assert np.array_equal(y_b[c].view(np.uint32), y1.cpu().numpy().view(np.uint32)), f"channel {c}"
            assert np.array_equal(s_b[c], s1.cpu().numpy()), f"state of channel {c}"
        sp[:, : w.M - 1] = s_b  # the per-channel reference continues from the same state
    # one channel against the oracle, first call only (fresh data, same initial state)
    c = channels - 1
    xp0, sp0 = _bank(w, channels)
    h = W.oracle_h(w)
    if n * w.M <= 3e8:
        want, _ = oracle.direct(xp0[c, :n], h, sp0[c, : w.M - 1])
        xd0 = to_dev(xp0)
        yd0 = torch.empty_like(xd0)
        sd0 = to_dev(sp0)
        plan.execute_batched(xd0[:, :n], yd0[:, :n], sd0[:, : w.M - 1])
        torch.cuda.synchronize()
        assert_parity(yd0[c, :n].cpu().numpy(), want, h, xp0[c, :n], f"{w.name} batched channel {c}")
    plan.close()


@pytest.mark.parametrize("case", ["block L < M-1", "resident n < M-1"])
def test_batched_state_kernel_path(case):
    """Where the block kernel cannot write S0' itself (L < M-1: several units read S0) or the
    resident kernel has n < M-1, the per-channel state kernel writes it."""
    import dataclasses
    torch = pytest.importorskip("torch")
    if case.startswith("block"):
        w = dataclasses.replace(W.WORKLOADS["C2"], M=3000).with_calls((5000,))
    else:
        w = W.WORKLOADS["C3"].with_calls((5000,))
    n = w.n
    plan = make_plan(w)
    assert plan.launches(n) == 2
    xp, sp = _bank(w, 3)
    xd, sd = to_dev(xp), to_dev(sp)
    yd = torch.empty_like(xd)
    plan.execute_batched(xd[:, :n], yd[:, :n], sd[:, : w.M - 1])
    torch.cuda.synchronize()
    for c in range(3):
        x1, s1 = to_dev(xp[c, :n]), to_dev(sp[c, : w.M - 1])
        y1 = torch.empty_like(x1)
        plan.execute(x1, y1, s1)
        torch.cuda.synchronize()
        assert np.array_equal(yd[c, :n].cpu().numpy().view(np.uint32), y1.cpu().numpy().view(np.uint32))
        assert np.array_equal(sd[c, : w.M - 1].cpu().numpy(), s1.cpu().numpy())
        # S0' = last M-1 samples of concat(S0, x)
        want = np.concatenate([sp[c, : w.M - 1], xp[c, :n]])[-(w.M - 1):]
        assert np.array_equal(s1.cpu().numpy(), want)
    plan.close()


def test_batched_full_size_bank_sampled():
    """The benchmark's C2x16 bank at full size: sampled outputs of two channels vs the oracle."""
    torch = pytest.importorskip("torch")
    w = W.WORKLOADS["C2x16"]
    plan = make_plan(w)
    x = W.make_x_channels(w)
    xd = to_dev(x)
    yd = torch.empty_like(xd)
    sd = torch.zeros((w.channels, w.M - 1), dtype=xd.dtype, device="cuda")
    plan.execute_batched(xd, yd, sd)
    torch.cuda.synchronize()
    plan.device_status()
    h = W.oracle_h(w)
    for c in (0, w.channels - 1):
        idx = W.sample_indices(w.n, w.L, seed=11 + c, n_random=1 << 12)
        want = oracle.direct_at(x[c], h, None, idx)
        assert_parity(yd[c].cpu().numpy()[idx], want, h, x[c], f"C2x16 channel {c} sampled")
        assert np.array_equal(sd[c].cpu().numpy(), x[c, -(w.M - 1):])
    plan.close()


def test_batched_argument_checks():
    torch = pytest.importorskip("torch")
    from frequency_domain_order_gb300 import fir_os
    w = W.scaled(W.WORKLOADS["C2"], 2, 0)
    plan = make_plan(w)
    L = fir_os.lib()
    x = torch.zeros((3, w.n), dtype=torch.complex64, device="cuda")
    y = torch.zeros_like(x)
    s = torch.zeros((3, w.M - 1), dtype=torch.complex64, device="cuda")
    h = plan._h
    ok = L.fir_os_execute_batched(h, x.data_ptr(), w.n, y.data_ptr(), w.n, s.data_ptr(), w.M - 1, w.n, 3, None)
    assert ok == 0
    torch.cuda.synchronize()
    bad = [
        (x.data_ptr(), w.n, y.data_ptr(), w.n, s.data_ptr(), w.M - 1, w.n, 0),          # channels 0
        (x.data_ptr(), w.n - 1, y.data_ptr(), w.n, s.data_ptr(), w.M - 1, w.n, 3),      # short x stride
        (x.data_ptr(), w.n, y.data_ptr(), w.n, s.data_ptr(), w.M - 2, w.n, 3),          # short state stride
        (x.data_ptr(), w.n, x.data_ptr() + 8 * w.n, w.n, s.data_ptr(), w.M - 1, w.n, 3),  # y inside x's extent
        (x.data_ptr(), w.n, y.data_ptr(), w.n, x.data_ptr(), w.M - 1, w.n, 3),          # state inside x
        (x.data_ptr(), w.n, y.data_ptr(), w.n, None, w.M - 1, w.n, 3),                  # no state, M > 1
    ]
    for a in bad:
        assert L.fir_os_execute_batched(h, *a, None) == fir_os.E_INVAL, a
    assert L.fir_os_execute_batched(h, x.data_ptr() + 4, w.n, y.data_ptr(), w.n, s.data_ptr(), w.M - 1, w.n,
                                    3, None) == fir_os.E_ALIGN
    plan.close()
