"""Failure handling on a GPU, without a GPU fault: every failure here is made on the host.

* A kernel's bounded wait for a bulk copy (the overlap gather of step 3 of the claim in
  "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法", 主权项, staged into shared memory by the
  N <= 8192 kernels) is made to run out by setting the plan's wait limit to 0, which fails every
  such wait at once.  The kernel must report it (fir_os_device_status returns FIR_OS_E_DEVICE),
  let the copy that missed the wait land before it reuses the buffer, gather with plain loads
  instead and still produce the oracle's outputs; the next call with the default limit must be
  clean and give the same outputs bit for bit.
* Allocation failures are injected by fir_os_debug_fail_alloc, one allocation at a time: the
  failing call returns FIR_OS_E_NOMEM and the library's live-allocation count shows that it
  released everything it had allocated.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_parity, make_plan, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fo():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frequency_domain_order_gb300 import build, fir_os
    build.build()
    return fir_os


def _run(plan, x, s0, calls):
    import torch
    xd = to_dev(x)
    yd = torch.empty_like(xd)
    st = to_dev(s0.copy())
    off = 0
    for c in calls:
        plan.execute(xd[off: off + c], yd[off: off + c], st)
        off += c
    torch.cuda.synchronize()
    return yd.cpu().numpy(), st.cpu().numpy()


# workloads of the kernels that stage their windows by bulk copies: several units per group,
# windows at the state and at a ragged end, complex and packed real data, and a call of less
# than one wave (the variant with its tables in shared memory)
WAIT_CASES = [("C2", 300, 777, 1), ("C2", 40, 5, 3), ("C4", 3000, 606, 1), ("C4", 50, 11, 2),
              ("C1", 5000, 17, 1), ("C1", 20, 3, 1)]


@pytest.mark.parametrize("name,blocks,tail,calls", WAIT_CASES)
def test_wait_that_runs_out_falls_back_and_reports(fo, name, blocks, tail, calls):
    w = W.scaled(W.WORKLOADS[name], blocks, tail, calls)
    x = W.make_x(w)
    rng = np.random.Generator(np.random.PCG64(blocks + tail))
    s0 = (rng.standard_normal(w.M - 1).astype(np.float32) if w.real else
          (rng.standard_normal(w.M - 1) + 1j * rng.standard_normal(w.M - 1)).astype(np.complex64))
    plan = make_plan(w)
    plan.device_status()  # clean before
    plan.set_wait_limit(0)
    y0, st0 = _run(plan, x, s0, w.calls)
    with pytest.raises(fo.FirOsError) as err:
        plan.device_status()
    assert err.value.status == fo.E_DEVICE
    h = W.oracle_h(w)
    want, s_want = oracle.direct(x, h, s0)
    assert_parity(y0, want, h, x, f"{w.name} with every bulk-copy wait run out")
    assert np.array_equal(st0, (s_want.real if w.real else s_want).astype(st0.dtype))
    # the default limit again: a clean call with the same outputs
    plan.set_wait_limit(1_000_000_000)
    y1, st1 = _run(plan, x, s0, w.calls)
    plan.device_status()
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    assert np.array_equal(st0, st1)
    plan.close()


def test_wait_limit_argument_checks(fo):
    plan = make_plan(W.scaled(W.WORKLOADS["C1"], 4))
    for bad in (-1, 61 * 10**9):
        with pytest.raises(fo.FirOsError) as err:
            plan.set_wait_limit(bad)
        assert err.value.status == fo.E_INVAL
    plan.set_wait_limit(60 * 10**9)
    plan.close()


def _create_until_success(fo, make, what):
    """Inject a failure at allocation k = 1, 2, ... of make() until it succeeds; each failure
    must be FIR_OS_E_NOMEM with nothing left allocated.  Returns (the object, failures seen)."""
    base = fo.debug_live_allocs()
    for k in range(1, 40):
        fo.debug_fail_alloc(k)
        try:
            obj = make()
        except fo.FirOsError as e:
            fo.debug_fail_alloc(0)
            assert e.status == fo.E_NOMEM, (what, k, str(e))
            assert fo.debug_live_allocs() == base, (what, k)
            continue
        fo.debug_fail_alloc(0)
        return obj, k - 1
    raise AssertionError(f"{what}: never succeeded")


# (allocations plan_create makes, of which the plan keeps): the plan object, H, the error word
# and the pass twiddles; for N >= 16384 the split twiddles and H in c-major order; from taps the
# two float64 working buffers of step 1, freed before it returns
@pytest.mark.parametrize("name,expect,kept", [("C2", 6, 4), ("C3", 8, 6), ("C5", 6, 6), ("C4", 6, 4)])
def test_plan_create_allocation_failures(fo, name, expect, kept):
    import torch
    w = W.scaled(W.WORKLOADS[name], 3, 9)
    base = fo.debug_live_allocs()
    plan, failures = _create_until_success(fo, lambda: make_plan(w), name)
    # every allocation of plan_create was made to fail once
    assert failures == expect, (name, failures)
    assert fo.debug_live_allocs() == base + kept
    x = W.make_x(w)
    y, _ = _run(plan, x, np.zeros(w.M - 1, x.dtype), w.calls)
    plan.device_status()
    h = W.oracle_h(w)
    want, _ = oracle.direct(x, h)
    assert_parity(y, want, h, x, f"{name} after injected failures")
    plan.close()
    assert fo.debug_live_allocs() == base
    torch.cuda.synchronize()


def test_host_path_allocation_failures(fo):
    """The host-buffer call of a long-transform plan allocates its chunk buffers on first use;
    a failure there returns FIR_OS_E_NOMEM, frees what that call made, and a later call
    succeeds with the device path's outputs."""
    import torch
    w = W.scaled(W.WORKLOADS["C3"], 3, 9)
    base = fo.debug_live_allocs()
    plan = make_plan(w)
    with_plan = fo.debug_live_allocs()
    x = W.make_x(w)
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    sh = torch.zeros(w.M - 1, dtype=xh.dtype).pin_memory()
    for k in range(1, 6):  # two chunk buffers each for x and y, then the state
        fo.debug_fail_alloc(k)
        with pytest.raises(fo.FirOsError) as err:
            plan.execute_host(xh, yh, sh)
        fo.debug_fail_alloc(0)
        assert err.value.status == fo.E_NOMEM
        assert fo.debug_live_allocs() == with_plan, k
    sh.zero_()
    plan.execute_host(xh, yh, sh)
    y_dev, _ = _run(plan, x, np.zeros(w.M - 1, x.dtype), w.calls)
    assert np.array_equal(yh.numpy().view(np.uint32), y_dev.view(np.uint32))
    assert fo.debug_live_allocs() == with_plan + 5
    plan.close()
    assert fo.debug_live_allocs() == base


def test_channelizer_allocation_failures(fo):
    import torch
    c = W.CHANNELIZERS["P1"]
    h = torch.from_numpy(W.chan_prototype(c).astype(np.float32)).cuda()
    base = fo.debug_live_allocs()
    plan, failures = _create_until_success(fo, lambda: fo.ChanPlan(c.K, c.D, h, real=True), "P1")
    assert failures == 3  # the plan object, the pass twiddles, the padded prototype
    plan.close()
    assert fo.debug_live_allocs() == base
