"""Helpers for the GPU parity tests: run the CUDA path through the binding, compare with the
oracle under the parity bar (relative L2 error <= 1e-5 and max abs error <=
1e-4 * ||h||_1 * max|x|, measured in float64)."""
import numpy as np

import workloads as W


def torch_mod():
    import torch
    return torch


def to_dev(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def make_plan(w: W.Workload):
    from frequency_domain_order_gb300 import fir_os
    if w.coef == "freq":
        coef = to_dev(W.make_H_given(w))
        kind = fir_os.COEF_FREQ
    else:
        coef = to_dev(W.make_h_device(w))
        kind = fir_os.COEF_TIME
    return fir_os.Plan(w.M, w.N, coef, real=w.real, coef_kind=kind)


def run_calls(plan, x: np.ndarray, calls, state0=None):
    """Filter x on the GPU as consecutive calls with the state carried; returns (y, state)
    as numpy arrays."""
    torch = torch_mod()
    xd = to_dev(x)
    yd = torch.empty_like(xd)
    st = (to_dev(state0) if state0 is not None
          else torch.zeros(max(plan.M - 1, 0), dtype=xd.dtype, device="cuda"))
    off = 0
    for c in calls:
        plan.execute(xd[off: off + c], yd[off: off + c], st if plan.M > 1 else None)
        off += c
    assert off == x.size
    torch.cuda.synchronize()
    plan.device_status()
    return yd.cpu().numpy(), st.cpu().numpy()


def run_device(plan, xd, calls, st=None):
    """Same, with the input already on the device; returns the device output tensor."""
    torch = torch_mod()
    yd = torch.empty_like(xd)
    if st is None:
        st = torch.zeros(max(plan.M - 1, 0), dtype=xd.dtype, device="cuda")
    off = 0
    for c in calls:
        plan.execute(xd[off: off + c], yd[off: off + c], st if plan.M > 1 else None)
        off += c
    torch.cuda.synchronize()
    plan.device_status()
    return yd, st


def assert_parity(got, want, h, x, label=""):
    rel_tol, abs_tol = W.tolerance(h, x)
    rel, mx = W.errors(got, want)
    assert np.all(np.isfinite(np.asarray(got).view(np.float32))), f"{label}: non-finite output"
    assert rel <= rel_tol and mx <= abs_tol, (
        f"{label}: rel-L2 {rel:.3g} (bar {rel_tol:g}), max-abs {mx:.3g} (bar {abs_tol:.3g})")
    return rel, mx
