"""Sharding one stream into independently filtered pieces (frequency_domain_order_gb300/shard.py).

A shard's call gets the M-1 samples in front of it (its halo) as its state; with shard starts on
the transform span (L, or 2L for real data) the shards' outputs concatenate to one call's output
and the last shard's state is the stream's S0'.  Checked with the float64 oracle on the CPU (one
process, and two gloo ranks launched like the benchmark), and on the GPU in test_gpu_parity.py.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads as W
from frequency_domain_order_gb300.shard import halo, shard_ranges, shard_states

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("n,L,parts,real", [
    (12352, 193, 2, False), (12352, 193, 3, False), (12352, 193, 64, False), (12352, 193, 100, False),
    (1 << 20, 770, 4, True), (1000, 770, 2, True), (0, 5, 3, False), (7, 1, 7, False), (6176, 193, 1, False),
])
def test_ranges_cover_contiguous_aligned(n, L, parts, real):
    r = shard_ranges(n, L, parts, real)
    span = L * (2 if real else 1)
    assert len(r) == parts
    assert r[0][0] == 0 and r[-1][1] == n
    for (a, b), (c, _) in zip(r, r[1:]):
        assert b == c and a <= b
    for a, _ in r:
        assert a % span == 0
    whole = [(b - a) // span for a, b in r[:-1]] + [(r[-1][1] - r[-1][0]) // span]
    assert max(whole) - min(whole) <= 1  # whole spans dealt out evenly


def test_ranges_reject_bad_arguments():
    for args in [(-1, 5, 2), (10, 0, 2), (10, 5, 0)]:
        with pytest.raises(ValueError):
            shard_ranges(*args)


def test_halo_takes_state_then_stream():
    x = np.arange(10, 20, dtype=np.float32)
    s0 = np.arange(1, 5, dtype=np.float32)  # M - 1 = 4, newest last
    assert halo(x, s0, 0, 5).tolist() == [1, 2, 3, 4]
    assert halo(x, s0, 2, 5).tolist() == [3, 4, 10, 11]
    assert halo(x, s0, 4, 5).tolist() == [10, 11, 12, 13]
    assert halo(x, s0, 7, 5).tolist() == [13, 14, 15, 16]
    assert halo(x, s0, 3, 1).tolist() == []


@pytest.mark.parametrize("name,parts", [("C1", 2), ("C1", 5), ("C4", 3)])
def test_sharded_oracle_equals_one_call(name, parts):
    w = W.WORKLOADS[name]
    if name == "C4":
        w = W.scaled(w, 9, 333)
    x, h = W.make_x(w), W.oracle_h(w)
    s0 = W.make_x(W.scaled(w, 1))[: w.M - 1]  # a nonzero S0, so shard 0's halo is checked too
    ranges = shard_ranges(len(x), w.L, parts, real=w.real)
    states = shard_states(x, s0, ranges, w.M)
    outs = [oracle.direct(x[a:b], h, st) for (a, b), st in zip(ranges, states)]
    y1, s1 = oracle.direct(x, h, s0)
    assert np.array_equal(np.concatenate([y for y, _ in outs]), y1)
    assert np.array_equal(outs[-1][1], s1)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_filter_one_stream(tmp_path):
    out = tmp_path / "result.json"
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}",
           os.path.join(ROOT, "tests", "shard_worker.py"), str(out)]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    v = json.loads(out.read_text())
    for name in ("C1", "C4"):
        assert v[name]["outputs_equal"], v[name]
        assert v[name]["state_equal"], v[name]
        assert v[name]["ranges"][0][0] == 0
    assert v["reduce_max"] == 2.0
