"""The multi-process host path on CPU: two gloo ranks, each with half of a batch, reduce the
auxiliary value of the whole batch and the slowest rank's time."""
import json
import os
import socket
import subprocess
import sys

import pytest

import oracle
from sparse_mixture_experts_70_b300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reduce_aux_and_timing():
    world, port = 2, _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE=str(world), LOCAL_RANK=str(r), OMP_NUM_THREADS="1")
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, "dist_worker.py")],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    w = wl.small(T=96, d=32, f=64, E=6, k=2, router_bias_var=1.0, seed=41)
    ref = oracle.route(w, wl.generate_router_inputs(w))
    for o in outs:
        assert o["aux"] == pytest.approx(ref["aux"], rel=1e-12)
        assert o["zloss"] == pytest.approx(ref["zloss"], rel=1e-12)
        assert o["slowest"] == [2.0, 10.0]
        assert o["value"] == pytest.approx(48 * 2 / 2e-3)
    # a rank alone sees only its own half: its aux differs from the batch's
    half = w.with_(T=48)
    inp = wl.generate_router_inputs(w)
    inp["h"] = inp["h"][:48].contiguous()
    assert oracle.route(half, inp)["aux"] != pytest.approx(ref["aux"], rel=1e-6)
