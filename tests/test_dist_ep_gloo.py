"""Expert parallelism on CPU: two gloo ranks, each holding half of the experts and its own tokens,
exchange rows with all_to_all and must produce exactly the layer output of their tokens."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle
from sparse_mixture_experts_70_b300 import ep
from sparse_mixture_experts_70_b300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
from ep_worker import CASES  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(case: str, world: int = 2) -> list[dict]:
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE=str(world), LOCAL_RANK=str(r), OMP_NUM_THREADS="1")
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, "ep_worker.py"), case],
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
    return sorted(outs, key=lambda o: o["rank"])


def test_expert_ranges_cover_every_expert_once():
    for E in (1, 2, 3, 5, 8, 128, 257):
        for world in (1, 2, 3, 4, 8):
            if world > E:
                continue
            r = [ep.expert_range(q, world, E) for q in range(world)]
            assert r[0][0] == 0 and r[-1][1] == E
            assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
            sizes = [hi - lo for lo, hi in r]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def test_send_splits_and_single_rank_exchange():
    """Rows sent per owner are the sums of the owner's block of counts; with one process the
    count exchange returns this rank's block unchanged."""
    import torch
    counts = torch.tensor([5, 0, 3, 7, 1], dtype=torch.int32)
    assert ep.send_splits(counts, 2) == [8, 8]        # experts 0-2 | 3-4
    assert ep.send_splits(counts, 3) == [5, 10, 1]    # 0-1 | 2-3 | 4
    assert ep.send_splits(counts, 1) == [16]
    got = ep.exchange_counts(counts, 1)
    assert got.shape == (1, 5) and got.tolist() == [[5, 0, 3, 7, 1]]


@pytest.mark.parametrize("case", list(CASES))
def test_two_ranks_match_the_layer_on_their_tokens(case):
    w, _ = CASES[case]
    inputs = wl.generate(w)
    outs = _run(case)
    # every rank runs the layer on its own tokens: its reference is the oracle layer over exactly
    # those tokens (with a capacity, the capacity of that rank's batch)
    per_rank_counts = []
    for o in outs:
        lo_t, hi_t = o["tokens"]
        mine = w.with_(T=hi_t - lo_t)
        sub = dict(inputs, h=inputs["h"][lo_t:hi_t].contiguous())
        ref = oracle.reference(mine, sub)
        y = np.asarray(o["y"], dtype=np.float64).reshape(hi_t - lo_t, w.d)
        np.testing.assert_allclose(y, ref["y"], rtol=1e-12, atol=1e-12)
        assert o["counts"] == ref["counts"].tolist()
        per_rank_counts.append(ref["offsets"][1:] - ref["offsets"][:-1])
    # the rows a rank received are, per source and local expert, the rows the source kept for it
    for o in outs:
        lo, hi = o["experts"]
        assert o["recv_counts"] == [c[lo:hi].tolist() for c in per_rank_counts]
    # the reduced z-loss is the whole batch's; so is the auxiliary value without a capacity
    full = oracle.route(w, inputs)
    for o in outs:
        assert o["zloss"] == pytest.approx(full["zloss"], rel=1e-12)
        if w.capacity_factor == 0:
            assert o["aux"] == pytest.approx(full["aux"], rel=1e-12)
