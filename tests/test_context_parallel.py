"""Context parallelism, host side (CPU): several gloo ranks each run
ssd_forward_context_parallel on a slice of one sequence, with the per-rank
device steps replaced by the fp64 oracle (tests/_cp_worker.py).  The slices'
outputs and the last rank's final state must equal the single-sequence
oracle: the recurrence is linear in its initial state, so the two-pass
scheme is exact up to rounding."""
import socket

import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("bounds", [(0, 150, 400), (0, 64, 65, 300)])
def test_context_parallel_ranks_match_the_whole_sequence(tmp_path, bounds):
    import torch.multiprocessing as mp
    import _cp_worker
    wl = I.small_workload(batch=2, seqlen=bounds[-1], nheads=3, headdim=8, dstate=16, ngroups=1,
                          chunk=64, dtype="f32", init="normal", seed=41)
    fi = I.make_forward_inputs(wl)
    data = tmp_path / "data.npz"
    np.savez(data, x=fi.x, dt=fi.dt, A=fi.A, B=fi.B, C=fi.C, D=fi.D, init=fi.init,
             bounds=np.array(bounds))
    world = len(bounds) - 1
    prefix = str(tmp_path / "out")
    mp.start_processes(_cp_worker.run, args=(world, _free_port(), str(data), prefix),
                       nprocs=world, start_method="spawn")
    y_ref, fin_ref = oracle.ssd_scan(fi.x, fi.dt, fi.A, fi.B, fi.C, fi.D, fi.init)
    ys = [np.load(f"{prefix}{r}.npz") for r in range(world)]
    y = np.concatenate([o["y"] for o in ys], axis=1)
    assert oracle.rel_err(y, y_ref) < 1e-12
    assert oracle.rel_err(ys[-1]["fin"], fin_ref) < 1e-12
    # every rank's end state is the state after its slice
    for r in range(world - 1):
        _, fin_r = oracle.ssd_scan(fi.x[:, :bounds[r + 1]], fi.dt[:, :bounds[r + 1]], fi.A,
                                   fi.B[:, :bounds[r + 1]], fi.C[:, :bounds[r + 1]], fi.D, fi.init)
        assert oracle.rel_err(ys[r]["fin"], fin_r) < 1e-12
