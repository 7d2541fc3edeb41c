"""Worker of the multi-process context-parallel test: one gloo rank running
ssd_forward_context_parallel on its slice, with the per-rank device steps
replaced by the fp64 oracle (test infrastructure: the exchange and state
composition logic is what is under test here)."""
import os

import numpy as np
import torch

import oracle


def oracle_ops():
    from state_space_sequence_05_b300.context_parallel import CPOps

    def forward(x, dt, A, B, C, D, chunk_size, init):
        y, fin = oracle.ssd_scan(x.numpy(), dt.numpy(), A.numpy(), B.numpy(), C.numpy(),
                                 None if D is None else D.numpy(),
                                 None if init is None else init.numpy())
        return torch.from_numpy(y), torch.from_numpy(fin)

    def states(x, dt, A, B, chunk_size):
        # the state a slice leaves from a zero state: the recurrence's final
        # state, whose value does not depend on C
        zeros = np.zeros(B.shape, dtype=B.numpy().dtype)
        _, fin = oracle.ssd_scan(x.numpy(), dt.numpy(), A.numpy(), B.numpy(), zeros, None, None)
        return torch.from_numpy(fin)

    def decay(dt, A):
        return dt.double().sum(dim=1) * A.double()

    def combine(a, S, init):
        R = S.shape[0]
        out = torch.zeros((R + 1,) + tuple(S.shape[1:]), dtype=torch.float64)
        if init is not None:
            out[0] = init
        for r in range(R):
            out[r + 1] = torch.exp(a[r])[:, :, None, None] * out[r] + S[r]
        return out

    return CPOps(forward, decay, combine, states)


def run(rank, world, port, data_path, out_prefix):
    import torch.distributed as dist
    from state_space_sequence_05_b300.context_parallel import ssd_forward_context_parallel
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = np.load(data_path)
        lo, hi = int(d["bounds"][rank]), int(d["bounds"][rank + 1])
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        y, fin = ssd_forward_context_parallel(
            t(d["x"][:, lo:hi]), t(d["dt"][:, lo:hi]), t(d["A"]), t(d["B"][:, lo:hi]),
            t(d["C"][:, lo:hi]), t(d["D"]), 64, t(d["init"]), ops=oracle_ops())
        np.savez(f"{out_prefix}{rank}.npz", y=y.numpy(), fin=fin.numpy())
    finally:
        dist.destroy_process_group()
