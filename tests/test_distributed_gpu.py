"""The sharded search with its default per-rank solver (the CUDA path) in a one-rank group."""
import os
import socket

import numpy as np
import pytest

import oracle
import qubo_instances as qi

pytestmark = pytest.mark.gpu


def test_solve_distributed_single_rank_uses_the_cuda_path():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import torch.distributed as dist
    from exact_qubo_exhaustive_gb300 import distributed as qd

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("GLOO_SOCKET_IFNAME", "lo")
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        for Q, k in ((qi.random_upper_int(24, -500, 500, 621), 6), (qi.random_symmetric_normal_f32(22, 622), 5)):
            e, x, t = qd.solve_distributed(Q, k)
            we, wx, wt = oracle.get().solve(Q)
            if Q.dtype == np.float32:
                assert abs(e - we) <= 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
                assert t == wt and (x == wx).all()  # the exact fp64 minimiser, lowest rank
            else:
                assert (e, t) == (we, wt) and (x == wx).all()
    finally:
        dist.destroy_process_group()
