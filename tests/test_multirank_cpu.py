"""World-size-2 checks of the multi-rank logic on CPU (gloo).

Rows shard across ranks with no exchange inside the norm; the two
cross-rank reductions a sharded user performs are a MAX of the delayed
scaling amax and a SUM of dgamma/dbeta.  Each rank runs the oracle on its
row shard; the combined results must equal the unsharded oracle.  The
benchmark's rank aggregation (max of per-rank time, rows summed over ranks)
is checked the same way.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
        w = WORKLOADS["rms_bwd_add_bf16_32768x12288"].with_shape(64, 256)
        inp = make_inputs(w, seed=0)                     # same full batch on every rank
        shard = slice(rank * 32, (rank + 1) * 32)        # 32-row shards
        z, _, rs = oracle.norm_fwd(inp["x"][shard], inp["gamma"], None, 1, False, w.eps)
        _, amax, _ = oracle.quant_delayed(z, 1.0)
        t = torch.tensor([float(amax)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        _, dg, _ = oracle.norm_bwd(inp["dz"][shard], inp["x"][shard], None,
                                   rs.astype(np.float32), inp["gamma"], None, 1, False)
        g = torch.from_numpy(dg)
        dist.all_reduce(g, op=dist.ReduceOp.SUM)
        # bench aggregation: per-rank elapsed -> max; rows summed over ranks
        el = torch.tensor([1.0 + rank], dtype=torch.float64)
        dist.all_reduce(el, op=dist.ReduceOp.MAX)
        if rank == 0:
            q.put((float(t.item()), g.numpy().copy(), float(el.item())))
    finally:
        dist.destroy_process_group()


def test_sharded_amax_and_dgamma_match_unsharded():
    import oracle
    from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    amax, dg, el = q.get()
    w = WORKLOADS["rms_bwd_add_bf16_32768x12288"].with_shape(64, 256)
    inp = make_inputs(w, seed=0)
    z, _, rs = oracle.norm_fwd(inp["x"], inp["gamma"], None, 1, False, w.eps)
    _, amax_ref, _ = oracle.quant_delayed(z, 1.0)
    assert amax == float(amax_ref)                      # max is exact
    _, dg_ref, _ = oracle.norm_bwd(inp["dz"], inp["x"], None, rs.astype(np.float32),
                                   inp["gamma"], None, 1, False)
    np.testing.assert_allclose(dg, dg_ref, rtol=1e-12, atol=1e-12)
    assert el == 2.0
