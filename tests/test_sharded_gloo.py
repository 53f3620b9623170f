"""The vocabulary-sharded top-16 exchange on CPU: two and three gloo ranks on
127.0.0.1, each holding one slice of every row.  The GPU partial and merge are
replaced by the oracle's (same signatures), so this checks the host side --
the slice bounds, the one all-gather and its rank order -- against the
oracle's whole-row top-16.  The GPU kernels themselves are checked against
the oracle in tests/test_gpu_shard.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fns():
    import oracle

    def shard_fn(z, off, V_total, params=None, rows_per_param=1):
        i, zz, m, s = oracle.topk16_shard(z, off, V_total, params=params, rows_per_param=rows_per_param)
        return torch.from_numpy(i), torch.from_numpy(zz), torch.from_numpy(m), torch.from_numpy(s)

    def merge_fn(pi, pz, pm, ps, V_total, params=None, rows_per_param=1):
        i, U, lse, _ = oracle.topk16_merge(pi.numpy(), pz.numpy(), pm.numpy(), ps.numpy(), V_total,
                                           params=params, rows_per_param=rows_per_param)
        return i, U, lse

    return shard_fn, merge_fn


def _rows(seed):
    from dflash_draft_selection_gb300 import synth
    g = torch.Generator().manual_seed(seed)
    z = (torch.randn(6, 5003, generator=g) * 2).bfloat16()
    z[0, 4000] = z[0, 17] = z[0].max() + 1     # a tie of the maximum across two slices
    params = synth.make_params(3, [0.0, 1.0, 0.7], [0, 20, 0], [1.0, 0.95, 1.0])
    return z, params


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    from dflash_draft_selection_gb300 import sharded
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        z, params = _rows(world)
        lo, hi = sharded.slice_bounds(z.shape[1], world, rank)
        shard_fn, merge_fn = _oracle_fns()
        idx, U, lse = sharded.sharded_topk16(z[:, lo:hi].contiguous(), lo, z.shape[1], params=params,
                                             rows_per_param=2, shard_fn=shard_fn, merge_fn=merge_fn)
        out[rank] = (idx.tolist(), U.tolist(), lse.tolist(), (lo, hi))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_agree_with_the_whole_row(ref, world):
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    bounds = [res[r][3] for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == 5003
    assert all(bounds[r][1] == bounds[r + 1][0] for r in range(world - 1))
    z, params = _rows(world)
    w_idx, w_U, w_lse, _ = ref.topk16(z, params=params, rows_per_param=2)
    for r in range(world):
        idx, U, lse, _ = res[r]
        np.testing.assert_array_equal(np.array(idx), w_idx)
        np.testing.assert_allclose(np.array(U), w_U, rtol=0, atol=1e-12)
        np.testing.assert_allclose(np.array(lse), w_lse, rtol=0, atol=1e-12)
    assert w_idx[0, 0] == 17 and w_idx[0, 1] == 4000
