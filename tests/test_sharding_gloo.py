"""Row sharding across ranks, world size 2, gloo on the CPU.

The host logic of nvfp4_block_quantization_quantize_gb300.sharding (shard
boundaries, row_offset, the one all-reduce MAX of the tensor amax) runs
between two CPU processes; the per-shard quantization is done by the oracle
standing in for the GPU library, and the gathered shards must equal the
oracle's unsharded result byte for byte.
"""
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
    names = {"rtn": oracle.RTN, "sr": oracle.SR, "1x16": oracle.BLOCK_1X16, "16x16": oracle.BLOCK_16X16,
             "none": oracle.GAMAX_NONE, "tensor_given": oracle.GAMAX_TENSOR_GIVEN, "row": oracle.GAMAX_ROW,
             "mae": oracle.ERR_MAE, "mse": oracle.ERR_MSE}

    def quantize_fn(x, row_offset=0, gamax_mode="none", gamax=None, rounding="rtn", block="1x16",
                    err_mode=None, residual=None, **kw):
        g = None if gamax is None else gamax.numpy()
        res = None if residual is None else residual.numpy()      # shares memory: updated in place
        r = oracle.quantize(x.numpy(), row_offset=row_offset, gamax_mode=names[gamax_mode], gamax=g,
                            rounding=names[rounding], block=names[block], residual=res,
                            err_mode=names[err_mode] if err_mode else oracle.ERR_NONE, **kw)
        return {k: torch.from_numpy(v) for k, v in r.items() if v is not None}

    def amax_fn(x, residual=None):
        return torch.from_numpy(oracle.amax(x.numpy(), residual=None if residual is None else residual.numpy()))
    return quantize_fn, amax_fn


def _worker(rank, world, port, x, cases, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from nvfp4_block_quantization_quantize_gb300.sharding import shard_rows, sharded_quantize
    quantize_fn, amax_fn = _oracle_fns()
    results = []
    for kw in cases:
        kw = dict(kw)
        r0, r1 = shard_rows(x.shape[0], world, rank)
        res = None
        if kw.pop("ef", False):
            res = torch.from_numpy(_residual(x.shape)[r0:r1].copy())
            kw["residual"] = res
        out = sharded_quantize(torch.from_numpy(x[r0:r1].copy()), r0, quantize_fn=quantize_fn,
                               amax_fn=amax_fn, **kw)
        got = {k: v.numpy() for k, v in out.items()}
        if res is not None:
            got["residual"] = res.numpy()
        gathered = [None] * world
        dist.all_gather_object(gathered, got)
        results.append(gathered)
    if rank == 0:
        q.put(results)
    dist.barrier()
    dist.destroy_process_group()


def _residual(shape):
    return (np.random.default_rng(9).standard_normal(shape) * 0.5).astype(np.float32)


# "ef": each rank passes its rows of one residual; with a per-tensor scale the
# exchanged amax is that of x + residual, as the unsharded call takes it
CASES = [dict(rounding="sr", seed=5, step=2),
         dict(gamax_mode="tensor", rounding="sr", seed=3, step=4, ef=True),
         dict(gamax_mode="tensor", rounding="rtn", ef=True),
         dict(gamax_mode="tensor", err_mode="mse", scale_bound=256.0, block="16x16", colwise=True),
         dict(gamax_mode="tensor", rounding="rtn"),
         dict(gamax_mode="row", err_mode="mae", scale_bound=256.0)]


def test_row_shards_over_gloo_match_unsharded():
    import nvfp4_workloads as W
    import oracle
    x = W.matrix((96, 80), seed=21, outlier_frac=0.05, outlier_factor=40.0)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, x, CASES, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    quantize_fn, _ = _oracle_fns()
    for kw, gathered in zip(CASES, results):
        okw = {k: v for k, v in kw.items() if k not in ("gamax_mode", "ef")}
        res = torch.from_numpy(_residual(x.shape)) if kw.get("ef") else None
        if res is not None:
            okw["residual"] = res
        if kw.get("gamax_mode") == "tensor":      # the unsharded tensor's own amax (of x + residual)
            A = torch.from_numpy(oracle.amax(x, residual=None if res is None else res.numpy()))
            whole = quantize_fn(torch.from_numpy(x), gamax_mode="tensor_given", gamax=A, **okw)
            assert all(np.array_equal(g["gamax"], A.numpy()) for g in gathered)
        else:
            whole = quantize_fn(torch.from_numpy(x), gamax_mode=kw.get("gamax_mode", "none"), **okw)
        if res is not None:
            assert np.array_equal(np.concatenate([g["residual"] for g in gathered]), res.numpy())
        assert np.array_equal(np.concatenate([g["codes"] for g in gathered]), whole["codes"].numpy())
        assert np.array_equal(np.concatenate([g["scales"] for g in gathered]), whole["scales"].numpy())
        if kw.get("colwise"):
            assert np.array_equal(np.concatenate([g["codes_col"] for g in gathered], axis=1),
                                  whole["codes_col"].numpy())
            assert np.array_equal(np.concatenate([g["scales_col"] for g in gathered], axis=1),
                                  whole["scales_col"].numpy())


def test_shard_rows_partition():
    from nvfp4_block_quantization_quantize_gb300.sharding import shard_rows
    for M, world in ((96, 2), (160, 3), (16, 4), (4096, 8)):
        spans = [shard_rows(M, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == M
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        assert all(r0 % 16 == 0 for r0, _ in spans)
    with pytest.raises(ValueError):
        shard_rows(100, 2, 0)
