"""Multi-process host logic on CPU (gloo, world size 2): the replica timing helpers of
bench.py (barrier, max over ranks) and the KV-sharded algebra of the path — each rank
attends over its own KV shard, the partial (out, lse) pairs are exchanged and merged
by LSE, and the result equals one pass over the whole KV (the ring / Helix exchange
step of the pages, done here with the oracle on CPU ranks)."""
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
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _replica_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import bench
        bench.barrier(world)
        v = bench.max_over_ranks(10.0 + rank, world)
        q.put((rank, v))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover
        q.put((rank, repr(e)))


def _kv_shard_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import oracle.mla_oracle as mo
        from mla_attention_gb300 import inputs as gen
        T, H, Tkv = 48, 4, 48
        P = gen.prefill_inputs(T=T, H=H, Tkv=Tkv, seed=17)
        shard = Tkv // world
        k0 = rank * shard
        o, l_ = mo.mla_prefill(P.q, P.kv[k0:k0 + shard], P.scale, causal=True, q_pos0=0, kv_pos0=k0)
        ot = torch.from_numpy(np.ascontiguousarray(o))
        lt = torch.from_numpy(np.ascontiguousarray(l_))
        og = [torch.empty_like(ot) for _ in range(world)]
        lg = [torch.empty_like(lt) for _ in range(world)]
        dist.all_gather(og, ot)
        dist.all_gather(lg, lt)
        mo_, ml_ = og[0].numpy(), lg[0].numpy()
        for r in range(1, world):
            mo_, ml_T = mo.merge(mo_, ml_.T, og[r].numpy(), lg[r].numpy().T)
            ml_ = ml_T.T
        ref_o, ref_l = mo.mla_prefill(P.q, P.kv, P.scale, causal=True)
        err_o = float(np.abs(mo_ - ref_o).max())
        fin = np.isfinite(ref_l)
        err_l = float(np.abs(ml_[fin] - ref_l[fin]).max())
        q.put((rank, (err_o, err_l, bool((np.isneginf(ml_) == np.isneginf(ref_l)).all()))))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover
        q.put((rank, repr(e)))


def _run(worker, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    return res


def test_replica_barrier_and_max_over_ranks():
    res = _run(_replica_worker)
    assert res == {0: 11.0, 1: 11.0}, res


def test_kv_sharded_partials_merge_to_one_pass():
    res = _run(_kv_shard_worker)
    for rank, v in res.items():
        assert not isinstance(v, str), v
        err_o, err_l, pattern = v
        assert err_o < 1e-12 and err_l < 1e-12 and pattern, (rank, v)
