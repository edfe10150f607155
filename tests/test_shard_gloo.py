"""Head sharding on CPU ranks (gloo, world size 2): each rank runs the oracle on its
slice of the heads; gathered, the slices equal the unsharded result bit for bit, and
the ranks' timing reduction takes the maximum.  No GPU."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from qkv_rope_kv_gb300 import shard


def test_shard_ranges_cover_rows_once():
    for nh, nkv, hd, world in ((40, 8, 128, 2), (40, 8, 128, 8), (28, 4, 128, 4), (14, 2, 64, 2)):
        R = (nh + 2 * nkv) * hd
        hits = np.zeros(R, int)
        for r in range(world):
            s = shard.head_shard(nh, nkv, hd, world, r)
            assert s.n_head * world == nh and s.n_head_kv * world == nkv
            for a, b in s.concat_rows:
                hits[a:b] += 1
        assert np.all(hits == 1)
    with pytest.raises(ValueError):
        shard.head_shard(28, 4, 128, 8, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import torch
    import oracle
    from qkv_rope_kv_gb300 import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    nh, nkv, hd, H, n_ctx, pos = 8, 4, 16, 96, 6, 5
    nqt, nkt = nh * hd, nkv * hd
    W = synth.weight_rows(0, 2, 0, nqt + 2 * nkt, H, "bf16")
    b = synth.bias(0, 2, nqt + 2 * nkt)
    x = synth.hidden(0, 2, pos, H)
    s = shard.head_shard(nh, nkv, hd, world, rank)
    rows = np.concatenate([np.arange(a, c) for a, c in s.concat_rows])
    kk = np.zeros((n_ctx, s.n_head_kv * hd), np.uint16)
    vv = np.zeros_like(kk)
    st, q, k, v = oracle.Oracle().decode(W[rows], x, b[rows], s.n_head, s.n_head_kv, hd, 1e6, 1.0, pos, kk, vv)
    local = torch.from_numpy(np.concatenate([q, k, v, kk.view(np.float16).astype(np.float32).ravel(),
                                             vv.view(np.float16).astype(np.float32).ravel()]))
    gathered = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(gathered, local)
    m = shard.max_over_ranks(float(rank + 1))
    if rank == 0:
        out.put((st, [g.numpy() for g in gathered], m))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_oracle_equals_unsharded():
    import oracle
    from qkv_rope_kv_gb300 import synth
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    st, gathered, m = out.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert st == 0 and m == float(world)
    nh, nkv, hd, H, n_ctx, pos = 8, 4, 16, 96, 6, 5
    nqt, nkt = nh * hd, nkv * hd
    W = synth.weight_rows(0, 2, 0, nqt + 2 * nkt, H, "bf16")
    b = synth.bias(0, 2, nqt + 2 * nkt)
    x = synth.hidden(0, 2, pos, H)
    kk = np.zeros((n_ctx, nkt), np.uint16)
    vv = np.zeros_like(kk)
    st, q, k, v = oracle.Oracle().decode(W, x, b, nh, nkv, hd, 1e6, 1.0, pos, kk, vv)
    for r in range(world):
        s = shard.head_shard(nh, nkv, hd, world, r)
        g = gathered[r]
        lq, lk = s.n_head * hd, s.n_head_kv * hd
        a, c = s.q_rows
        ka, kc = s.kv_rows
        assert np.array_equal(g[:lq].view(np.uint32), q[a:c].view(np.uint32))
        assert np.array_equal(g[lq:lq + lk].view(np.uint32), k[ka:kc].view(np.uint32))
        assert np.array_equal(g[lq + lk:lq + 2 * lk].view(np.uint32), v[ka:kc].view(np.uint32))
        off = lq + 2 * lk
        kreg = g[off:off + n_ctx * lk].reshape(n_ctx, lk)
        vreg = g[off + n_ctx * lk:].reshape(n_ctx, lk)
        assert np.array_equal(kreg, kk[:, ka:kc].view(np.float16).astype(np.float32))
        assert np.array_equal(vreg, vv[:, ka:kc].view(np.float16).astype(np.float32))
