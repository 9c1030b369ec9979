"""The exchange of sequence-parallel attention on CPU ranks (gloo, world size 2 and 3).

Each rank holds one contiguous shard of the keys (uneven shards, one of them past the end of
a short sequence, so that some rows see none of its keys) and produces the state (m, l, u) of
every query row over it -- here with the float64 oracle's key_state, which stands in for the
GPU's attn_fwd_partial -- then online_softmax_fa2_gb300.seqpar.gather_states exchanges the
states and every rank merges them (the oracle's merge_states).  The result must equal the
oracle's attention over the whole key axis, with every empty row exactly (0, -inf): the merge
of the states of disjoint key sets is the state of their union ("How Does FlashAttention
Preserve Global Softmax Across Tiles?", sections 3 and 4)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

SHARDS = {2: [0, 23, 40], 3: [0, 9, 30, 40]}  # key ranges [c_r, c_r+1) of a 40-key axis


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    g = torch.Generator().manual_seed(5)
    B, Nq, Nk, H, dk, dv = 3, 17, 40, 2, 8, 6
    q = torch.randn(B, Nq, H, dk, generator=g)
    k = torch.randn(B, Nk, H, dk, generator=g)
    v = torch.randn(B, Nk, H, dv, generator=g)
    kv_lens = [40, 12, 0]  # sequence 1 ends inside shard 0 or 1; sequence 2 has no keys
    return q, k, v, kv_lens


def _worker(rank, world, port, causal, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    from online_softmax_fa2_gb300 import seqpar
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, kv_lens = _inputs()
        c = SHARDS[world]
        # this rank's shard: the state of every row over keys [c[rank], c[rank+1])
        part = torch.from_numpy(oracle.key_state(q, k, v, c[rank], c[rank + 1], kv_lens=kv_lens,
                                                 causal=causal))
        allp = seqpar.gather_states(part)                      # [R, B, H, Nq, 2 + dv]
        states = allp.permute(1, 2, 3, 0, 4).contiguous().numpy()  # [B, H, Nq, R, 2 + dv]
        o, lse = oracle.merge_states(states)
        queue.put((rank, o, lse, allp.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_gathered_shard_states_merge_to_whole_attention(world, causal):
    import oracle

    port = _free_port()
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, causal, queue)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        results = sorted((queue.get(timeout=600) for _ in range(world)), key=lambda t: t[0])
    finally:
        for p in procs:
            p.join(120)
    assert [p.exitcode for p in procs] == [0] * world
    q, k, v, kv_lens = _inputs()
    o_ref, lse_ref, _ = oracle.attn_fwd(q, k, v, kv_lens=kv_lens, causal=causal)  # [B, Nq, H, dv], [B, H, Nq]
    o_ref = np.transpose(o_ref, (0, 2, 1, 3))
    c = SHARDS[world]
    for rank, o, lse, allp in results:
        # every rank gathered the same states, in rank order
        assert np.array_equal(allp, results[0][3])
        for r in range(world):
            want = oracle.key_state(q, k, v, c[r], c[r + 1], kv_lens=kv_lens, causal=causal)
            assert np.array_equal(allp[r], want)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.all(lse[~fin] == -np.inf) and np.all(o[~fin] == 0.0)
        assert np.allclose(o[fin], o_ref[fin], atol=1e-12, rtol=1e-12)
        assert np.allclose(lse[fin], lse_ref[fin], atol=1e-12, rtol=1e-12)
