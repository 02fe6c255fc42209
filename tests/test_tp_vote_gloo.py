"""Head-sharded voting between CPU ranks (the tensor-parallel pattern for one
sequence): each of two gloo ranks holds half of the query heads, forms its
heads' softmax sum, and one all-reduce (sum) of the N-float vote gives every
rank the vote of all heads, hence the same deterministic selection. Checked
against the single-process oracle. TokenSelect deep notes, "Head soft vote"
(the vote is a sum over heads, so a sum of per-shard sums)."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, ws, port, logits, n, k, s, w, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank))
    import torch
    import torch.distributed as dist

    from oracle import tokenselect_oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    H = logits.shape[0]
    mine = logits[rank * H // ws:(rank + 1) * H // ws]      # this rank's query heads
    v = torch.from_numpy(O.soft_vote(mine))
    dist.all_reduce(v, op=dist.ReduceOp.SUM)                 # the one exchange: N floats
    idx, _ = O.select_topk(v.numpy(), n, k, s, w)
    q.put((rank, v.numpy(), idx))
    dist.destroy_process_group()


def test_two_ranks_holding_half_the_heads_select_what_one_process_selects():
    import workloads as W
    from oracle import tokenselect_oracle as O
    sp = W.spec(1, n0=(3001,), steps=1, k=256, n_local=64)
    wl = W.generate(sp, "cpu")
    n = int(wl.n0[0])
    q = O.as_f64(wl.q[0][0][0].float().numpy())
    pool = wl.k_pool[0].float().numpy()
    page_row = wl.page_table[0].numpy()
    logits = O.head_logits(q, pool, page_row, n)            # [H][n]
    want_v = O.soft_vote(logits)
    want, _ = O.select_topk(want_v, n, sp.k, sp.n_sink, sp.n_local)
    ws = 2
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, logits, n, sp.k, sp.n_sink, sp.n_local, qu))
             for r in range(ws)]
    for p in procs:
        p.start()
    got = [qu.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, v, idx in got:
        assert np.allclose(v, want_v, rtol=1e-12, atol=0.0), rank
        assert np.array_equal(idx, want), rank
    assert abs(want_v.sum() - sp.n_q_heads) < 1e-9      # the vote sums to H
