"""Chunk-wise prefill selection (ts_prefill_chunk) against the CPU oracle, through the C ABI.

A chunk's c queries are the first c queries of a workload's AR(1) trajectory
(consecutive queries are similar, as in a prefill); the chunk's own tokens are
the last c cached tokens. The GPU averages the queries, selects once from the
mean (the persistent kernel's score and selection), and runs the causal
attention of all c queries on the tensor cores. Checks: the index set against
the oracle's selection from the mean query (the same tie band and at-risk
margin as the decode tests), the mean query's votes, and every query's output
and lse against the oracle's causal sparse attention (2e-3 max-abs relative
per (query, head) row, lse within 1e-3), on the oracle's set or, where the
two sets differ inside the tie band, on the GPU's.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity import LSE_ABS, check_attention, check_topk_set, kv_flag, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(sp, c, check_every=1):
    T = tsl()
    wl = W.generate(sp, DEV)
    B, H, d = sp.batch, sp.n_q_heads, sp.head_dim
    ctx = T.Context(H, sp.n_kv_heads, d, kv_flag(T, sp), B, wl.page_table.shape[1], wl.num_pages,
                    page_size=sp.page_size)
    q = torch.stack([wl.q[i][0] for i in range(c)], dim=1).contiguous()          # [B][c][H][d]
    cap = sp.k + sp.n_sink + sp.n_local
    idx = torch.full((B, cap), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.full((B, c, H, d), float("nan"), device=DEV)
    lse = torch.full((B, c, H), float("nan"), device=DEV)
    vote = torch.zeros(B, ctx.max_tokens, device=DEV)
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
    seq = wl.seq_lens(0)
    ctx.prefill_chunk(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt, out, lse, vote=vote)
    assert ctx.status() == 0
    kp, vp, pt = W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0]), W.host_copy(wl.page_table)
    qh = W.host_copy(q)
    g_idx, g_cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    g_out, g_lse, g_vote = out.cpu().numpy(), lse.cpu().numpy(), vote.cpu().numpy()
    worst = 0.0
    for b in range(B):
        n = wl.n0[b]
        where = f"{sp.name} c={c} seq {b}"
        r = O.prefill_chunk(qh[b], kp, vp, pt[b], n, k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local)
        gi = g_idx[b, :g_cnt[b]]
        rel = np.abs(g_vote[b, :n] - r["vote"]) / r["vote"]
        assert float(rel.max()) <= 1e-4, f"{where}: mean-query vote rel err {rel.max():.2e}"
        check_topk_set(gi, r["idx"], r["vote"], n, sp.k, sp.n_sink, sp.n_local, where, gpu_vote=g_vote[b])
        same = np.array_equal(gi, r["idx"])
        for i in range(0, c, check_every):
            if same:
                ro, rl = r["out"][i], r["lse"][i]
            else:
                ro, rl = O.sparse_attention(qh[b, i], kp, vp, pt[b], gi[gi <= n - c + i])
            check_attention(g_out[b, i], g_lse[b, i], ro, rl, f"{where} query {i}")
            den = np.max(np.abs(ro), axis=1)
            worst = max(worst, float((np.max(np.abs(g_out[b, i] - ro), axis=1) / den).max()))
    print(f"{where}: worst attention rel err {worst:.2e}")
    ctx.close()
    return g_idx, g_cnt


@pytest.mark.parametrize("c", [1, 16, 100])
def test_prefill_llama_small(c):
    # 100 queries x 4 heads = 400 rows: three full query tiles and a ragged one
    sp = W.spec(1, n0=(5003,), steps=c, k=512, n_local=128)
    _run(sp, c)


def test_prefill_qwen_batched_gqa7():
    sp = W.spec(2, n0=(4000, 2600), n0_range=None, batch=2, steps=24, k=300, n_local=64)
    _run(sp, 24)


def test_prefill_head_dim_64():
    sp = W.spec(1, n0=(3001,), steps=20, k=200, n_local=64, n_q_heads=8, n_kv_heads=4, head_dim=64)
    _run(sp, 20)


def test_prefill_chunk_of_one_selects_like_a_decode_step():
    T = tsl()
    sp = W.spec(1, n0=(7001,), steps=1, k=384, n_local=96)
    g_idx, g_cnt = _run(sp, 1)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    cap = sp.k + sp.n_sink + sp.n_local
    idx = torch.full((1, cap), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.zeros(1, sp.n_q_heads, sp.head_dim, device=DEV)
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
    ctx.decode_step(wl.q[0][0], wl.k_pool[0], wl.v_pool[0], wl.page_table, wl.seq_lens(0), prm, idx, cnt, out)
    assert ctx.status() == 0
    assert np.array_equal(idx.cpu().numpy()[0, :int(cnt[0])], g_idx[0, :g_cnt[0]])   # the same selection, bit for bit
    ctx.close()


def test_prefill_128k_chunk_of_512():
    # the 128K workload with a 512-query chunk: 2048 query rows per KV head, 16 query tiles x 8 KV
    # heads, 21 key tiles (2564 selected tokens, the last one ragged); every 8th query checked
    sp = W.spec(1, steps=512)
    _run(sp, 512, check_every=8)


def test_prefill_rejects_what_it_does_not_serve():
    T = tsl()
    sp = W.spec(0)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_F32, 1, wl.page_table.shape[1], wl.num_pages)
    q = torch.zeros(1, 4, sp.n_q_heads, sp.head_dim, device=DEV)
    idx = torch.zeros(1, 100, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.zeros(1, 4, sp.n_q_heads, sp.head_dim, device=DEV)
    with pytest.raises(T.TokenSelectError) as e:       # fp32 pools: no tensor-core chunk attention
        ctx.prefill_chunk(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, wl.seq_lens(0), T.params(k=64), idx, cnt, out)
    assert e.value.status == T.STATUS_CODE["TS_ERR_UNSUPPORTED"]
    ctx.close()


def test_prefill_page1_pool():
    # one token per page: the chunk's selection on the separate kernels, attention rows by token
    sp = W.spec(1, n0=(5003,), steps=40, k=512, n_local=128, page_size=1)
    _run(sp, 40)
