"""Block-level selection (ts_select_blocks) against the CPU oracle, and the recall contrast of
token-level and block-level selection (the TokenSelect review's figure 2(b)) on the 128K
workload's needles.

The GPU votes come from ts_score; blocks are scored by their largest vote and the budget /
block best are taken. The selected block sets are compared with the oracle's on the oracle's
votes with the same tie band and at-risk margin as the token selections; recall@2048 of the
best tokens by vote is reported for every granularity and must fall as blocks grow.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity import check_topk_set, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_block_selection_and_recall_against_granularity():
    T = tsl()
    sp = W.spec(1, steps=1)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    n, budget = wl.n0[0], 2048
    seq = wl.seq_lens(0)
    vote = torch.zeros(1, ctx.max_tokens, device=DEV)
    ctx.score(wl.q[0][0], wl.k_pool[0], wl.page_table, seq, vote)
    gv = vote.cpu().numpy()[0]
    ov = O.soft_vote(O.head_logits(W.host_copy(wl.q[0][0])[0], W.host_copy(wl.k_pool[0]),
                                   W.host_copy(wl.page_table)[0], n))
    idx = torch.zeros(1, budget + 128, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    recalls = []
    for block in (1, 4, 16, 64, 128):
        ctx.select_blocks(vote, seq, block, budget, idx, cnt)
        assert ctx.status() == 0
        sel = idx[0, :int(cnt[0])].cpu().numpy()
        assert np.all(np.diff(sel) > 0)
        nb = -(-n // block)
        gb = np.array([gv[j * block:min(n, (j + 1) * block)].max() for j in range(nb)])
        ob = np.array([ov[j * block:min(n, (j + 1) * block)].max() for j in range(nb)])
        gblocks = np.unique(sel // block)
        oblocks = np.unique(O.select_blocks(ov, n, budget, block) // block)
        check_topk_set(gblocks, oblocks, ob, nb, budget // block, 0, 0, f"blocks of {block}", gpu_vote=gb)
        expect = np.concatenate([np.arange(j * block, min(n, (j + 1) * block)) for j in gblocks])
        assert np.array_equal(sel, expect), f"blocks of {block}: tokens are not the selected blocks' tokens"
        recalls.append(O.recall_at(sel, ov, n, budget))
    print("recall@2048 by block size 1, 4, 16, 64, 128:", [round(r, 4) for r in recalls])
    assert recalls[0] > 0.999
    assert all(recalls[i] >= recalls[i + 1] - 1e-3 for i in range(len(recalls) - 1))
    assert recalls[-1] < recalls[0]
    ctx.close()
