"""Selection overlap against query cosine (the TokenSelect review's figure 3(b)) measured on the
GPU path, against the CPU oracle.

Queries at cosines from 0.5 to 0.999 to a base query each select through ts_decode_step (no
Selection Cache); every selection is checked against the oracle's (same tie band and at-risk
margin as the decode tests), so the overlap curve the benchmark reports is the oracle's up to
tie-band swaps. The curve must rise with the cosine: the observation the Selection Cache rests
on (the pages' Lemma 1, pinned in the oracle, is its limit: above a threshold cosine the top-k
does not change at all).
"""
import numpy as np
import pytest
import torch

import bench
import oracle as O
import workloads as W
from parity import check_topk_set, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_overlap_rises_with_cosine_and_matches_the_oracle():
    T = tsl()
    sp = W.spec(1, n0=(32771,), steps=1, k=1024, n_local=128)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
    idx = torch.zeros(1, sp.k + sp.n_sink + sp.n_local, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    kp, pt = W.host_copy(wl.k_pool[0]), W.host_copy(wl.page_table)
    n = wl.n0[0]

    def both(q):
        part = bench.selected_part(T, ctx, wl, sp, q, idx, cnt, prm)
        vote = O.soft_vote(O.head_logits(W.host_copy(q)[0], kp, pt[0], n))
        ref_idx, ref_part = O.select_topk(vote, n, sp.k, sp.n_sink, sp.n_local)
        check_topk_set(idx[0, :int(cnt[0])].cpu().numpy(), ref_idx, vote, n, sp.k, sp.n_sink, sp.n_local,
                       "overlap query")
        return part, ref_part

    base, base_ref = both(wl.q[0][0])
    curve = []
    for rho, c, _, q2 in bench.overlap_pairs(wl, (0.5, 0.9, 0.99, 0.999), 1, DEV):
        part, ref = both(q2)
        ov, ov_ref = O.selection_overlap(base, part), O.selection_overlap(base_ref, ref)
        assert abs(ov - ov_ref) <= 4.0 / sp.k, (rho, ov, ov_ref)      # tie-band swaps only
        curve.append((c, ov))
    print("overlap vs cosine:", [(round(c, 4), round(o, 4)) for c, o in curve])
    assert all(curve[i][1] <= curve[i + 1][1] + 1e-9 for i in range(len(curve) - 1))
    assert curve[-1][1] > 0.9
    assert ctx.status() == 0
    ctx.close()
