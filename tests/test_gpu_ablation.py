"""The selection-function ablations on the GPU against the CPU oracle, through the C ABI.

The pages compare the head soft vote with two simpler selection functions
(TokenSelect deep notes, "Evolution of the selection function"; TokenSelect
review, section 3.1 and table 4): plain TopK(Q.K^T) over the concatenated
heads (the sum of the per-head logits, signed) and the head hard vote (each
query head's own top-k, counted). Both run through ts_score_fn + ts_select +
ts_sparse_attend and through ts_decode_step with params.score_fn.

Tolerances (derived here; the method's stated 1e-6 band is for the soft vote):

* logit sum: every GPU logit is an fp32 dot product of d exact bf16 products
  (any summation order) scaled by an fp32 alpha, so its error is at most
  (d + 4) 2^-24 alpha sum_e |q_e k_e| (the classical gamma_d bound plus the
  scaling); the sum over heads is compensated. Per token the bound B_i sums
  that over the heads, from the oracle's own |q| . |k| products. Tokens
  within B_i + B_tau of the k-th score are ambiguous; every other token must
  be decided as the oracle decides it.
* hard vote: a head's vote for a token is ambiguous when the token's logit is
  within the same per-logit bound (its own plus the head's k-th token's) of
  that head's k-th logit. GPU counts must equal the oracle's for tokens with
  no ambiguous vote and differ by at most their number of ambiguous votes
  otherwise; the GPU's index set must then equal, bit for bit, the oracle's
  top-k of the GPU's own counts (integer keys, ties to the lower index).
* attention on the GPU's set against the oracle's definition on that set,
  ATTN_REL = 2e-3 per (sequence, head) row, as everywhere.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity import check_attention, kv_flag, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _abs_pool(pool):
    """|K| of a host pool (bf16 bit patterns lose their sign bit)."""
    return (pool & np.uint16(0x7FFF)) if pool.dtype == np.uint16 else np.abs(pool)


def _gamma(d):
    return (d + 4) * 2.0 ** -24


def _setup(sp, wl):
    T = tsl()
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, kv_flag(T, sp), sp.batch, wl.page_table.shape[1],
                    wl.num_pages)
    B = sp.batch
    cap = sp.k + sp.n_sink + sp.n_local
    bufs = dict(idx=torch.full((B, cap), -1, dtype=torch.int32, device=DEV),
                count=torch.zeros(B, dtype=torch.int32, device=DEV),
                out=torch.zeros(B, sp.n_q_heads, sp.head_dim, device=DEV),
                lse=torch.zeros(B, sp.n_q_heads, device=DEV),
                vote=torch.zeros(B, ctx.max_tokens, device=DEV))
    return T, ctx, bufs


def _check_logit_sum(gs, idx, lg, lga, gam, n, k, s, w, where):
    ref = O.logit_sum_scores(lg)
    bound = gam * lga.sum(axis=0)
    err = np.abs(gs[:n].astype(np.float64) - ref)
    assert np.all(err <= bound), f"{where}: logit sum off by {float((err - bound).max()):.3e} beyond the bound"
    exp, _ = O.select_topk(ref, n, k, s, w)
    g, o = set(map(int, idx)), set(map(int, exp))
    assert len(g) == len(o) and np.all(np.diff(idx) > 0), f"{where}: set size or order"
    s_end, ls = O.budget_segments(n, s, w)
    cand = np.arange(s_end, ls)
    if len(cand) > k > 0:
        order = cand[np.argsort(-ref[cand], kind="stable")]
        t = order[k - 1]
        bad = [i for i in g ^ o if abs(ref[i] - ref[t]) > bound[i] + bound[t]]
        assert not bad, f"{where}: {len(bad)} tokens decided against the oracle outside the fp32 bound"
    return len(g ^ o)


def _check_hard_vote(gc, idx, lg, lga, gam, n, k, s, w, where):
    ref = O.hard_vote_counts(lg, n, k, s, w)
    s_end, ls = O.budget_segments(n, s, w)
    cand = np.arange(s_end, ls)
    amb = np.zeros(n, dtype=np.int64)
    if len(cand) > k > 0:
        for h in range(lg.shape[0]):
            order = cand[np.argsort(-lg[h, cand], kind="stable")]
            t = order[k - 1]
            band = gam * (lga[h, cand] + lga[h, t])
            amb[cand[np.abs(lg[h, cand] - lg[h, t]) <= band]] += 1
    gcn = gc[:n].astype(np.float64)
    assert np.all(gcn == np.round(gcn)), f"{where}: counts are not integers"
    diff = np.abs(gcn - ref)
    assert np.all(diff <= amb), f"{where}: counts differ beyond the ambiguous per-head votes"
    exp, _ = O.select_topk(gcn, n, k, s, w)          # the selection on the GPU's own counts: exact
    assert np.array_equal(np.asarray(idx), exp), f"{where}: index set differs from the top-k of the GPU counts"
    return int((diff > 0).sum())


def _run(sp, fn_name, steps=1, separate=False):
    wl = W.generate(sp, DEV)
    T, ctx, bufs = _setup(sp, wl)
    fn = {"logit_sum": T.TS_SCORE_LOGIT_SUM, "hard_vote": T.TS_SCORE_HEAD_HARD_VOTE}[fn_name]
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0, score_fn=fn)
    kp = W.host_copy(wl.k_pool[0])
    kpa = _abs_pool(kp)
    vp = W.host_copy(wl.v_pool[0])
    pt = W.host_copy(wl.page_table)
    moved = 0
    for t in range(steps):
        q = wl.q[t][0]
        seq = wl.seq_lens(t)
        bufs["vote"].zero_()
        if separate:
            ctx.score_fn(prm, q, wl.k_pool[0], wl.page_table, seq, bufs["vote"])
            ctx.select(bufs["vote"], seq, prm, bufs["idx"], bufs["count"])
            ctx.sparse_attend(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, bufs["idx"], bufs["count"],
                              bufs["out"], bufs["lse"])
        else:
            ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, bufs["idx"], bufs["count"],
                            bufs["out"], bufs["lse"], vote=bufs["vote"])
        assert ctx.status() == 0
        qh = W.host_copy(q)
        cnt = bufs["count"].cpu().numpy()
        idx = bufs["idx"].cpu().numpy()
        votes = bufs["vote"].cpu().numpy()
        out, lse = bufs["out"].cpu().numpy(), bufs["lse"].cpu().numpy()
        for b in range(sp.batch):
            n = wl.n0[b] + t
            where = f"{fn_name} step {t} seq {b}"
            lg = O.head_logits(qh[b], kp, pt[b], n)
            lga = O.head_logits(np.abs(qh[b]), kpa, pt[b], n)       # alpha sum_e |q_e k_e| per logit
            gi = idx[b, :cnt[b]]
            if fn_name == "logit_sum":
                moved += _check_logit_sum(votes[b], gi, lg, lga, _gamma(sp.head_dim), n, sp.k, sp.n_sink,
                                          sp.n_local, where)
            else:
                moved += _check_hard_vote(votes[b], gi, lg, lga, _gamma(sp.head_dim), n, sp.k, sp.n_sink,
                                          sp.n_local, where)
            ro, rl = O.sparse_attention(qh[b], kp, vp, pt[b], gi)
            check_attention(out[b], lse[b], ro, rl, where)
    print(f"{sp.name} {fn_name} separate={separate}: steps={steps} band_moves={moved}")
    ctx.close()


@pytest.mark.parametrize("fn_name", ["logit_sum", "hard_vote"])
@pytest.mark.parametrize("separate", [False, True])
def test_ablation_small(fn_name, separate):
    sp = W.spec(1, n0=(9001,), steps=2, k=256, n_local=64)
    _run(sp, fn_name, steps=2, separate=separate)


@pytest.mark.parametrize("fn_name", ["logit_sum", "hard_vote"])
def test_ablation_batched_gqa_and_edges(fn_name):
    # Qwen2-7B geometry (G = 7), a sequence shorter than k + s + w, one with few candidates
    sp = W.spec(2, n0=(3000, 400, 2700), n0_range=None, batch=3, steps=1, k=300, n_local=50)
    _run(sp, fn_name)


@pytest.mark.parametrize("fn_name", ["logit_sum", "hard_vote"])
def test_ablation_128k_full(fn_name):
    sp = W.spec(1, steps=1)
    _run(sp, fn_name)


def test_ablations_reject_top_p():
    T = tsl()
    sp = W.spec(0)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_F32, 1, wl.page_table.shape[1], wl.num_pages)
    prm = T.params(mode=T.TS_SELECT_TOPP, top_p=0.9, score_fn=T.TS_SCORE_LOGIT_SUM)
    vote = torch.zeros(1, ctx.max_tokens, device=DEV)
    with pytest.raises(T.TokenSelectError):
        ctx.score_fn(prm, wl.q[0][0], wl.k_pool[0], wl.page_table, wl.seq_lens(0), vote)
    ctx.close()
