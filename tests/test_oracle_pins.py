"""Pins of the CPU oracle against things other than itself.

Each test fixes one part of the oracle by a value or property the pages and
the mathematics determine: hand-derived worked examples (tests/golden), closed
forms (dense attention via torch's SDPA, logsumexp), brute force on tiny
inputs, and invariants. Together they are meant to catch a dropped term, a
wrong sign or index, or a transposed operand anywhere in the oracle.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def one_page_pool(rows_by_head, d, P=16):
    """pool[1][H_kv][P][d] holding rows_by_head[g][i] at slot i; page table [0]."""
    Hkv = len(rows_by_head)
    pool = np.zeros((1, Hkv, P, d))
    for g, rows in enumerate(rows_by_head):
        for i, r in enumerate(rows):
            pool[0, g, i, :] = r
    return pool, np.array([0], dtype=np.int32)


def key_with_logit_axis(logit, axis, d, alpha):
    k = np.zeros(d)
    k[axis] = logit / alpha
    return k


# ------------------------------------------------------------------ golden

def test_bf16_widening_golden():
    for bits, val in GOLD["bf16"]["cases"]:
        got = O.as_f64(np.array([bits], dtype=np.uint16))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val)
    # and against torch's own bf16 -> float conversion on random patterns
    bits = np.random.default_rng(0).integers(0, 2**16, 4096).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]          # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.as_f64(bits), ref)


def test_soft_vote_mha_golden():
    c = GOLD["soft_vote_mha"]
    d = c["head_dim"]
    alpha = 1 / math.sqrt(d)
    rows0 = [key_with_logit_axis(math.log(a), 0, d, alpha) for a in c["head0_weights"]]
    rows1 = [key_with_logit_axis(math.log(b), 1, d, alpha) for b in c["head1_weights"]]
    pool, pt = one_page_pool([rows0, rows1], d)
    q = np.array(c["q"], dtype=np.float64)
    v = O.soft_vote(O.head_logits(q, pool, pt, 3))
    np.testing.assert_allclose(v, c["vote"], rtol=0, atol=1e-15)
    assert list(O.select_topk(v, 3, 1, 0, 0)[0]) == c["top1"]
    assert list(O.select_topk(v, 3, 2, 0, 0)[0]) == c["top2"]


def test_soft_vote_gqa_golden():
    c = GOLD["soft_vote_gqa"]
    d, alpha = 4, 0.5
    kv0 = [key_with_logit_axis(math.log(3), 0, d, alpha), np.zeros(d)]
    kv1 = [np.zeros(d), key_with_logit_axis(math.log(7), 2, d, alpha)]
    pool, pt = one_page_pool([kv0, kv1], d)
    v = O.soft_vote(O.head_logits(np.array(c["q"], float), pool, pt, 2))
    np.testing.assert_allclose(v, c["vote"], rtol=0, atol=1e-15)


def test_attention_golden():
    c = GOLD["attention"]
    d = 4
    kp, pt = one_page_pool([[np.zeros(d), key_with_logit_axis(math.log(3), 0, d, 0.5)]], d)
    vp, _ = one_page_pool([c["values"]], d)
    out, lse = O.sparse_attention(np.array([[1.0, 0, 0, 0]]), kp, vp, pt, [0, 1])
    np.testing.assert_allclose(out[0], c["out"], atol=1e-15)
    assert abs(lse[0] - c["lse"]) < 1e-15


def test_segments_golden():
    c = GOLD["segments"]
    w = np.array(c["weights"], float)
    vote = w / w.sum()                    # one head: its softmax is the normalised weights
    idx, part = O.select_topk(vote, len(w), c["k"], c["n_sink"], c["n_local"])
    assert list(idx) == c["idx"] and list(part) == c["part"]


def test_topp_golden():
    c = GOLD["topp"]
    v = np.array(c["vote"])
    for p, want in c["cases"]:
        idx, part = O.select_topp(v, 4, p, 1.0, 0, 0)
        assert list(part) == want, (p, part)


def test_cosine_golden():
    for a, b, want in GOLD["cosine"]["cases"]:
        assert abs(O.cosine(np.array(a, float), np.array(b, float)) - want) < 1e-15


# ------------------------------------------------------------ page tables

def test_gather_follows_page_table():
    P, d, Hkv = 4, 3, 2
    n_pages = 5
    pool = np.zeros((n_pages, Hkv, P, d))
    for p in range(n_pages):
        for g in range(Hkv):
            for s in range(P):
                pool[p, g, s] = [p, g, s]
    pt = np.array([3, 0, 4, 1, 2], dtype=np.int32)
    rows = O.gather_rows(pool, pt, np.arange(10), 1)
    for i in range(10):
        assert list(rows[i]) == [pt[i // P], 1, i % P]
    with pytest.raises(ValueError):
        O.gather_rows(pool, np.array([0, 7], dtype=np.int32), np.arange(8), 0)


def _random_case(seed, H=4, Hkv=2, d=16, n=70, P=16, scale_heads=True, dtype="f64"):
    rng = np.random.default_rng(seed)
    pages = -(-n // P)
    kp = rng.standard_normal((pages + 3, Hkv, P, d))
    if scale_heads:
        kp *= 10.0 ** rng.uniform(-2, 1, size=(1, Hkv, 1, 1))
    vp = rng.standard_normal((pages + 3, Hkv, P, d))
    pt = rng.permutation(pages + 3)[:pages].astype(np.int32)
    q = rng.standard_normal((H, d))
    return q, kp, vp, pt


def test_page_permutation_invariance():
    q, kp, vp, pt = _random_case(1)
    n = 70
    perm = np.random.default_rng(2).permutation(kp.shape[0])      # new physical slot of page p
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    pt2 = perm[pt].astype(np.int32)
    v1 = O.soft_vote(O.head_logits(q, kp, pt, n))
    v2 = O.soft_vote(O.head_logits(q, kp2, pt2, n))
    assert np.array_equal(v1, v2)
    idx = O.select_topk(v1, n, 8, 2, 5)[0]
    a1 = O.sparse_attention(q, kp, vp, pt, idx)
    a2 = O.sparse_attention(q, kp2, vp2, pt2, idx)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1])


def test_one_token_pages_hold_the_same_sequence():
    # token granularity (page size 1, TokenSelect review, section 3.4): token i sits in page
    # page_row[i], slot 0. The same logical cache in 16-token pages and in one-token pages gives
    # the same rows, votes, selection and attention.
    q, kp, vp, pt = _random_case(5, n=70)
    n = 70
    perm = np.random.default_rng(6).permutation(n + 9)[:n]          # one page per token
    kp1 = np.zeros((n + 9, kp.shape[1], 1, kp.shape[3]))
    vp1 = np.zeros_like(kp1)
    for i in range(n):
        kp1[perm[i], :, 0] = kp[pt[i // 16], :, i % 16]
        vp1[perm[i], :, 0] = vp[pt[i // 16], :, i % 16]
    pt1 = perm.astype(np.int32)
    for g in range(kp.shape[1]):
        assert np.array_equal(O.gather_rows(kp1, pt1, np.arange(n), g), O.gather_rows(kp, pt, np.arange(n), g))
    v16 = O.soft_vote(O.head_logits(q, kp, pt, n))
    v1 = O.soft_vote(O.head_logits(q, kp1, pt1, n))
    assert np.array_equal(v16, v1)
    idx = O.select_topk(v1, n, 8, 2, 5)[0]
    a16 = O.sparse_attention(q, kp, vp, pt, idx)
    a1 = O.sparse_attention(q, kp1, vp1, pt1, idx)
    assert np.array_equal(a16[0], a1[0]) and np.array_equal(a16[1], a1[1])


# ------------------------------------------------------------ invariants

def test_vote_sums_to_H_and_is_positive():
    for seed in range(4):
        q, kp, _, pt = _random_case(seed, H=8, Hkv=2, n=130)
        v = O.soft_vote(O.head_logits(q, kp, pt, 130))
        assert abs(v.sum() - 8) < 1e-12
        assert (v > 0).all()


def test_vote_invariant_to_per_head_logit_shift():
    # MHA: shifting every key of head h by c * q_h / (alpha |q_h|^2) adds c to all
    # its logits; each head's softmax, hence the vote, must not change.
    q, kp, _, pt = _random_case(3, H=3, Hkv=3, d=8, n=40)
    alpha = 1 / math.sqrt(8)
    v1 = O.soft_vote(O.head_logits(q, kp, pt, 40))
    kp2 = kp.copy()
    for h, c in enumerate([5.0, -3.0, 11.0]):
        kp2[:, h, :, :] += c * q[h] / (alpha * (q[h] @ q[h]))
    v2 = O.soft_vote(O.head_logits(q, kp2, pt, 40))
    np.testing.assert_allclose(v1, v2, rtol=1e-9, atol=0)


def test_vote_uniform_for_identical_keys():
    d, n, H = 8, 33, 4
    kp = np.tile(np.random.default_rng(5).standard_normal((1, 2, 1, d)), (3, 1, 16, 1))
    pt = np.array([2, 0, 1], dtype=np.int32)
    q = np.random.default_rng(6).standard_normal((H, d))
    v = O.soft_vote(O.head_logits(q, kp, pt, n))
    np.testing.assert_allclose(v, H / n, rtol=1e-13)


def test_logits_scale_and_explicit_scale():
    q, kp, _, pt = _random_case(7, H=2, Hkv=1, d=16, n=20)
    l_def = O.head_logits(q, kp, pt, 20)
    l_one = O.head_logits(q, kp, pt, 20, scale=1.0)
    np.testing.assert_allclose(l_def, l_one / 4.0, rtol=1e-15)
    K = O.gather_rows(kp, pt, np.arange(20), 0)
    ref = torch.from_numpy(q) @ torch.from_numpy(K).T       # library matmul, both heads on KV 0
    np.testing.assert_allclose(l_one, ref.numpy(), rtol=1e-13)


def test_single_head_selection_is_topk_of_logits():
    # H = 1: the softmax is monotone, so the vote ranks tokens like the logit.
    for seed in range(5):
        q, kp, _, pt = _random_case(10 + seed, H=1, Hkv=1, d=16, n=200)
        l = O.head_logits(q, kp, pt, 200)[0]
        v = O.soft_vote(O.head_logits(q, kp, pt, 200))
        s, w, k = 3, 20, 25
        _, part = O.select_topk(v, 200, k, s, w)
        cand = torch.arange(s, 200 - w)
        _, order = torch.sort(-torch.from_numpy(l)[cand], stable=True)
        want = np.sort(cand[order[:k]].numpy())
        assert np.array_equal(part, want)


def test_topk_nesting_and_sizes():
    q, kp, _, pt = _random_case(20, n=300)
    v = O.soft_vote(O.head_logits(q, kp, pt, 300))
    prev = set()
    for k in [1, 5, 17, 60, 200, 290, 400]:
        idx, part = O.select_topk(v, 300, k, 4, 16)
        assert prev <= set(part)
        assert len(idx) == 4 + 16 + min(k, 300 - 20)
        assert np.all(np.diff(idx) > 0)
        prev = set(part)


# ------------------------------------------------------------- brute force

def _dyadic_votes(rng, n):
    return rng.choice([0.125, 0.25, 0.375, 0.5, 0.75], size=n)


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(30)
    for trial in range(40):
        n = int(rng.integers(1, 15))
        s = int(rng.integers(0, 3))
        w = int(rng.integers(0, 3))
        k = int(rng.integers(0, 6))
        v = _dyadic_votes(rng, n)
        s_end, ls = O.budget_segments(n, s, w)
        cand = list(range(s_end, ls))
        kk = min(k, len(cand))
        best = None
        for sub in itertools.combinations(cand, kk):        # lexicographic order
            tot = sum(v[list(sub)]) if sub else 0.0
            if best is None or tot > best[0]:
                best = (tot, sub)
        idx, part = O.select_topk(v, n, k, s, w)
        assert tuple(part) == best[1], (v, s, w, k)
        assert set(idx) == set(range(s_end)) | set(best[1]) | set(range(ls, n))


def test_topp_brute_force_minimal_prefix():
    rng = np.random.default_rng(31)
    for trial in range(40):
        n = int(rng.integers(1, 11))
        v = _dyadic_votes(rng, n)
        total = float(v.sum())
        p = float(rng.choice([0.1, 0.3, 0.5, 0.7, 0.9, 0.99]))
        target = p * total
        m_star = None
        for m in range(1, n + 1):
            if any(sum(v[list(c)]) >= target for c in itertools.combinations(range(n), m)):
                m_star = m
                break
        _, part = O.select_topp(v, n, p, total, 0, 0)
        assert len(part) == m_star
        assert v[part].sum() >= target
        # a descending prefix: nothing left out beats anything kept; ties kept by lower index
        out = np.setdiff1d(np.arange(n), part)
        if len(out):
            assert v[out].max() <= v[part].min()
            lo = v[part].min()
            tied_out = out[v[out] == lo]
            tied_in = part[v[part] == lo]
            if len(tied_out):
                assert tied_in.max() < tied_out.min()


# --------------------------------------------------------------- attention

def test_dense_closed_form_matches_sdpa():
    # k + s + w >= N: the selection is every token and O-hat is dense SDPA.
    for seed, (H, Hkv) in enumerate([(4, 4), (8, 2), (6, 3)]):
        n = 45
        q, kp, vp, pt = _random_case(40 + seed, H=H, Hkv=Hkv, d=16, n=n)
        v = O.soft_vote(O.head_logits(q, kp, pt, n))
        idx, _ = O.select_topk(v, n, 40, 4, 16)
        assert np.array_equal(idx, np.arange(n))
        out, lse = O.sparse_attention(q, kp, vp, pt, idx)
        K = np.stack([O.gather_rows(kp, pt, np.arange(n), g) for g in range(Hkv)])
        V = np.stack([O.gather_rows(vp, pt, np.arange(n), g) for g in range(Hkv)])
        tq = torch.from_numpy(q)[None, :, None, :]             # [1, H, 1, d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, torch.from_numpy(K)[None], torch.from_numpy(V)[None], enable_gqa=True)
        np.testing.assert_allclose(out, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)
        G = H // Hkv
        Kh = torch.from_numpy(K).repeat_interleave(G, dim=0)      # [H, n, d]
        logits = torch.einsum("hd,hnd->hn", torch.from_numpy(q), Kh) / math.sqrt(16)
        np.testing.assert_allclose(lse, torch.logsumexp(logits, dim=1).numpy(), rtol=1e-13)


def test_sparse_attention_matches_masked_sdpa():
    H, Hkv, d, n = 8, 4, 16, 64
    q, kp, vp, pt = _random_case(50, H=H, Hkv=Hkv, d=d, n=n)
    idx = np.sort(np.random.default_rng(51).choice(n, 19, replace=False))
    out, _ = O.sparse_attention(q, kp, vp, pt, idx)
    K = torch.from_numpy(np.stack([O.gather_rows(kp, pt, np.arange(n), g) for g in range(Hkv)]))
    V = torch.from_numpy(np.stack([O.gather_rows(vp, pt, np.arange(n), g) for g in range(Hkv)]))
    mask = torch.zeros(1, 1, 1, n, dtype=torch.bool)
    mask[..., idx] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], K[None], V[None], attn_mask=mask, enable_gqa=True)
    np.testing.assert_allclose(out, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_lse_merge_of_partition():
    # O-hat over idx equals the log-sum-exp merge of O-hat over any partition of idx.
    H, Hkv, d, n = 4, 2, 16, 90
    q, kp, vp, pt = _random_case(60, H=H, Hkv=Hkv, d=d, n=n)
    idx = np.arange(n)
    out, lse = O.sparse_attention(q, kp, vp, pt, idx)
    parts = np.array_split(idx, 4)
    res = [O.sparse_attention(q, kp, vp, pt, p) for p in parts]
    M = np.max([r[1] for r in res], axis=0)
    wts = [np.exp(r[1] - M) for r in res]
    Z = np.sum(wts, axis=0)
    merged = sum(w[:, None] * r[0] for w, r in zip(wts, res)) / Z[:, None]
    np.testing.assert_allclose(merged, out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(M + np.log(Z), lse, rtol=1e-14)


# --------------------------------------------------------- selection cache

def test_cache_compares_with_last_miss_query():
    # Algorithm 1 only writes C_Q on a miss: q2 is close to q1 (a hit's query)
    # but far from q0 (the last miss), so it must miss.
    def unit(deg):
        r = math.radians(deg)
        return np.array([[math.cos(r), math.sin(r)]])
    theta = math.cos(math.radians(30))
    st = O.CacheState()
    assert O.cache_decision(st, unit(0), theta)[0] is False
    st.first, st.cq = False, unit(0)
    hit1, c1 = O.cache_decision(st, unit(20), theta)
    assert hit1 and abs(c1 - math.cos(math.radians(20))) < 1e-15
    hit2, c2 = O.cache_decision(st, unit(40), theta)
    assert not hit2 and abs(c2 - math.cos(math.radians(40))) < 1e-15


def test_cache_threshold_edges():
    st = O.CacheState(first=False, cq=np.array([[1.0, 0.0]]))
    assert O.cache_decision(st, np.array([[2.0, 0.0]]), 1.0)[0]                 # equality is a hit
    assert not O.cache_decision(st, np.array([[2.0, 0.0]]), np.nextafter(1.0, 2.0))[0]
    assert not O.cache_decision(st, np.array([[0.0, 0.0]]), -5.0)[0]            # zero query misses


def _traj(theta, steps=6, seed=70, mode="topk"):
    sp = W.spec(0, n0=(300,), steps=steps, theta=theta, k=16, n_local=8)
    wl = W.generate(sp, "cpu")
    kp, vp = W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0])
    pt = W.host_copy(wl.page_table)[0]
    st = O.CacheState()
    res = []
    for t in range(steps):
        q = W.host_copy(wl.q[t][0])[0]
        res.append(O.decode_step(st, q, kp, vp, pt, wl.n0[0] + t, mode=mode, k=sp.k,
                                 n_sink=sp.n_sink, n_local=sp.n_local, theta=theta))
    return res, wl


def test_cache_disabled_and_always():
    never, _ = _traj(theta=1.5)
    assert not any(r["hit"] for r in never)
    always, _ = _traj(theta=-1.0)
    assert not always[0]["hit"] and all(r["hit"] for r in always[1:])
    # a hit keeps the cached part and rebuilds the sinks/window at the current length
    for t, r in enumerate(always[1:], start=1):
        assert np.array_equal(r["part"], always[0]["part"])
        n = 300 + t
        assert set(range(n - 8, n)) <= set(r["idx"]) and set(range(4)) <= set(r["idx"])
        assert np.all(np.diff(r["idx"]) > 0)


def test_identical_query_hits():
    st = O.CacheState()
    q, kp, vp, pt = _random_case(80, n=64)
    r0 = O.decode_step(st, q, kp, vp, pt, 64, k=8, n_sink=2, n_local=4, theta=0.9)
    r1 = O.decode_step(st, q.copy(), kp, vp, pt, 64, k=8, n_sink=2, n_local=4, theta=0.9)
    assert not r0["hit"] and r1["hit"] and np.array_equal(r0["idx"], r1["idx"])


def test_miss_steps_equal_fresh_selection():
    res, wl = _traj(theta=1.5, steps=4)
    kp, vp = W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0])
    pt = W.host_copy(wl.page_table)[0]
    for t, r in enumerate(res):
        q = W.host_copy(wl.q[t][0])[0]
        v = O.soft_vote(O.head_logits(q, kp, pt, 300 + t))
        assert np.array_equal(r["idx"], O.select_topk(v, 300 + t, 16, 4, 8)[0])


# ---------------------------------------------------------------- needles

@pytest.mark.parametrize("cfg,overrides", [
    (0, {}),
    (1, dict(n0=(8192,), steps=1)),
    (2, dict(batch=2, n0=(6000, 9000), n0_range=None, steps=1)),
])
def test_needles_selected_at_step0(cfg, overrides):
    sp = W.spec(cfg, **overrides)
    wl = W.generate(sp, "cpu")
    kp, pt_all = W.host_copy(wl.k_pool[0]), W.host_copy(wl.page_table)
    for b in range(sp.batch):
        q = W.host_copy(wl.q[0][0])[b]
        n = wl.n0[b]
        v = O.soft_vote(O.head_logits(q, kp, pt_all[b], n))
        idx, _ = O.select_topk(v, n, sp.k, sp.n_sink, sp.n_local)
        needles = set(wl.needle_pos[0][b].flatten().tolist())
        assert needles and needles <= set(idx.tolist())


def test_decode_step_keeps_last_miss_query():
    # Through decode_step: q1 hits against q0, q2 is close to q1 but far from q0.
    # Algorithm 1 keeps C_Q = q0 across the hit, so q2 must miss.
    d, n = 2, 20
    rng = np.random.default_rng(90)
    kp = rng.standard_normal((2, 1, 16, d))
    vp = rng.standard_normal((2, 1, 16, d))
    pt = np.array([1, 0], dtype=np.int32)
    theta = math.cos(math.radians(30))
    st = O.CacheState()
    hits = []
    for deg in (0, 20, 40):
        r = math.radians(deg)
        q = np.array([[math.cos(r), math.sin(r)]])
        hits.append(O.decode_step(st, q, kp, vp, pt, n, k=4, n_sink=1, n_local=2, theta=theta)["hit"])
    assert hits == [False, True, False]


def test_equal_keys_tie_exactly_and_go_to_lower_index():
    # Identical keys must give identical votes; the tie then goes to the lower index.
    rng = np.random.default_rng(95)
    d, n = 64, 300
    kp = rng.standard_normal((n // 16 + 1, 2, 16, d))
    pt = rng.permutation(n // 16 + 1).astype(np.int32)
    q = rng.standard_normal((4, d))
    tied = [17, 90, 144, 201, 260]
    for g in range(2):                       # the same key at every tied position, in every KV head
        key = 3.0 * q[2 * g] / np.linalg.norm(q[2 * g])
        for i in tied:
            kp[pt[i // 16], g, i % 16] = key
    v = O.soft_vote(O.head_logits(q, kp, pt, n))
    assert len(set(v[tied].tolist())) == 1
    _, part = O.select_topk(v, n, 3, 0, 0)
    assert list(part) == tied[:3]


# ------------------------------------------- selection-function ablations (R10, R11)

def test_ablation_selectors_golden():
    g = GOLD["ablation_selectors"]
    lg = np.array(g["logits"], dtype=np.float64)
    n, k, s, w = g["n"], g["k"], g["n_sink"], g["n_local"]
    c = O.hard_vote_counts(lg, n, k, s, w)
    assert c.tolist() == g["hard_vote_counts"]
    idx, _ = O.select_topk(c, n, k, s, w)
    assert idx.tolist() == g["hard_vote_idx"]
    ls = O.logit_sum_scores(lg)
    assert ls.tolist() == g["logit_sum"]
    idx, _ = O.select_topk(ls, n, k, s, w)
    assert idx.tolist() == g["logit_sum_idx"]


def _brute_topk(scores, cand, k):
    """The k-subset of cand with the largest score sum; ties -> lexicographically smallest."""
    best, best_key = None, None
    for sub in itertools.combinations(cand, min(k, len(cand))):
        key = (sum(scores[i] for i in sub), tuple(-i for i in sub))
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return sorted(best)


def test_hard_vote_brute_force_with_ties():
    rng = np.random.default_rng(7)
    for trial in range(40):
        H, n, k = 3, 11, int(rng.integers(1, 5))
        lg = rng.integers(0, 4, size=(H, n)).astype(np.float64)     # many ties
        s, w = 1, 2
        cand = list(range(s, n - w))
        counts = np.zeros(n)
        for h in range(H):
            for i in _brute_topk(lg[h], cand, k):
                counts[i] += 1
        assert np.array_equal(O.hard_vote_counts(lg, n, k, s, w), counts)
        _, part = O.select_topk(counts, n, k, s, w)
        assert list(part) == _brute_topk(counts, cand, k)


def test_logit_sum_is_the_concatenated_dot_product():
    # GQA 4/2: the concatenated query against each token's keys, each KV head repeated for its
    # G query heads, is one flat dot product per token
    rng = np.random.default_rng(3)
    H, Hkv, d, n = 4, 2, 8, 37
    G = H // Hkv
    q = rng.normal(size=(H, d))
    pool = rng.normal(size=(3, Hkv, 16, d))
    pt = np.array([2, 0, 1], dtype=np.int32)
    lg = O.head_logits(q, pool, pt, n)
    flat = np.empty(n)
    for i in range(n):
        rows = pool[pt[i // 16], :, i % 16, :]                  # [Hkv][d]
        kcat = np.repeat(rows, G, axis=0).reshape(-1)            # [H*d]
        flat[i] = np.dot(q.reshape(-1), kcat) / math.sqrt(d)
    assert np.allclose(O.logit_sum_scores(lg), flat, rtol=1e-12, atol=1e-12)


def test_single_head_all_selection_functions_agree():
    rng = np.random.default_rng(5)
    n, k, s, w = 300, 17, 4, 20
    lg = rng.normal(size=(1, n)) * 3.0
    sets = [tuple(O.select_topk(O.selection_scores(lg, f, n, k, s, w), n, k, s, w)[0]) for f in O.SCORE_FNS]
    assert sets[0] == sets[1] == sets[2]


def test_logit_sum_is_dominated_by_the_high_norm_head_and_soft_vote_is_not():
    # the pages' reason for the head soft vote: one head with logits a thousand times larger
    # decides the plain TopK alone, while the soft vote weighs every head's softmax equally
    rng = np.random.default_rng(9)
    H, n, k, s, w = 4, 400, 10, 0, 0
    lg = rng.normal(size=(H, n))
    lg[2] *= 1000.0
    part_sum = O.select_topk(O.logit_sum_scores(lg), n, k, s, w)[1]
    part_h2 = O.select_topk(lg[2], n, k, s, w)[1]
    assert list(part_sum) == list(part_h2)
    part_soft = O.select_topk(O.soft_vote(lg), n, k, s, w)[1]
    assert set(part_soft) != set(part_h2)


def test_identical_heads_hard_vote_is_the_single_head_topk():
    rng = np.random.default_rng(11)
    n, k, s, w = 200, 12, 4, 16
    row = rng.normal(size=n)
    lg = np.stack([row] * 5)
    c = O.hard_vote_counts(lg, n, k, s, w)
    assert set(np.unique(c)) <= {0.0, 5.0}
    assert list(O.select_topk(c, n, k, s, w)[1]) == list(O.select_topk(row, n, k, s, w)[1])


def test_decode_step_with_ablation_scores():
    wl = W.generate(W.spec(0, steps=1), "cpu")
    kp, vp, pt = W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0]), W.host_copy(wl.page_table)
    q = W.host_copy(wl.q[0][0])[0]
    n = wl.n0[0]
    lg = O.head_logits(q, kp, pt[0], n)
    for f in O.SCORE_FNS:
        r = O.decode_step(O.CacheState(), q, kp, vp, pt[0], n, k=64, n_sink=4, n_local=16, theta=2.0, score_fn=f)
        exp, _ = O.select_topk(O.selection_scores(lg, f, n, 64, 4, 16), n, 64, 4, 16)
        assert np.array_equal(r["idx"], exp)
    with pytest.raises(ValueError):
        O.decode_step(O.CacheState(), q, kp, vp, pt[0], n, mode="topp", score_fn="hard_vote")


# ------------------------------------------------------- chunk-wise prefill (R12)

def _tiny_pools(rng, Hkv=2, d=8, pages=5):
    kp = rng.normal(size=(pages, Hkv, 16, d))
    vp = rng.normal(size=(pages, Hkv, 16, d))
    pt = rng.permutation(pages).astype(np.int32)
    return kp, vp, pt


def test_prefill_chunk_of_one_is_a_decode_step():
    rng = np.random.default_rng(21)
    kp, vp, pt = _tiny_pools(rng)
    n, H = 70, 4
    q = rng.normal(size=(1, H, 8))
    r = O.prefill_chunk(q, kp, vp, pt, n, k=9, n_sink=2, n_local=6)
    d = O.decode_step(O.CacheState(), q[0], kp, vp, pt, n, k=9, n_sink=2, n_local=6, theta=2.0)
    assert np.array_equal(r["idx"], d["idx"])
    assert np.allclose(r["out"][0], d["out"], rtol=1e-12, atol=1e-12)
    assert np.allclose(r["lse"][0], d["lse"], rtol=1e-12, atol=1e-12)


def test_prefill_dense_closed_form_is_causal_sdpa():
    # k + s + w >= n: every token is selected, so each chunk query sees exactly the tokens up to
    # its own position: the causal attention of the last c positions over the whole cache
    rng = np.random.default_rng(22)
    kp, vp, pt = _tiny_pools(rng)
    n, c, H, Hkv, d = 53, 7, 4, 2, 8
    G = H // Hkv
    q = rng.normal(size=(c, H, d))
    r = O.prefill_chunk(q, kp, vp, pt, n, k=200, n_sink=2, n_local=6)
    assert np.array_equal(r["idx"], np.arange(n))
    K = np.stack([kp[pt[i // 16], :, i % 16, :] for i in range(n)], axis=1)     # [Hkv][n][d]
    V = np.stack([vp[pt[i // 16], :, i % 16, :] for i in range(n)], axis=1)
    Kq = torch.tensor(np.repeat(K, G, axis=0))                                  # [H][n][d]
    Vq = torch.tensor(np.repeat(V, G, axis=0))
    Q = torch.tensor(q.transpose(1, 0, 2))                                      # [H][c][d]
    pos = torch.arange(n - c, n).view(c, 1)
    mask = torch.arange(n).view(1, n) <= pos                                    # [c][n]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, Kq, Vq, attn_mask=mask).numpy()
    assert np.allclose(r["out"], ref.transpose(1, 0, 2), rtol=1e-10, atol=1e-10)


def test_prefill_selection_ignores_the_order_of_the_chunk():
    rng = np.random.default_rng(23)
    kp, vp, pt = _tiny_pools(rng)
    n, c = 64, 6
    q = rng.normal(size=(c, 4, 8))
    a = O.prefill_chunk(q, kp, vp, pt, n, k=7, n_sink=2, n_local=5)
    b = O.prefill_chunk(q[::-1].copy(), kp, vp, pt, n, k=7, n_sink=2, n_local=5)
    assert np.array_equal(a["idx"], b["idx"])
    assert np.allclose(a["q_mean"], q.mean(axis=0), rtol=1e-14, atol=1e-14)


def test_prefill_selection_brute_force_on_the_mean_query():
    rng = np.random.default_rng(24)
    kp, vp, pt = _tiny_pools(rng, pages=1)
    n, c, k, s, w = 14, 3, 4, 1, 2
    q = rng.normal(size=(c, 4, 8))
    r = O.prefill_chunk(q, kp, vp, pt, n, k=k, n_sink=s, n_local=w)
    # the soft vote of the mean query, from scores computed without the oracle's helpers
    qm = q.mean(axis=0)
    alpha = 1 / math.sqrt(8)
    v = np.zeros(n)
    for h in range(4):
        sc = np.array([alpha * float(qm[h] @ kp[pt[0], h // 2, i]) for i in range(n)])
        e = np.exp(sc - sc.max())
        v += e / e.sum()
    best = _brute_topk(v, list(range(s, n - w)), k)
    assert list(r["part"]) == best
    # query i of the chunk sees no token after its own position
    for i in range(c):
        vis = r["idx"][r["idx"] <= n - c + i]
        o, _ = O.sparse_attention(q[i], kp, vp, pt, vis)
        assert np.allclose(r["out"][i], o, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------- Lemma 1 (R13)

def _topk_set(scores, k):
    return set(np.argsort(-scores, kind="stable")[:k].tolist())


def test_lemma1_threshold_is_sufficient():
    # queries built at a cosine just above eps in random orthogonal directions never change the
    # dot-product top-k
    rng = np.random.default_rng(31)
    for trial in range(30):
        n, d, k = 200, 16, 10
        K = rng.normal(size=(n, d))
        q1 = rng.normal(size=d)
        eps = O.lemma1_epsilon(q1, K, k)
        base = _topk_set(K @ q1, k)
        u = q1 / np.linalg.norm(q1)
        for _ in range(20):
            p = rng.normal(size=d)
            p -= (p @ u) * u
            p /= np.linalg.norm(p)
            c = eps + (1.0 - eps) * rng.uniform(1e-3, 1.0)
            q2 = (u * c + p * math.sqrt(1.0 - c * c)) * rng.uniform(0.5, 2.0)
            assert O.cosine(q1, q2) > eps
            assert _topk_set(K @ q2, k) == base


def test_lemma1_bound_is_met_by_an_adversarial_direction():
    # moving q1 towards the direction that favours the (k+1)-th key over the k-th swaps them once
    # cot t < (difference of their orthogonal components) / gap: the lemma's bound lies at or above
    # that critical cosine, and below it the selection does change
    rng = np.random.default_rng(32)
    n, d, k = 60, 8, 5
    K = rng.normal(size=(n, d))
    q1 = rng.normal(size=d)
    u = q1 / np.linalg.norm(q1)
    order = np.argsort(-(K @ u), kind="stable")
    i, j = order[k - 1], order[k]
    diff = K[j] - K[i]
    perp = diff - (diff @ u) * u
    p = perp / np.linalg.norm(perp)
    gap = float((K[i] - K[j]) @ u)
    t_crit = math.atan2(gap, float(np.linalg.norm(perp)))      # cot t = |perp| / gap
    eps = O.lemma1_epsilon(q1, K, k)
    assert eps >= math.cos(t_crit) - 1e-12
    t = t_crit * 1.05
    q2 = u * math.cos(t) + p * math.sin(t)
    assert _topk_set(K @ q2, k) != _topk_set(K @ u, k)


def test_selection_overlap_definition():
    assert O.selection_overlap(np.array([1, 2, 3, 4]), np.array([3, 4, 5])) == 0.5
    assert O.selection_overlap(np.array([7]), np.array([7])) == 1.0


# ----------------------------------------------- block-level selection contrast (R14)

def test_select_blocks_hand_case():
    v = np.array([0.1, 0.9, 0.2, 0.2, 0.5, 0.0, 0.3, 0.3, 0.3, 0.1])
    # blocks of 3: [0.1 0.9 0.2] [0.2 0.5 0.0] [0.3 0.3 0.3] [0.1] -> maxima 0.9, 0.5, 0.3, 0.1
    assert O.select_blocks(v, 10, 6, 3).tolist() == [0, 1, 2, 3, 4, 5]
    assert O.select_blocks(v, 10, 5, 3).tolist() == [0, 1, 2]          # 5 // 3 = one block
    assert O.select_blocks(v, 10, 12, 3).tolist() == list(range(10))   # the ragged last block too
    # token granularity: the budget best tokens, ties to the lower index
    assert O.select_blocks(v, 10, 3, 1).tolist() == [1, 4, 6]
    assert O.recall_at(np.array([1, 4, 6]), v, 10, 3) == 1.0
    assert O.recall_at(np.array([0, 1, 2]), v, 10, 3) == pytest.approx(1 / 3)


def test_block_granularity_one_is_token_topk_and_recall_falls_with_block_size():
    # the review's figure 2(b) on scattered needles: token-level selection recalls every one of
    # the best m tokens, 128-token blocks recall far fewer within the same budget
    rng = np.random.default_rng(41)
    n, m = 1 << 14, 256
    v = rng.exponential(size=n) * 1e-3
    v[rng.choice(n, m, replace=False)] += 1.0                         # isolated important tokens
    assert O.recall_at(O.select_blocks(v, n, m, 1), v, n, m) == 1.0
    rec = [O.recall_at(O.select_blocks(v, n, m, b), v, n, m) for b in (1, 4, 16, 64, 128)]
    assert all(rec[i] >= rec[i + 1] for i in range(len(rec) - 1))
    assert rec[-1] < 0.1
