"""Kernel-level GPU checks through the C ABI: selection on generator-made votes
(bit-exact: integer work), attention on generator-made index sets, edge cases,
device error reporting and determinism."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity import ATTN_REL, LSE_ABS, GpuRunner, check_attention, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _ctx(T, H=4, Hkv=4, d=64, kv="f32", B=1, max_pages=64, num_pages=64):
    return T.Context(H, Hkv, d, T.TS_KV_F32 if kv == "f32" else T.TS_KV_BF16, B, max_pages, num_pages)


def _votes(rng, B, n, ties):
    if ties:
        v = rng.choice(np.array([1, 2, 3, 4, 6, 8], dtype=np.float32) / 64.0, size=(B, n))
    else:
        v = (rng.random((B, n)) * 4 + 1e-3).astype(np.float32)
    return v


@pytest.mark.parametrize("n,k,s,w,ties", [
    (70000, 2048, 4, 512, True), (70000, 2048, 4, 512, False), (4097, 100, 0, 0, True),
    (300, 290, 4, 16, False), (50, 2048, 4, 16, True), (9000, 0, 4, 16, False), (1, 5, 4, 16, True),
])
def test_topk_select_bit_exact(n, k, s, w, ties):
    T = tsl()
    rng = np.random.default_rng(n + k)
    B = 3
    ns = [n, max(1, n // 2), max(1, n - 7)]
    ctx = _ctx(T, B=B, max_pages=(n + 15) // 16 + 1, num_pages=1)
    v = _votes(rng, B, ctx.max_tokens, ties)
    vote = torch.from_numpy(v).to(DEV)
    seq = torch.tensor(ns, dtype=torch.int32, device=DEV)
    cap = k + s + w + 1
    idx = torch.full((B, cap), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    ctx.select(vote, seq, T.params(k=k, n_sink=s, n_local=w), idx, cnt)
    assert ctx.status() == 0
    for b in range(B):
        want, _ = O.select_topk(v[b].astype(np.float64), ns[b], k, s, w)
        got = idx[b, :int(cnt[b])].cpu().numpy()
        assert np.array_equal(got, want), (b, len(got), len(want))


@pytest.mark.parametrize("n,p,s,w", [(60000, 0.9, 4, 512), (60000, 0.99, 0, 0), (5000, 0.5, 4, 16),
                                     (777, 1.0, 4, 16), (3000, 0.01, 0, 0)])
def test_topp_select_bit_exact_on_dyadic_votes(n, p, s, w):
    # dyadic votes make every partial sum exact on both sides
    T = tsl()
    rng = np.random.default_rng(int(p * 1000) + n)
    H = 4
    B = 2
    ctx = _ctx(T, H=H, Hkv=4, B=B, max_pages=(n + 15) // 16, num_pages=1)
    raw = rng.choice(np.array([1, 2, 3, 5, 8, 13], dtype=np.float64), size=(B, ctx.max_tokens)) * rng.choice(
        [2.0 ** -12, 2.0 ** -10], size=(B, ctx.max_tokens))
    raw[:, n:] = 0
    raw = raw / raw[:, :n].sum(axis=1, keepdims=True) * H          # not exact: re-quantise below
    v = (np.round(raw * 2 ** 24) / 2 ** 24).astype(np.float32)
    vote = torch.from_numpy(v).to(DEV)
    seq = torch.tensor([n, n], dtype=torch.int32, device=DEV)
    idx = torch.full((B, ctx.max_tokens), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    ctx.select(vote, seq, T.params(mode=T.TS_SELECT_TOPP, top_p=p, n_sink=s, n_local=w), idx, cnt)
    assert ctx.status() == 0
    for b in range(B):
        want, _ = O.select_topp(v[b].astype(np.float64), n, p, float(H), s, w)
        got = idx[b, :int(cnt[b])].cpu().numpy()
        assert np.array_equal(got, want), (b, len(got), len(want))


@pytest.mark.parametrize("cfg,overrides", [
    (1, dict(n0=(20000,), steps=1)), (0, dict()), (2, dict(batch=2, n0=(3000, 9000), n0_range=None, steps=1)),
])
def test_attend_on_generated_index_sets(cfg, overrides):
    T = tsl()
    sp = W.spec(cfg, **overrides)
    wl = W.generate(sp, DEV)
    rng = np.random.default_rng(5)
    B = sp.batch
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_F32 if sp.kv_dtype == "f32" else T.TS_KV_BF16,
                    B, wl.page_table.shape[1], wl.num_pages)
    sizes = [int(rng.integers(1, min(3000, wl.n0[b]) + 1)) for b in range(B)]
    cap = max(sizes)
    idx_np = np.full((B, cap), -1, dtype=np.int32)
    for b in range(B):
        idx_np[b, :sizes[b]] = np.sort(rng.choice(wl.n0[b], sizes[b], replace=False))
    idx = torch.from_numpy(idx_np).to(DEV)
    cnt = torch.tensor(sizes, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, sp.n_q_heads, sp.head_dim, device=DEV)
    lse = torch.zeros(B, sp.n_q_heads, device=DEV)
    q = wl.q[0][0]
    ctx.sparse_attend(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, idx, cnt, out, lse)
    assert ctx.status() == 0
    kp, vp, pt = W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0]), W.host_copy(wl.page_table)
    qh = W.host_copy(q)
    for b in range(B):
        ro, rl = O.sparse_attention(qh[b], kp, vp, pt[b], idx_np[b, :sizes[b]])
        check_attention(out[b].cpu().numpy(), lse[b].cpu().numpy(), ro, rl, f"seq {b}")


def test_empty_selection_gives_zero_output():
    T = tsl()
    sp = W.spec(0, n0=(40,), steps=1)
    wl = W.generate(sp, DEV)
    ctx = T.Context(4, 4, 64, T.TS_KV_F32, 1, wl.page_table.shape[1], wl.num_pages)
    idx = torch.zeros(1, 8, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((1, 4, 64), 5.0, device=DEV)
    lse = torch.zeros(1, 4, device=DEV)
    ctx.sparse_attend(wl.q[0][0], wl.k_pool[0], wl.v_pool[0], wl.page_table, idx, cnt, out, lse)
    assert ctx.status() == 0
    assert torch.all(out == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)


def test_zero_length_sequence_in_batch():
    sp = W.spec(2, batch=2, n0=(0, 500), n0_range=None, steps=1, k=40, n_local=8, needles="lnN2")
    wl = W.generate(sp, DEV)
    g = GpuRunner(wl, theta=2.0)
    r = g.step(0)
    assert len(r["idx"][0]) == 0 and np.all(r["out"][0] == 0)
    assert len(r["idx"][1]) == 4 + 40 + 8


def test_device_errors_are_reported():
    T = tsl()
    sp = W.spec(0, n0=(100,), steps=1)
    wl = W.generate(sp, DEV)
    ctx = T.Context(4, 4, 64, T.TS_KV_F32, 1, wl.page_table.shape[1], wl.num_pages)
    q = wl.q[0][0]
    vote = torch.zeros(1, ctx.max_tokens, device=DEV)
    # a page id outside the pool
    bad_pt = wl.page_table.clone()
    bad_pt[0, 2] = wl.num_pages + 5
    ctx.score(q, wl.k_pool[0], bad_pt, torch.tensor([100], dtype=torch.int32, device=DEV), vote)
    assert ctx.status() == T.STATUS_CODE["TS_ERR_PAGE_OOB"]
    assert ctx.status() == 0                      # read and cleared
    # a length beyond the page table
    ctx.score(q, wl.k_pool[0], wl.page_table, torch.tensor([ctx.max_tokens + 1], dtype=torch.int32, device=DEV),
              vote)
    assert ctx.status() == T.STATUS_CODE["TS_ERR_SEQ_LEN"]
    # an index buffer too small for k + s + w
    ctx.score(q, wl.k_pool[0], wl.page_table, torch.tensor([100], dtype=torch.int32, device=DEV), vote)
    idx = torch.zeros(1, 10, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    ctx.select(vote, torch.tensor([100], dtype=torch.int32, device=DEV), T.params(k=64, n_sink=4, n_local=16), idx,
               cnt)
    assert ctx.status() == T.STATUS_CODE["TS_ERR_CAPACITY"]
    assert int(cnt[0]) == 0
    # the context still works afterwards
    idx = torch.zeros(1, 84, dtype=torch.int32, device=DEV)
    ctx.select(vote, torch.tensor([100], dtype=torch.int32, device=DEV), T.params(k=64, n_sink=4, n_local=16), idx,
               cnt)
    assert ctx.status() == 0 and int(cnt[0]) == 84


def test_repeat_runs_are_bit_identical():
    sp = W.spec(1, n0=(40000,), steps=1)
    wl = W.generate(sp, DEV)
    g = GpuRunner(wl, theta=2.0)
    a = g.step(0)
    b = g.step(0)
    assert np.array_equal(a["vote"], b["vote"]) and np.array_equal(a["out"], b["out"])
    assert all(np.array_equal(x, y) for x, y in zip(a["idx"], b["idx"]))


def test_page_permutation_is_bit_identical():
    sp = W.spec(1, n0=(30000,), steps=1)
    wl = W.generate(sp, DEV)
    g = GpuRunner(wl, theta=2.0)
    a = g.step(0)
    perm = torch.randperm(wl.num_pages, generator=torch.Generator().manual_seed(3)).to(DEV)
    inv = torch.argsort(perm)
    wl.k_pool[0] = wl.k_pool[0][inv].contiguous()      # page p moves to slot perm[p]
    wl.v_pool[0] = wl.v_pool[0][inv].contiguous()
    pt = wl.page_table.clone()
    valid = pt >= 0
    pt[valid] = perm[pt[valid].long()].to(torch.int32)
    wl.page_table = pt
    g2 = GpuRunner(wl, theta=2.0)
    b = g2.step(0)
    assert np.array_equal(a["vote"], b["vote"]) and np.array_equal(a["out"], b["out"])
    assert all(np.array_equal(x, y) for x, y in zip(a["idx"], b["idx"]))


def test_cache_always_and_never():
    sp = W.spec(1, n0=(5000,), steps=4, k=128, n_local=32)
    wl = W.generate(sp, DEV)
    never = GpuRunner(wl, theta=1.5)
    assert not any(bool(never.step(t)["hit"][0]) for t in range(4))
    always = GpuRunner(wl, theta=-1.0)
    hits = [bool(always.step(t)["hit"][0]) for t in range(4)]
    assert hits == [False, True, True, True]


def test_graph_capture_replay_and_kernel_timing():
    T = tsl()
    sp = W.spec(1, n0=(20000,), steps=2)
    wl = W.generate(sp, DEV)
    B, H, d = 1, sp.n_q_heads, sp.head_dim
    ctx = T.Context(H, sp.n_kv_heads, d, T.TS_KV_BF16, B, wl.page_table.shape[1], wl.num_pages)
    prm = T.params(theta=2.0)
    cap = sp.k + sp.n_sink + sp.n_local
    q = wl.q[0][0].clone()
    seq = wl.seq_lens(0)
    idx = torch.zeros(B, cap, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, H, d, device=DEV)
    ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt, out)
    torch.cuda.synchronize()
    direct = (idx.clone(), out.clone())
    T.ts_profile_enable(ctx.handle, True)
    k0 = T.ts_kernel_count(ctx.handle)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt, out)
    per_replay = T.ts_kernel_count(ctx.handle) - k0
    assert per_replay == 1                      # the persistent whole-step kernel
    idx.zero_()
    out.zero_()
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        prof = T.ts_profile_read(ctx.handle, keep=True)
        ms, n = prof["step"]
        assert n == 1 and ms > 0, prof
    assert torch.equal(idx, direct[0]) and torch.equal(out, direct[1])
    assert ctx.status() == 0


def test_multi_kernel_path_launch_count(monkeypatch):
    monkeypatch.setenv("TOKENSELECT_MULTI_KERNEL", "1")
    T = tsl()
    sp = W.spec(1, n0=(5000,), steps=1)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1],
                    wl.num_pages)
    cap = sp.k + sp.n_sink + sp.n_local
    idx = torch.zeros(1, cap, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.zeros(1, sp.n_q_heads, sp.head_dim, device=DEV)
    k0 = T.ts_kernel_count(ctx.handle)
    ctx.decode_step(wl.q[0][0], wl.k_pool[0], wl.v_pool[0], wl.page_table, wl.seq_lens(0), T.params(theta=2.0),
                    idx, cnt, out)
    assert ctx.status() == 0
    assert T.ts_kernel_count(ctx.handle) - k0 >= 8


def test_misaligned_query_takes_the_cuda_core_scan_with_the_same_result():
    # a caller query that is only 4-byte aligned: no tensor-core scan and no staged cache test;
    # selection and output agree with the aligned query (tensor-core scan)
    T = tsl()
    sp = W.spec(1, n0=(12001,), steps=1, k=512, n_local=64)
    wl = W.generate(sp, DEV)
    H, Hkv, d = sp.n_q_heads, sp.n_kv_heads, sp.head_dim
    n = int(wl.n0[0])
    ctx = T.Context(H, Hkv, d, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    seq = torch.tensor([n], dtype=torch.int32, device=DEV)
    q = wl.q[0][0].contiguous()
    qbuf = torch.zeros(q.numel() + 1, dtype=torch.float32, device=DEV)
    qbuf[1:] = q.reshape(-1)
    q_odd = qbuf[1:].view(1, H, d)
    assert q_odd.data_ptr() % 16 != 0
    res = []
    for qq in (q, q_odd):
        idx = torch.full((1, n), -1, dtype=torch.int32, device=DEV)
        cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = torch.zeros(1, H, d, device=DEV)
        vote = torch.zeros(1, ctx.max_tokens, device=DEV)
        ctx.decode_step(qq, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, T.params(k=512, n_local=64, theta=2.0),
                        idx, cnt, out, vote=vote)
        assert ctx.status() == 0
        res.append((idx[0, :int(cnt[0])].cpu().numpy(), out.cpu(), vote[0, :n].cpu()))
    (ia, oa, va), (ib, ob, vb) = res
    rel = ((va.double() - vb.double()).abs() / va.double().abs().clamp_min(1e-30)).max().item()
    assert rel < 1e-5, rel
    if np.array_equal(ia, ib):
        assert (oa - ob).abs().max().item() <= ATTN_REL * max(1.0, oa.abs().max().item())
    else:   # a token within the vote tolerance of the k-th may swap
        assert len(ia) == len(ib) and len(np.setxor1d(ia, ib)) <= 4


@pytest.mark.parametrize("ntie", [1500, 3000])
def test_step_kernel_exact_vote_ties_go_to_the_lower_index(ntie):
    # ntie tokens get the K rows of the highest-vote token: their votes are equal bit for bit
    # and straddle the k-th place (1500: candidates ranked with ties; 3000: more tied tokens
    # than candidates, the last radix level's tie mode). The selection must equal the top-k
    # of the kernel's own votes with ties to the lower index (integer work: exact).
    T = tsl()
    k, s, w = 1024, 4, 64
    sp = W.spec(1, n0=(20011,), steps=1, k=k, n_local=w)
    wl = W.generate(sp, DEV)
    H, Hkv, d, P = sp.n_q_heads, sp.n_kv_heads, sp.head_dim, sp.page_size
    n = int(wl.n0[0])
    seq = torch.tensor([n], dtype=torch.int32, device=DEV)
    q = wl.q[0][0].contiguous()
    prm = T.params(k=k, n_sink=s, n_local=w, theta=2.0)

    def step():
        ctx = T.Context(H, Hkv, d, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
        idx = torch.full((1, n), -1, dtype=torch.int32, device=DEV)
        cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = torch.zeros(1, H, d, device=DEV)
        vote = torch.zeros(1, ctx.max_tokens, device=DEV)
        ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt, out, vote=vote)
        assert ctx.status() == 0
        return idx[0, :int(cnt[0])].cpu().numpy(), vote[0, :n].cpu()

    _, v0 = step()
    src = int(torch.argmax(v0[s:n - w]).item()) + s
    t0 = 6000
    toks = torch.arange(t0, t0 + ntie, device=DEV)
    pages = wl.page_table[0, (toks // P).long()].long()
    sp_ = wl.page_table[0, src // P].long()
    kp = wl.k_pool[0]
    kp[pages, :, (toks % P).long(), :] = kp[sp_, :, src % P, :].unsqueeze(0)
    got, v = step()
    tied = v[t0:t0 + ntie]
    assert bool((tied == tied[0]).all()), "identical keys must give identical votes"
    want, _ = O.select_topk(v.double().numpy(), n, k, s, w)
    assert np.array_equal(got, want)
    # the cut fell inside the tied group: some of it selected, the rest not, lower indices first
    chosen = np.intersect1d(got, np.arange(t0, t0 + ntie))
    assert 0 < len(chosen) < ntie and np.array_equal(chosen, np.arange(t0, t0 + len(chosen)))
