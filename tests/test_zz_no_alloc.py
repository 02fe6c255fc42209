"""The no-alloc sparse attention (ts_sparse_attend_noalloc) against the
context-based ts_sparse_attend, through the C ABI.

ts_sparse_attend_noalloc serves callers that cannot call cudaMalloc (a memory
arena or framework allocator they do not own, or device memory frozen after
start-up): it takes no context and keeps its scratch in a fixed static device
array. This file is collected last so that a failure here does not stop the
rest of a run that halts at the first failure.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity import ATTN_REL, LSE_ABS, check_attention, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs():
    sp = W.spec(1, n0=(20000, 7000), batch=2, steps=1)
    wl = W.generate(sp, DEV)
    rng = np.random.default_rng(11)
    sizes = [2564, 1500]
    idx_np = np.full((2, 2564), -1, dtype=np.int32)
    for b in range(2):
        idx_np[b, :sizes[b]] = np.sort(rng.choice(wl.n0[b], sizes[b], replace=False))
    return sp, wl, torch.from_numpy(idx_np).to(DEV), torch.tensor(sizes, dtype=torch.int32, device=DEV)


def test_noalloc_matches_context_attention_twice():
    T = tsl()
    sp, wl, idx, cnt = _inputs()
    B, H, d = sp.batch, sp.n_q_heads, sp.head_dim
    q = wl.q[0][0]
    ctx = T.Context(H, sp.n_kv_heads, d, T.TS_KV_BF16, B, wl.page_table.shape[1], wl.num_pages)
    ref_out = torch.zeros(B, H, d, device=DEV)
    ref_lse = torch.zeros(B, H, device=DEV)
    ctx.sparse_attend(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, idx, cnt, ref_out, ref_lse)
    assert ctx.status() == 0
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(2):
        out = torch.full((B, H, d), float("nan"), device=DEV)
        lse = torch.full((B, H), float("nan"), device=DEV)
        T.ts_sparse_attend_noalloc(H, sp.n_kv_heads, d, T.TS_KV_BF16, q, wl.k_pool[0], wl.v_pool[0],
                                   wl.num_pages, wl.page_table, wl.page_table.shape[1], idx, idx.stride(0), cnt,
                                   B, 0.0, out, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o, r = out.cpu().numpy(), ref_out.cpu().numpy()
        for b in range(B):
            for h in range(H):
                err = np.max(np.abs(o[b, h] - r[b, h])) / np.max(np.abs(r[b, h]))
                assert err <= ATTN_REL, (call, b, h, err)
        assert np.max(np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy())) <= LSE_ABS


def test_noalloc_at_its_batch_limit_against_the_oracle():
    # B = 48, the largest batch the fixed array serves (partials of 48 x 8 KV heads x 4 heads x
    # 130 floats per split): two calls in a row, each checked against the CPU oracle's
    # definition of the sparse attention
    T = tsl()
    B = 48
    sp = W.spec(1, n0=tuple(600 + 37 * b for b in range(B)), batch=B, steps=1, needles="lnN2")
    wl = W.generate(sp, DEV)
    rng = np.random.default_rng(48)
    cap = 400
    idx_np = np.full((B, cap), -1, dtype=np.int32)
    sizes = []
    for b in range(B):
        m = int(rng.integers(1, cap + 1))
        idx_np[b, :m] = np.sort(rng.choice(wl.n0[b], m, replace=False))
        sizes.append(m)
    idx = torch.from_numpy(idx_np).to(DEV)
    cnt = torch.tensor(sizes, dtype=torch.int32, device=DEV)
    q = wl.q[0][0]
    kp, vp, pt, qh = (W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0]), W.host_copy(wl.page_table),
                      W.host_copy(q))
    refs = [O.sparse_attention(qh[b], kp, vp, pt[b], idx_np[b, :sizes[b]]) for b in range(B)]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(2):
        out = torch.full((B, sp.n_q_heads, sp.head_dim), float("nan"), device=DEV)
        lse = torch.full((B, sp.n_q_heads), float("nan"), device=DEV)
        T.ts_sparse_attend_noalloc(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, q, wl.k_pool[0],
                                   wl.v_pool[0], wl.num_pages, wl.page_table, wl.page_table.shape[1], idx,
                                   idx.stride(0), cnt, B, 0.0, out, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o, l_ = out.cpu().numpy(), lse.cpu().numpy()
        for b in range(B):
            check_attention(o[b], l_[b], refs[b][0], refs[b][1], f"call {call} seq {b}")


def test_noalloc_rejects_a_nan_scale():
    T = tsl()
    sp, wl, idx, cnt = _inputs()
    out = torch.zeros(sp.batch, sp.n_q_heads, sp.head_dim, device=DEV)
    with pytest.raises(T.TokenSelectError) as e:
        T.ts_sparse_attend_noalloc(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, wl.q[0][0],
                                   wl.k_pool[0], wl.v_pool[0], wl.num_pages, wl.page_table,
                                   wl.page_table.shape[1], idx, idx.stride(0), cnt, sp.batch, float("nan"), out)
    assert e.value.status == T.STATUS_CODE["TS_ERR_INVALID_ARG"]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T = tsl()
    sp, wl, idx, cnt = _inputs()
    out = torch.zeros(49, sp.n_q_heads, sp.head_dim, device=DEV)
    with pytest.raises(T.TokenSelectError) as e:
        T.ts_sparse_attend_noalloc(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, wl.q[0][0],
                                   wl.k_pool[0], wl.v_pool[0], wl.num_pages, wl.page_table,
                                   wl.page_table.shape[1], idx, idx.stride(0), cnt, 49, 0.0, out)
    assert e.value.status == T.STATUS_CODE["TS_ERR_SCRATCH_LIMIT"]
