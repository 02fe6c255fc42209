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

import workloads as W
from parity import ATTN_REL, LSE_ABS, tsl

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


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T = tsl()
    sp, wl, idx, cnt = _inputs()
    out = torch.zeros(49, sp.n_q_heads, sp.head_dim, device=DEV)
    with pytest.raises(T.TokenSelectError) as e:
        T.ts_sparse_attend_noalloc(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, wl.q[0][0],
                                   wl.k_pool[0], wl.v_pool[0], wl.num_pages, wl.page_table,
                                   wl.page_table.shape[1], idx, idx.stride(0), cnt, 49, 0.0, out)
    assert e.value.status == T.STATUS_CODE["TS_ERR_SCRATCH_LIMIT"]
