"""The time-out path of the persistent decode-step kernel, exercised without a fault.

Every wait of the kernel is bounded; when one runs out the kernel records
TS_ERR_TIMEOUT, raises the abort word, drains its own copies, frees its tensor
memory and returns. Here the run-out is made on the host's request: for one
launch, one CTA leaves at a grid barrier without arriving
(ts_inject_barrier_skip), with a 1 ms wait limit (ts_set_wait_limit), so the
other CTAs' bounded barrier wait runs out. Nothing traps, faults or hangs: a
missing arrival is exactly the condition the bounded wait exists for. The test
then checks that the next launch on the same context starts from clean barrier
words and gives bit-identical results to a fresh context.
"""
import pytest
import torch

import workloads as W
from parity import kv_flag, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _setup(T, wl, sp):
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, kv_flag(T, sp), sp.batch,
                    wl.page_table.shape[1], wl.num_pages)
    B = sp.batch
    cap = sp.k + sp.n_sink + sp.n_local
    bufs = dict(idx=torch.full((B, cap), -1, dtype=torch.int32, device=DEV),
                count=torch.zeros(B, dtype=torch.int32, device=DEV),
                out=torch.zeros(B, sp.n_q_heads, sp.head_dim, device=DEV),
                lse=torch.zeros(B, sp.n_q_heads, device=DEV),
                vote=torch.zeros(B, ctx.max_tokens, device=DEV))
    return ctx, bufs


def _step(T, ctx, wl, sp, bufs, prm):
    ctx.decode_step(wl.q[0][0], wl.k_pool[0], wl.v_pool[0], wl.page_table, wl.seq_lens(0), prm,
                    bufs["idx"], bufs["count"], bufs["out"], bufs["lse"], vote=bufs["vote"])


@pytest.mark.parametrize("barrier", [0, 1, 2])
def test_bounded_barrier_wait_runs_out_and_the_next_launch_is_clean(barrier):
    T = tsl()
    sp = W.spec(1, n0=(30011,), steps=1, k=512, n_local=64)
    wl = W.generate(sp, DEV)
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)

    ref_ctx, ref = _setup(T, wl, sp)
    _step(T, ref_ctx, wl, sp, ref, prm)
    assert ref_ctx.status() == 0

    ctx, bufs = _setup(T, wl, sp)
    T.ts_set_wait_limit(ctx.handle, 1_000_000)          # 1 ms
    T.ts_inject_barrier_skip(ctx.handle, 5, barrier)    # CTA 5 leaves at that barrier, this launch only
    _step(T, ctx, wl, sp, bufs, prm)
    st = ctx.status()
    assert st == T.STATUS_CODE["TS_ERR_TIMEOUT"], T.STATUS.get(st, st)

    # the context is usable: the next launch passes every barrier and matches a fresh context
    for name in bufs:
        bufs[name].zero_()
    _step(T, ctx, wl, sp, bufs, prm)
    assert ctx.status() == 0
    for name in ("idx", "count", "out", "lse", "vote"):
        assert torch.equal(bufs[name], ref[name]), f"{name} differs from a fresh context after the time-out"
    ctx.close()
    ref_ctx.close()


def test_wait_limit_rejects_zero():
    T = tsl()
    sp = W.spec(0)
    wl = W.generate(sp, DEV)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_F32, 1, wl.page_table.shape[1],
                    wl.num_pages)
    with pytest.raises(T.TokenSelectError):
        T.ts_set_wait_limit(ctx.handle, 0)
    ctx.close()
