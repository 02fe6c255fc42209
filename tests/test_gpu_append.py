"""ts_append_kv: the current token's K/V rows into the paged pools, through the C ABI."""
import pytest
import torch

import workloads as W
from parity import kv_flag, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("page_size", [16, 1])
@pytest.mark.parametrize("cfg", [0, 2])
def test_append_writes_the_last_position_and_nothing_else(cfg, page_size):
    T = tsl()
    sp = (W.spec(cfg, steps=2, page_size=page_size) if cfg == 0 else
          W.spec(2, n0=(1000, 37, 4096), n0_range=None, batch=3, steps=2, page_size=page_size))
    wl = W.generate(sp, DEV)
    B, Hkv, d = sp.batch, sp.n_kv_heads, sp.head_dim
    ctx = T.Context(sp.n_q_heads, Hkv, d, kv_flag(T, sp), B, wl.page_table.shape[1], wl.num_pages,
                    page_size=sp.page_size)
    dt = wl.k_pool[0].dtype
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    k_new = torch.randn(B, Hkv, d, generator=g, device=DEV).to(dt)
    v_new = torch.randn(B, Hkv, d, generator=g, device=DEV).to(dt)
    kp, vp = wl.k_pool[0].clone(), wl.v_pool[0].clone()
    seq = wl.seq_lens(1)                                # one token more than step 0
    ctx.append_kv(k_new, v_new, wl.page_table, seq, kp, vp)
    assert ctx.status() == 0
    ek, ev = wl.k_pool[0].clone(), wl.v_pool[0].clone()
    for b in range(B):
        pos = int(seq[b]) - 1
        page, slot = int(wl.page_table[b, pos // page_size]), pos % page_size
        ek[page, :, slot, :] = k_new[b]
        ev[page, :, slot, :] = v_new[b]
    assert torch.equal(kp, ek) and torch.equal(vp, ev)
    bad = torch.zeros(B, dtype=torch.int32, device=DEV)   # no token to append
    ctx.append_kv(k_new, v_new, wl.page_table, bad, kp, vp)
    assert ctx.status() == T.STATUS_CODE["TS_ERR_SEQ_LEN"]
    assert torch.equal(kp, ek) and torch.equal(vp, ev)
    ctx.close()
