"""A token-granular pool (one token per page) against the CPU oracle and against 16-token pages.

The method selects and stores single tokens (TokenSelect review, section 3: token-level
KV-cache selection; the paged-KV implementation of section 3.4 can use a page size of one).
A context created with page_size 1 runs the separate kernels: the score kernel fills its
16-token stages from 16 one-token pages, and attention, append and chunk attention address
a row as page_table[b][t], slot 0. Checks:
- trajectories (cache on, hits and misses) against the oracle, which reads the pool's page
  size from its shape;
- bit-identical votes, indices, outputs and lse against the same logical cache held in
  16-token pages, because the stage contents and so every sum are the same;
- a page id outside the pool for one token is reported.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import workloads as W
from parity import GpuRunner, kv_flag, run_trajectory, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _to_page1(wl):
    """The same logical K/V cache of ``wl`` (16-token pages) in a pool of one-token pages,
    laid out by a seeded permutation; returns (k_pools, v_pools, page_table)."""
    P = wl.spec.page_size
    B, n_tok = wl.page_table.shape[0], wl.page_table.shape[1] * P
    toks = []                                   # (b, t) of every cached position
    for b in range(B):
        n_pages = int((wl.page_table[b] >= 0).sum())
        toks.append(n_pages * P)
    total = sum(toks)
    g = torch.Generator(device="cpu")
    g.manual_seed(4242)
    perm = torch.randperm(total, generator=g).to(torch.int32)
    pt1 = torch.full((B, n_tok), -1, dtype=torch.int32)
    src_page = torch.empty(total, dtype=torch.long)
    src_slot = torch.empty(total, dtype=torch.long)
    off = 0
    for b in range(B):
        t = torch.arange(toks[b])
        pt1[b, :toks[b]] = perm[off:off + toks[b]]
        src_page[perm[off:off + toks[b]].long()] = wl.page_table[b, (t // P).to(DEV)].long().cpu()
        src_slot[perm[off:off + toks[b]].long()] = t % P
        off += toks[b]
    sp_, ss = src_page.to(DEV), src_slot.to(DEV)
    kps = [kp[sp_, :, ss, :].unsqueeze(2).contiguous() for kp in wl.k_pool]   # [total][H_kv][1][d]
    vps = [vp[sp_, :, ss, :].unsqueeze(2).contiguous() for vp in wl.v_pool]
    return kps, vps, pt1.to(DEV)


def _page1_workload(sp):
    wl = W.generate(sp, DEV)
    kps, vps, pt1 = _to_page1(wl)
    wl1 = W.Workload(spec=replace(sp, page_size=1), q=wl.q, k_pool=kps, v_pool=vps, page_table=pt1,
                     n0=wl.n0, needle_pos=wl.needle_pos, key_scales=wl.key_scales, rho=wl.rho)
    return wl, wl1


def _report(name, rep):
    print(f"{name}: steps={rep.steps} hits={rep.hits} band_swaps={rep.band_swaps} "
          f"worst_vote_rel={rep.worst_vote_rel:.2e} at_risk={rep.at_risk}")


def test_page1_tiny_fp32_trajectory():
    sp = W.spec(0, page_size=1)
    rep = run_trajectory(W.generate(sp, DEV), 8)
    _report(sp.name, rep)
    assert rep.steps == 8


@pytest.mark.parametrize("cfg", [1, 2])
def test_page1_trajectory_against_the_oracle(cfg):
    # 1: one sequence of 5003 tokens (a ragged last stage); 2: three sequences with GQA 7
    sp = (W.spec(1, n0=(5003,), steps=6, k=512, n_local=128, page_size=1) if cfg == 1 else
          W.spec(2, n0=(4000, 2600, 777), n0_range=None, batch=3, steps=6, k=300, n_local=64, page_size=1))
    rep = run_trajectory(W.generate(sp, DEV), 6)
    _report(sp.name, rep)
    assert rep.steps == 6


def test_page1_topp_against_the_oracle():
    sp = W.spec(4, n0=(3000, 1500), batch=2, steps=4, page_size=1)
    rep = run_trajectory(W.generate(sp, DEV), 4)
    _report(sp.name, rep)
    assert rep.steps == 4


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_page1_bit_identical_to_16_token_pages(cfg):
    sp = {0: W.spec(0, steps=4),
          1: W.spec(1, n0=(9001,), steps=4, k=700, n_local=100),
          2: W.spec(2, n0=(5000, 1234), n0_range=None, batch=2, steps=4, k=256, n_local=64)}[cfg]
    wl16, wl1 = _page1_workload(sp)
    a = GpuRunner(wl16, multi_kernel=True)
    b = GpuRunner(wl1)
    assert a.ctx.max_tokens == wl16.max_tokens and b.ctx.max_tokens == wl1.max_tokens
    for t in range(4):
        ra, rb = a.step(t), b.step(t)
        n = wl16.seq_lens(t).cpu().numpy()
        for i in range(sp.batch):
            assert np.array_equal(ra["vote"][i, :n[i]], rb["vote"][i, :n[i]]), f"step {t} seq {i}: votes"
            assert np.array_equal(ra["idx"][i], rb["idx"][i]), f"step {t} seq {i}: indices"
        for key in ("out", "lse", "hit"):
            assert np.array_equal(ra[key], rb[key]), f"step {t}: {key}"
    a.ctx.close()
    b.ctx.close()


def test_page1_page_outside_the_pool_is_reported():
    T = tsl()
    sp = W.spec(0, steps=1, page_size=1)
    wl = W.generate(sp, DEV)
    pt = wl.page_table.clone()
    pt[0, 100] = wl.num_pages + 3
    r = GpuRunner(wl)
    r.ctx.decode_step(wl.q[0][0], wl.k_pool[0], wl.v_pool[0], pt, wl.seq_lens(0), r.params, r.idx, r.count,
                      r.out, r.lse, hit=r.hit, vote=r.vote, cache=r.cache, layer=0)
    assert r.ctx.status() == T.STATUS_CODE["TS_ERR_PAGE_OOB"]
    r.ctx.close()


def test_page1_128k_against_the_oracle():
    sp = W.spec(1, steps=3, page_size=1)
    rep = run_trajectory(W.generate(sp, DEV), 3)
    _report(sp.name, rep)
    assert rep.steps == 3
