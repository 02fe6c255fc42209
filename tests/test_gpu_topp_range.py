"""Top-p attention in the persistent kernel: the range attention against the gathered one and the oracle.

Top-p can keep most of a sequence (SeqO1, section 3.2: the cumulative-importance rule adapts the
budget to how flat the votes are). The persistent kernel then attends each CTA's own scanned
range from the scan's logits, streaming whole V pages (`range`, P.V on CUDA cores), or with P.V
on the tensor cores for bf16 pools with d = 128 (`range_tc`, on request).
Sparse selections keep the gathered attention, where the selected tokens are shared out evenly
over all CTAs (`gather`). TOKENSELECT_TOPP_ATTEND, read when the context is created, forces one
path for these tests.
Checks:
- trajectories against the oracle on each path (votes, index sets in the tie band, outputs
  within 2e-3 per row, lse within 1e-3);
- the same step on both paths gives the same index sets and outputs within the tolerance;
- cache hits of dense selections take the range attention too (the cached part, sinks and window
  over an even split of the pages, logits computed from K): against the oracle and the gathered
  attention over trajectories with hits;
- keys whose norms cycle over every four pages move the running max on many pages (the
  rescale path), against the oracle;
- the geometries of the other workloads (GQA 7 with 4 KV heads; fp32 pools with d = 64).
"""
import numpy as np
import pytest
import torch

import workloads as W
from parity import GpuRunner, check_attention, run_trajectory, tsl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _set_path(monkeypatch, path):
    if path == "auto":
        monkeypatch.delenv("TOKENSELECT_TOPP_ATTEND", raising=False)
    else:
        monkeypatch.setenv("TOKENSELECT_TOPP_ATTEND", path)


def _report(name, rep):
    print(f"{name}: steps={rep.steps} hits={rep.hits} band_swaps={rep.band_swaps} "
          f"worst_vote_rel={rep.worst_vote_rel:.2e} at_risk={rep.at_risk}")


@pytest.mark.parametrize("path", ["range", "range_tc", "gather", "auto"])
def test_topp_paths_against_the_oracle(path, monkeypatch):
    _set_path(monkeypatch, path)
    for p in (0.9, 0.99):
        sp = W.spec(4, n0=(6000, 6000, 7000, 9000), steps=3, top_p=p)
        rep = run_trajectory(W.generate(sp, DEV), 3)
        _report(f"{path} p={p}", rep)


@pytest.mark.parametrize("path", ["range", "range_tc", "gather"])
def test_topp_every_token_on_both_paths(path, monkeypatch):
    _set_path(monkeypatch, path)
    sp = W.spec(4, n0=(300, 4000, 17, 2500), steps=1, top_p=1.0, needles="lnN2")
    rep = run_trajectory(W.generate(sp, DEV), 1, theta=2.0)
    _report(path, rep)


def test_topp_paths_agree(monkeypatch):
    sp = W.spec(4, n0=(20000, 5000, 33000, 12000), steps=4, top_p=0.9)
    wl = W.generate(sp, DEV)
    res = {}
    for path in ("gather", "range", "range_tc"):
        _set_path(monkeypatch, path)
        r = GpuRunner(wl, theta=2.0)
        res[path] = [r.step(t) for t in range(4)]
        r.ctx.close()
    for other in ("range", "range_tc"):
        for t in range(4):
            a, b = res["gather"][t], res[other][t]
            for i in range(sp.batch):
                where = f"{other} step {t} seq {i}"
                assert np.array_equal(a["idx"][i], b["idx"][i]), f"{where}: index sets differ"
                check_attention(b["out"][i], b["lse"][i], a["out"][i], a["lse"][i], where)


@pytest.mark.parametrize("path", ["range", "gather", "auto"])
def test_topp_hits_against_the_oracle(path, monkeypatch):
    # theta 0.9 on a slowly drifting query: most steps hit, and p = 0.95 keeps most tokens
    _set_path(monkeypatch, path)
    sp = W.spec(4, n0=(20000, 5000, 33000, 2100), steps=6, top_p=0.95, rho=0.995)
    rep = run_trajectory(W.generate(sp, DEV), 6)
    _report(path, rep)
    assert rep.hits >= 8


def test_topp_hit_paths_agree(monkeypatch):
    sp = W.spec(4, n0=(20000, 5000, 33000, 12000), steps=5, top_p=0.9, rho=0.995)
    wl = W.generate(sp, DEV)
    res = {}
    for path in ("gather", "range"):
        _set_path(monkeypatch, path)
        r = GpuRunner(wl)
        res[path] = [r.step(t) for t in range(5)]
        r.ctx.close()
    nhit = 0
    for t in range(5):
        a, b = res["gather"][t], res["range"][t]
        assert np.array_equal(a["hit"], b["hit"]), f"step {t}: cache decisions differ"
        for i in range(sp.batch):
            where = f"step {t} seq {i} hit={bool(a['hit'][i])}"
            assert np.array_equal(a["idx"][i], b["idx"][i]), f"{where}: index sets differ"
            check_attention(b["out"][i], b["lse"][i], a["out"][i], a["lse"][i], where)
            nhit += int(a["hit"][i])
    assert nhit >= 8


@pytest.mark.parametrize("path", ["range", "range_tc", "gather"])
def test_topp_growing_keys_rescale(path, monkeypatch):
    # key norms cycle 0.05, 1, 3, 6 over every four pages: within each CTA's range the logits'
    # max jumps by more than the rescale gap several times, so the range attention moves its
    # running max (and rescales its sums and outputs) on many pages
    _set_path(monkeypatch, path)
    sp = W.spec(4, n0=(9000, 3000), batch=2, steps=2, top_p=0.95, needles="lnN2", key_scale="unit")
    wl = W.generate(sp, DEV)
    cyc = torch.tensor([0.05, 1.0, 3.0, 6.0], device=DEV)
    for b in range(sp.batch):
        npg = -(-(wl.n0[b] + sp.steps) // sp.page_size)
        pages = wl.page_table[b, :npg].long()
        f = cyc[torch.arange(npg, device=DEV) % 4]
        kp = wl.k_pool[0]
        kp[pages] = (kp[pages].float() * f.view(-1, 1, 1, 1)).to(kp.dtype)
    rep = run_trajectory(wl, 2, theta=2.0)
    _report(path, rep)


@pytest.mark.parametrize("path", ["range", "range_tc", "gather"])
def test_topp_qwen_geometry(path, monkeypatch):
    _set_path(monkeypatch, path)
    sp = W.spec(2, n0=(7000, 3100, 12000), n0_range=None, batch=3, steps=3, mode="topp", top_p=0.9,
                needles="topp_mix")
    rep = run_trajectory(W.generate(sp, DEV), 3)
    _report(path, rep)


@pytest.mark.parametrize("path", ["range", "gather"])
def test_topp_fp32_small_heads(path, monkeypatch):
    _set_path(monkeypatch, path)
    sp = W.spec(0, steps=4, mode="topp", top_p=0.9, n0=(1024,))
    rep = run_trajectory(W.generate(sp, DEV), 4)
    _report(path, rep)


@pytest.mark.parametrize("theta", [2.0, 0.9])
def test_topp_range_page_outside_the_pool_is_reported(theta, monkeypatch):
    # one sequence's page table names a page past the pool on a miss step (theta 2.0) and on a
    # dense hit (theta 0.9, the cached query again): the range attention skips the page and the
    # status reports it; the next step on a valid table is clean
    _set_path(monkeypatch, "range")
    T = tsl()
    sp = W.spec(4, n0=(3000, 1500, 700, 4000), steps=2, top_p=1.0, needles="lnN2")
    wl = W.generate(sp, DEV)
    r = GpuRunner(wl, theta=theta)
    r.step(0)                                          # fills the cache (a miss)
    bad = wl.page_table.clone()
    bad[1, 5] = wl.num_pages + 7
    r.ctx.decode_step(wl.q[0][0], wl.k_pool[0], wl.v_pool[0], bad, wl.seq_lens(0), r.params, r.idx, r.count,
                      r.out, r.lse, hit=r.hit, vote=r.vote, cache=r.cache, layer=0)
    assert r.ctx.status() == T.STATUS_CODE["TS_ERR_PAGE_OOB"]
    if theta <= 1.0:
        assert bool(r.hit.cpu().numpy().all())         # the same query: every sequence hit
    g = r.step(1)                                      # asserts a clean status
    assert np.all(np.isfinite(g["out"]))
    r.ctx.close()
