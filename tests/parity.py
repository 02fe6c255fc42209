"""Shared machinery of the GPU parity tests: run a decode trajectory through
the C ABI and through the CPU oracle on the same seeded inputs, and compare.

Tolerances (written here, used by every parity test):

* index sets: identical, except for tokens whose oracle vote lies within
  TIE_REL of the oracle's threshold vote (the k-th candidate, or the top-p
  crossing token); for top-p also a cut position whose oracle cumulative mass
  is within TIE_REL * p * H of p * H. TIE_REL = 1e-6 is the stated tolerance
  of the method's parity target.
* attention output: max_j |o_j - r_j| / max_j |r_j| <= ATTN_REL per (seq, head)
  row, ATTN_REL = 2e-3 (the stated tolerance for bf16 inputs). When the GPU
  set differs from the oracle's only inside the tie band, both are correct
  selections (equal votes may be broken either way within rounding), so the
  GPU output is checked against the definition evaluated on the GPU's set.
* lse: |lse - ref| <= LSE_ABS. fp32 dot products, exp and log over a few
  thousand terms carry a relative error of a few 1e-6 on values below ~100,
  so 1e-3 leaves a wide margin without hiding a wrong term.
* cache decisions: equal, except when |cos - theta| <= COS_BAND, where the
  GPU's decision is replayed in the oracle. The GPU forms the cosine from
  fp32 partial sums of 4096 products (relative error ~1e-7).
* tie-band margin: the set comparison above only means something if the GPU
  decides every token outside the band like the oracle. Each set check
  measures NEAR_ERR, the largest |v_gpu - v| / tau over the tokens whose
  oracle vote lies within NEAR_WIN of tau (the tokens a rounding error could
  move across the cut), and MARGIN, the smallest |v - tau| / tau over the
  tokens outside the band. Tokens outside the band but within
  MARGIN_FACTOR * NEAR_ERR of tau are "at risk": for each of them the check
  compares the GPU's own decision (its vote against its own threshold vote)
  with the oracle's and fails on any difference, and the number of at-risk
  tokens is reported, so a pass never rests on an unexamined token. fp32
  resolution bounds NEAR_ERR from below: near-threshold tokens of these
  workloads take most of their vote from high-scale heads where the logit is
  about 50, and an fp32 logit of 50 is resolved to about 2e-6, so a few
  times 1e-6 relative is the floor of any fp32 pipeline there, above the
  1e-6 band.
* votes: |v_gpu - v| <= VOTE_REL * v elementwise. Each vote is a sum over
  heads of exp(l - L) with l an fp32 dot product of up to 128 bf16*bf16
  products (exact) accumulated in fp32 (16-term chains, then a tree) and
  scaled by an fp32 alpha: the logit error stays below ~1e-6 * (1 + |l|) for
  |l| < 60, so exp(l - L) is off by at most ~6e-5 relative in the worst
  case; 1e-4 bounds it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import oracle as O
import workloads as W

TIE_REL = 1e-6
ATTN_REL = 2e-3
LSE_ABS = 1e-3
COS_BAND = 1e-6
VOTE_REL = 1e-4
NEAR_WIN = 1e-4
MARGIN_FACTOR = 2.0


def tsl():
    import token_level_sparse_gb300 as T
    from token_level_sparse_gb300 import build
    build.build()
    return T


def kv_flag(T, sp):
    return T.TS_KV_F32 if sp.kv_dtype == "f32" else T.TS_KV_BF16


class GpuRunner:
    """Drives ts_decode_step (or the three separate calls) over a workload."""

    def __init__(self, wl: W.Workload, theta=None, cache=True, mode=None, top_p=None, k=None,
                 n_sink=None, n_local=None, separate_calls=False, multi_kernel=False):
        T = tsl()
        self.T = T
        self.wl = wl
        sp = wl.spec
        self.sp = sp
        self.mode = mode or sp.mode
        self.params = T.params(
            mode=T.TS_SELECT_TOPK if self.mode == "topk" else T.TS_SELECT_TOPP,
            k=sp.k if k is None else k, n_sink=sp.n_sink if n_sink is None else n_sink,
            n_local=sp.n_local if n_local is None else n_local,
            top_p=(sp.top_p if top_p is None else top_p) or 0.9,
            theta=sp.theta if theta is None else theta)
        dev = wl.page_table.device
        B = sp.batch
        import os
        prev = os.environ.get("TOKENSELECT_MULTI_KERNEL")
        os.environ["TOKENSELECT_MULTI_KERNEL"] = "1" if multi_kernel else "0"
        try:
            self.ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, kv_flag(T, sp), B,
                                 wl.page_table.shape[1], wl.num_pages, page_size=sp.page_size)
        finally:
            if prev is None:
                del os.environ["TOKENSELECT_MULTI_KERNEL"]
            else:
                os.environ["TOKENSELECT_MULTI_KERNEL"] = prev
        mt = self.ctx.max_tokens
        cap = self.params.k + self.params.n_sink + self.params.n_local if self.mode == "topk" else mt
        self.cache = self.ctx.cache(sp.layers, self.params.k if self.mode == "topk" else mt) if cache else None
        self.idx = torch.full((B, cap), -7, dtype=torch.int32, device=dev)
        self.count = torch.zeros(B, dtype=torch.int32, device=dev)
        self.out = torch.zeros(B, sp.n_q_heads, sp.head_dim, dtype=torch.float32, device=dev)
        self.lse = torch.zeros(B, sp.n_q_heads, dtype=torch.float32, device=dev)
        self.hit = torch.zeros(B, dtype=torch.uint8, device=dev)
        self.vote = torch.zeros(B, mt, dtype=torch.float32, device=dev)
        self.separate = separate_calls

    def step(self, t, l=0):
        wl, T = self.wl, self.T
        seq = wl.seq_lens(t)
        q = wl.q[t][l]
        self.vote.zero_()
        if self.separate:
            self.ctx.score(q, wl.k_pool[l], wl.page_table, seq, self.vote)
            self.ctx.select(self.vote, seq, self.params, self.idx, self.count, cache=self.cache, layer=l, q=q)
            self.ctx.sparse_attend(q, wl.k_pool[l], wl.v_pool[l], wl.page_table, self.idx, self.count,
                                   self.out, self.lse)
            self.hit.zero_()
        else:
            self.ctx.decode_step(q, wl.k_pool[l], wl.v_pool[l], wl.page_table, seq, self.params, self.idx,
                                 self.count, self.out, self.lse, hit=self.hit, vote=self.vote,
                                 cache=self.cache, layer=l)
        st = self.ctx.status()
        assert st == 0, f"device status {T.STATUS.get(st, st)}"
        cnt = self.count.cpu().numpy()
        idx = self.idx.cpu().numpy()
        return dict(hit=self.hit.cpu().numpy().astype(bool), idx=[idx[b, :cnt[b]].copy() for b in range(len(cnt))],
                    out=self.out.cpu().numpy().copy(), lse=self.lse.cpu().numpy().copy(),
                    vote=self.vote.cpu().numpy().copy(), seq=seq.cpu().numpy())


class OracleRunner:
    """The CPU oracle on host copies of the same inputs, one CacheState per (layer, seq)."""

    def __init__(self, wl: W.Workload, layers=None, mode=None, top_p=None, k=None, n_sink=None, n_local=None,
                 theta=None):
        sp = wl.spec
        self.sp = sp
        self.wl = wl
        self.layers = list(range(sp.layers)) if layers is None else layers
        self.kp = {l: W.host_copy(wl.k_pool[l]) for l in self.layers}
        self.vp = {l: W.host_copy(wl.v_pool[l]) for l in self.layers}
        self.pt = W.host_copy(wl.page_table)
        self.state = {(l, b): O.CacheState() for l in self.layers for b in range(sp.batch)}
        self.mode = mode or sp.mode
        self.top_p = (sp.top_p if top_p is None else top_p) or 0.9
        self.k = sp.k if k is None else k
        self.n_sink = sp.n_sink if n_sink is None else n_sink
        self.n_local = sp.n_local if n_local is None else n_local
        self.theta = sp.theta if theta is None else theta
        self.last_miss = {}

    def step(self, t, l, b, force_hit=None):
        q = W.host_copy(self.wl.q[t][l])[b]
        n = self.wl.n0[b] + t
        theta = self.theta
        if force_hit is True:
            theta = -math.inf
        elif force_hit is False:
            theta = math.inf
        r = O.decode_step(self.state[(l, b)], q, self.kp[l], self.vp[l], self.pt[b], n, mode=self.mode,
                          k=self.k, n_sink=self.n_sink, n_local=self.n_local, top_p=self.top_p, theta=theta)
        if not r["hit"]:
            self.last_miss[(l, b)] = dict(vote=r["vote"], n=n, part=r["part"])
        r["n"] = n
        r["q"] = q
        return r


# ------------------------------------------------------------- comparisons

def threshold_topk(vote, n, k, n_sink, n_local):
    s_end, ls = O.budget_segments(n, n_sink, n_local)
    cand = np.arange(s_end, ls)
    if len(cand) <= k or k <= 0:
        return None
    order = cand[np.argsort(-vote[cand], kind="stable")]
    return vote[order[k - 1]]


def band_margin(vote, gpu_vote, tau, n, where="", gpu_set=None, ref_set=None, lo=0, hi=None):
    """(near_err, margin, at_risk) around the threshold vote tau. Every token of the selection
    domain [lo, hi) outside the tie band and within MARGIN_FACTOR * near_err of tau must be in
    the GPU's set exactly when it is in the oracle's."""
    if gpu_vote is None or tau is None or not tau > 0:
        return None
    hi = n if hi is None else hi
    v = vote[:n]
    gv = gpu_vote[:n].astype(np.float64)
    rel = np.abs(v - tau) / tau
    near = rel <= NEAR_WIN
    if not near.any():
        near = rel <= np.sort(rel)[min(63, n - 1)]
    near_err = float(np.max(np.abs(gv[near] - v[near])) / tau)
    out = rel > TIE_REL
    margin = float(rel[out].min()) if out.any() else math.inf
    risk = np.nonzero(out & (rel <= MARGIN_FACTOR * near_err))[0]
    risk = risk[(risk >= lo) & (risk < hi)]
    if risk.size and gpu_set is not None and ref_set is not None:
        wrong = [int(i) for i in risk if (int(i) in gpu_set) != (int(i) in ref_set)]
        assert not wrong, (f"{where}: at-risk tokens decided against the oracle: {wrong[:5]} "
                           f"(rel {[float(rel[i]) for i in wrong[:5]]}, near error {near_err:.2e})")
    return near_err, margin, int(risk.size)


@dataclass
class SetCheck:
    swaps: int
    near_err: float = 0.0
    margin: float = math.inf
    at_risk: int = 0


def check_topk_set(gpu_idx, ref_idx, vote, n, k, n_sink, n_local, where="", gpu_vote=None):
    g, o = set(map(int, gpu_idx)), set(map(int, ref_idx))
    assert len(gpu_idx) == len(g), f"{where}: duplicate indices"
    assert np.all(np.diff(gpu_idx) > 0), f"{where}: not ascending"
    assert len(g) == len(o), f"{where}: count {len(g)} vs oracle {len(o)}"
    tau = threshold_topk(vote, n, k, n_sink, n_local)
    bm = None
    if tau is not None:
        s_end, ls = O.budget_segments(n, n_sink, n_local)
        bm = band_margin(vote, gpu_vote, tau, n, where, g, o, s_end, ls)
    diff = g ^ o
    res = SetCheck(len(diff), *(bm if bm else ()))
    if not diff:
        return res
    assert tau is not None, f"{where}: sets differ although every candidate is taken"
    bad = [i for i in diff if abs(vote[i] - tau) > TIE_REL * tau]
    assert not bad, f"{where}: {len(bad)} tokens differ outside the tie band, e.g. {bad[:5]} " \
                    f"(rel {[abs(vote[i] - tau) / tau for i in bad[:5]]})"
    return res


def check_topp_set(gpu_idx, vote, n, p, H, n_sink, n_local, where="", gpu_vote=None):
    g = set(map(int, gpu_idx))
    assert len(gpu_idx) == len(g) and np.all(np.diff(gpu_idx) > 0), f"{where}: not a strictly ascending set"
    order = np.argsort(-vote[:n], kind="stable")
    cum = np.cumsum(vote[order])
    target = p * H
    s_end, ls = O.budget_segments(n, n_sink, n_local)
    fixed = set(range(s_end)) | set(range(ls, n))
    if p >= 1.0:
        cuts = [n]
        m_o = n
    else:
        m_o = min(n, int(np.searchsorted(cum, target, side="left")) + 1)
        cuts = {m_o}
        near = np.nonzero(np.abs(cum - target) <= TIE_REL * target)[0]
        for j in near:                     # cutting after position j (j+1 tokens) or just before it
            cuts.update({int(j) + 1, int(j) + 2})
        cuts = sorted(c for c in cuts if 1 <= c <= n)
    last_err = None
    for m in cuts:
        exp = fixed | set(map(int, order[:m]))
        diff = g ^ exp
        tau = vote[order[m - 1]]
        bad = [i for i in diff if abs(vote[i] - tau) > TIE_REL * tau]
        if not bad and len(g) == len(exp):
            # the matching cut's threshold: at-risk tokens around it are decided as the oracle does
            bm = band_margin(vote, gpu_vote, tau, n, where, g, exp, s_end, ls) if m < n else None
            return SetCheck(len(diff), *(bm if bm else ()))
        last_err = f"cut {m}: {len(diff)} differ, {len(bad)} outside the band"
    raise AssertionError(f"{where}: top-p set matches no admissible cut ({last_err}); |gpu|={len(g)}")


def check_attention(out, lse, ref_out, ref_lse, where=""):
    for h in range(ref_out.shape[0]):
        den = np.max(np.abs(ref_out[h]))
        err = np.max(np.abs(out[h] - ref_out[h])) / max(den, 1e-30)
        assert err <= ATTN_REL, f"{where} head {h}: attention rel err {err:.3e}"
        assert abs(lse[h] - ref_lse[h]) <= LSE_ABS, f"{where} head {h}: lse {lse[h]} vs {ref_lse[h]}"


def check_vote(gv, ov, n, where=""):
    rel = np.abs(gv[:n] - ov[:n]) / ov[:n]
    worst = float(rel.max())
    assert worst <= VOTE_REL, f"{where}: vote rel err {worst:.3e} at {int(rel.argmax())}"
    return worst


@dataclass
class TrajectoryReport:
    steps: int = 0
    hits: int = 0
    replays: int = 0
    band_swaps: int = 0
    worst_vote_rel: float = 0.0
    near_err: float = 0.0          # largest GPU vote error near a threshold (relative to it)
    margin: float = math.inf       # closest out-of-band token to a threshold (relative)
    at_risk: int = 0               # out-of-band tokens within 2 x near_err, each checked

    def add(self, sc):
        self.band_swaps += sc.swaps
        self.near_err = max(self.near_err, sc.near_err)
        self.margin = min(self.margin, sc.margin)
        self.at_risk += sc.at_risk


def run_trajectory(wl, steps, layers=(0,), theta=None, mode=None, top_p=None, check_votes=True,
                   separate_calls=False, multi_kernel=False, **sel):
    """Steps the GPU and the oracle together and checks every output."""
    sp = wl.spec
    gpu = GpuRunner(wl, theta=theta, mode=mode, top_p=top_p, separate_calls=separate_calls,
                    multi_kernel=multi_kernel, **sel)
    ora = OracleRunner(wl, layers=list(layers), mode=mode, top_p=top_p, theta=theta, **sel)
    rep = TrajectoryReport()
    H = sp.n_q_heads
    for t in range(steps):
        for l in layers:
            g = gpu.step(t, l)
            for b in range(sp.batch):
                where = f"step {t} layer {l} seq {b}"
                q = W.host_copy(wl.q[t][l])[b]
                hit_o, cos_o = O.cache_decision(ora.state[(l, b)], q, ora.theta)
                force = None
                if bool(g["hit"][b]) != hit_o:
                    assert abs(cos_o - ora.theta) <= COS_BAND, \
                        f"{where}: cache decision gpu={g['hit'][b]} oracle={hit_o} cos={cos_o}"
                    force = bool(g["hit"][b])          # replay the GPU's decision
                    rep.replays += 1
                r = ora.step(t, l, b, force_hit=force)
                rep.hits += int(r["hit"])
                lm = ora.last_miss[(l, b)]
                n = r["n"]
                if not r["hit"] and check_votes:
                    rep.worst_vote_rel = max(rep.worst_vote_rel, check_vote(g["vote"][b], r["vote"], n, where))
                if ora.mode == "topk":
                    if r["hit"]:
                        # the cached part came from the last miss: its band decides
                        tau_ref = threshold_topk(lm["vote"], lm["n"], ora.k, ora.n_sink, ora.n_local)
                        gi, oi = set(map(int, g["idx"][b])), set(map(int, r["idx"]))
                        diff = gi ^ oi
                        assert len(gi) == len(oi), f"{where}: hit count {len(gi)} vs {len(oi)}"
                        bad = [i for i in diff if tau_ref is None or abs(lm["vote"][i] - tau_ref) > TIE_REL * tau_ref]
                        assert not bad, f"{where}: hit set differs outside the band: {bad[:5]}"
                        rep.band_swaps += len(diff)
                    else:
                        rep.add(check_topk_set(g["idx"][b], r["idx"], r["vote"], n, ora.k, ora.n_sink,
                                               ora.n_local, where, gpu_vote=g["vote"][b]))
                else:
                    if not r["hit"]:
                        rep.add(check_topp_set(g["idx"][b], r["vote"], n, ora.top_p, H, ora.n_sink,
                                               ora.n_local, where, gpu_vote=g["vote"][b]))
                    else:
                        gi, oi = set(map(int, g["idx"][b])), set(map(int, r["idx"]))
                        if gi != oi:
                            # the cached part may differ by tie-band tokens of the last miss
                            ov = lm["vote"]
                            order = np.argsort(-ov[:lm["n"]], kind="stable")
                            m = len(lm["part"])
                            tau = ov[order[m - 1]]
                            bad = [i for i in gi ^ oi if i >= lm["n"] or abs(ov[i] - tau) > TIE_REL * tau]
                            assert not bad, f"{where}: top-p hit set differs outside the band"
                gi = np.asarray(g["idx"][b])
                if np.array_equal(gi, r["idx"]):
                    check_attention(g["out"][b], g["lse"][b], r["out"], r["lse"], where)
                else:
                    # The sets differ only inside the tie band (checked above): both are
                    # correct selections, so the GPU attention is checked against the
                    # definition evaluated on the GPU's own (valid) set.
                    vo, vl = O.sparse_attention(r["q"], ora.kp[l], ora.vp[l], ora.pt[b], gi)
                    check_attention(g["out"][b], g["lse"][b], vo, vl, where + " (tie-band set)")
            rep.steps += 1
    return rep
