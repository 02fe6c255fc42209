"""Plain fp64 CPU oracle of the TokenSelect decode step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports or runs this
module; ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline/reference
legs of ``bench.py`` are its only callers. It shares no code with the CUDA
library: it reads the same host copies of the seeded inputs and nothing else.

Every function is the written-out definition, in float64, in the order the
pages give it. Sources (page title, then section / equation):

* [TS-notes]  "TokenSelect: Efficient Long-Context Inference and Length
  Extrapolation for LLMs via Dynamic Token-Level KV Cache Selection"
  (papercache deep notes): "Formalising selective sparse attention"
  (equations for O and O-hat), "Evolution of the selection function",
  "Head soft vote" (equation T_head-soft-vote), "Selection Cache" and
  Appendix Algorithm 1, Appendix Algorithm 2 (Paged Dot Product Kernel).
* [TS-review] "TokenSelect: smashing block-level KV selection down to the
  token level" (ai-paper-analysis review): section 3.1 (head soft vote),
  section 3.2 (Algorithm 1, Selection Cache), figure 4 (page size 1, indices
  only), section 4.2 (the 2K selected + 512 local budget).
* [SeqO1]     SequenceO1 blog, section 3.2 (keep the tokens whose cumulative
  importance reaches a fraction p) - used for the top-p variant only.

Readings where the pages are silent or garbled:

R1  The vote softmax uses the attention scale alpha = 1/sqrt(d) (the printed
    vote omits it; the attention equations carry it). alpha is a parameter.
R2  Each head's softmax runs over all N cached tokens, sinks and window included.
R3  Top-k runs over the candidates [s, N-w) only; the result is then unioned
    with the sinks [0, s) and the local window [N-w, N), so the set has
    exactly k+s+w tokens when N >= k+s+w ("2K+512").
R4  Top-p sorts all N tokens by (vote desc, index asc) and keeps the shortest
    prefix whose vote mass reaches p*H (the crossing token included); p >= 1
    keeps every token. The prefix is then unioned with sinks and window.
R5  GQA: query head h reads KV head h // G, G = H / H_kv; the vote sums all H
    query heads; one index set serves all heads of a (sequence, layer).
R6  Algorithm 1 compares the query with C_Q, the query of the last miss (C_Q
    is only written on a miss); cos >= theta is a hit. The cosine is taken
    over the concatenated H*d query. A zero-norm query is a miss.
R7  A hit reuses only the selected part C_T; sinks and window are rebuilt at
    the current N and the union is deduplicated.
R8  Ties in the vote go to the lower token index. Index sets are returned in
    ascending order.
R9  The current token is the last cached position N-1, so the window holds it.
R10 The plain TopK selection function TopK(Q . K_cache^T) scores token i by the
    dot product of the concatenated multi-head query with the token's
    concatenated keys, i.e. the sum over query heads of the (scaled) per-head
    logits: the reading that makes it "dominated by the heads with the largest
    logit norms", as the pages say it is.
R12 Chunk-wise prefill selection: the cache already holds the chunk's c tokens
    (length n, the chunk at positions n-c .. n-1); the c queries are averaged
    into one query, which selects once (head soft vote, top-k over [s, n-w),
    united with sinks and window, no Selection Cache in prefill); chunk query
    i then attends causally to the selected tokens at positions <= n-c+i.
R13 Lemma 1 (TS-notes, Appendix C): for one query head and dot-product top-k,
    writing q2/|q2| = (q1/|q1|) cos t + p sin t with p a unit vector orthogonal
    to q1, every score of q2 is |q2| (cos t . s1_i + sin t . p.k_i) with
    s1_i = (q1/|q1|).k_i and |p.k_i| <= R = max_i |k_i|. The top-k cannot
    change while cos t . D > 2 R sin t, D the gap between the k-th and the
    (k+1)-th s1: the sufficient threshold is eps = 2R / sqrt(D^2 + 4R^2)
    (the constant the pages' proof arrives at is not legible; this is the
    plainest one the decomposition gives).
R14 Block-level selection (the contrast of TS-review figure 2(b), InfLLM-style):
    the n tokens form blocks of `block` consecutive tokens (the last one
    ragged); a block's score is the largest vote of its tokens (a block is
    taken as soon as one of its tokens matters, as the review describes);
    the budget // block best blocks are taken (ties to the lower block) and
    every token of them is selected. Recall@m of a selection is the share of
    the m best tokens by vote (ties to the lower index) that it holds.
R11 The head hard vote counts, per token, the query heads whose own TopK
    (k tokens, over the same candidates [s, N-w) as R3, ties to the lower
    index) contains it, then takes the TopK of the counts (ties to the lower
    index).

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "as_f64", "gather_rows", "head_logits", "soft_vote", "log_normalisers",
    "budget_segments", "select_topk", "select_topp", "refresh_hit",
    "sparse_attention", "dense_attention", "cosine", "CacheState",
    "cache_decision", "decode_step", "default_scale", "logit_sum_scores",
    "hard_vote_counts", "selection_scores", "SCORE_FNS", "prefill_chunk", "lemma1_epsilon",
    "selection_overlap", "select_blocks", "recall_at",
]


# --------------------------------------------------------------------- data

def as_f64(x: np.ndarray) -> np.ndarray:
    """Exact float64 copy of a KV-pool slice.

    ``uint16`` arrays are bf16 bit patterns: a bf16 value is the top half of
    the float32 with the same bits, so widening is a 16-bit shift.
    """
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def gather_rows(pool: np.ndarray, page_row: np.ndarray, tokens: np.ndarray, g: int) -> np.ndarray:
    """Rows of KV head ``g`` for logical ``tokens`` of one sequence, in float64.

    Paged layout (TS-notes, "Paged Dot Product Kernel design": logically
    contiguous tokens are not physically contiguous): token i of the sequence
    sits in physical page ``page_row[i // P]`` at slot ``i % P``.
    """
    P = pool.shape[2]
    tokens = np.asarray(tokens, dtype=np.int64)
    pages = np.asarray(page_row, dtype=np.int64)[tokens // P]
    if pages.size and (pages.min() < 0 or pages.max() >= pool.shape[0]):
        raise ValueError("page table entry outside the pool")
    return as_f64(pool[pages, g, tokens % P, :])


def default_scale(head_dim: int) -> float:
    """alpha = 1/sqrt(d) (TS-notes, equations for O and O-hat; reading R1)."""
    return 1.0 / math.sqrt(head_dim)


# ----------------------------------------------------------- score and vote

def head_logits(q: np.ndarray, k_pool: np.ndarray, page_row: np.ndarray, n: int,
                scale: Optional[float] = None) -> np.ndarray:
    """l[h, i] = alpha * <q_h, K_{g(h), i}> for the n cached tokens.

    Per-head criticality of every cached token (TS-notes, "Head soft vote":
    Q^h . K_cache^h^T; Appendix Algorithm 2: s = <q, k> per head and token).
    GQA mapping g(h) = h // G (reading R5). Each logit is its own row-wise dot
    product, so equal keys give equal logits and ties stay ties (reading R8).
    """
    q = np.asarray(q, dtype=np.float64)
    H, d = q.shape
    Hkv = k_pool.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    G = H // Hkv
    alpha = default_scale(d) if scale is None else float(scale)
    tokens = np.arange(n)
    out = np.empty((H, n))
    for g in range(Hkv):
        K = gather_rows(k_pool, page_row, tokens, g)          # [n, d]
        for j in range(G):
            h = g * G + j
            out[h] = alpha * np.einsum("nd,d->n", K, q[h])
    return out


def log_normalisers(logits: np.ndarray) -> np.ndarray:
    """L_h = log sum_i exp(l[h, i]), with the max shifted out (reading R2)."""
    m = logits.max(axis=1)
    return m + np.log(np.exp(logits - m[:, None]).sum(axis=1))


def soft_vote(logits: np.ndarray) -> np.ndarray:
    """v_i = sum_h softmax_h(l[h, :])_i.

    Head soft vote (TS-notes, "Head soft vote", equation T_head-soft-vote;
    TS-review section 3.1): normalise each head with its own softmax, then sum
    over the heads. The vote sums to H.
    """
    L = log_normalisers(logits)
    v = np.zeros(logits.shape[1])
    for h in range(logits.shape[0]):
        v += np.exp(logits[h] - L[h])
    return v


# ---------------------------------------------------------------- selection

def budget_segments(n: int, n_sink: int, n_local: int):
    """(end of sinks, start of local window) for a sequence of n tokens.

    Budget = k selected + sink tokens + local window (TS-review section 4.2,
    "2K+512"; reading R3). Sinks are [0, s_end), the window [local_start, n),
    the top-k candidates [s_end, local_start).
    """
    s_end = min(n_sink, n)
    local_start = max(s_end, n - n_local)
    return s_end, local_start


def _union_fixed(part: np.ndarray, n: int, n_sink: int, n_local: int) -> np.ndarray:
    s_end, local_start = budget_segments(n, n_sink, n_local)
    fixed = np.concatenate([np.arange(s_end), np.arange(local_start, n)])
    return np.union1d(fixed, np.asarray(part, dtype=np.int64)).astype(np.int64)


def _order_desc(vote: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """tokens sorted by (vote desc, index asc): a stable sort of -vote (reading R8)."""
    return tokens[np.argsort(-vote[tokens], kind="stable")]


def select_topk(vote: np.ndarray, n: int, k: int, n_sink: int, n_local: int):
    """TopK of the vote over the candidates, unioned with sinks and window.

    TS-notes, "Head soft vote" (TopK of the summed vote); reading R3. Returns
    (index set ascending, selected part ascending).
    """
    s_end, local_start = budget_segments(n, n_sink, n_local)
    cand = np.arange(s_end, local_start)
    part = np.sort(_order_desc(vote, cand)[:max(0, k)])
    return _union_fixed(part, n, n_sink, n_local), part


def select_topp(vote: np.ndarray, n: int, top_p: float, total_mass: float,
                n_sink: int, n_local: int):
    """Smallest (vote desc, index asc) prefix of all n tokens with mass >= p*H.

    Dynamic-budget variant (SeqO1 section 3.2: keep the tokens whose
    cumulative importance reaches the fraction p of the total); reading R4.
    Returns (index set ascending, selected part ascending).
    """
    order = _order_desc(vote, np.arange(n))
    if top_p >= 1.0 or n == 0:
        take = n
    else:
        cum = np.cumsum(vote[order])
        target = top_p * total_mass
        j = int(np.searchsorted(cum, target, side="left"))     # first cum >= target
        take = min(n, j + 1)
    part = np.sort(order[:take])
    return _union_fixed(part, n, n_sink, n_local), part


def refresh_hit(part: np.ndarray, n: int, n_sink: int, n_local: int) -> np.ndarray:
    """Index set on a cache hit: cached part united with the current sinks and window (R7)."""
    return _union_fixed(part, n, n_sink, n_local)


# ------------------------------------------------ selection-function ablations

def logit_sum_scores(logits: np.ndarray) -> np.ndarray:
    """s_i = sum_h l[h, i]: the plain TopK selection function's score (reading R10).

    TS-notes, "Evolution of the selection function": T_topk = TopK(Q . K_cache^T),
    the dot product of the current query with the cached keys; over all heads
    at once that is the concatenated query against the concatenated keys, the
    sum of the per-head logits. TS-review section 3.1: dominated by high-norm
    heads.
    """
    return np.asarray(logits, dtype=np.float64).sum(axis=0)


def hard_vote_counts(logits: np.ndarray, n: int, k: int, n_sink: int, n_local: int) -> np.ndarray:
    """c_i = sum_h [i in TopK_k(l[h, candidates])] (reading R11).

    TS-notes, "Evolution of the selection function": T_head-vote =
    TopK(sum_h I(i in TopK(Q^h . K_cache^h^T))), a 0/1 vote of every head's own
    top-k. Each head's TopK runs over the candidates [s, N-w) with ties to the
    lower index; tokens outside the candidates get no vote.
    """
    s_end, local_start = budget_segments(n, n_sink, n_local)
    cand = np.arange(s_end, local_start)
    counts = np.zeros(n)
    for h in range(logits.shape[0]):
        top = _order_desc(logits[h], cand)[:max(0, k)]
        counts[top] += 1.0
    return counts


SCORE_FNS = ("soft_vote", "logit_sum", "hard_vote")


def selection_scores(logits: np.ndarray, score_fn: str, n: int, k: int, n_sink: int, n_local: int):
    """The per-token score whose TopK is the selection: head soft vote (the method's),
    or one of the two selection functions it is compared with (TS-notes, "Evolution of
    the selection function"; TS-review section 4.4, table 4)."""
    if score_fn == "soft_vote":
        return soft_vote(logits)
    if score_fn == "logit_sum":
        return logit_sum_scores(logits)
    if score_fn == "hard_vote":
        return hard_vote_counts(logits, n, k, n_sink, n_local)
    raise ValueError(score_fn)


# ---------------------------------------------------------------- attention

def sparse_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                     page_row: np.ndarray, idx: np.ndarray, scale: Optional[float] = None):
    """O-hat_h = softmax(alpha q_h K_sel^T) V_sel for every query head h.

    TS-notes, "Formalising selective sparse attention", equation for O-hat
    (the selected keys include the current token, reading R9). Returns
    (out [H, d], lse [H]) with lse_h = log sum_{i in idx} exp(alpha q_h.k_i).
    """
    q = np.asarray(q, dtype=np.float64)
    H, d = q.shape
    Hkv = k_pool.shape[1]
    G = H // Hkv
    alpha = default_scale(d) if scale is None else float(scale)
    idx = np.asarray(idx, dtype=np.int64)
    out = np.zeros((H, d))
    lse = np.full(H, -np.inf)
    if idx.size == 0:
        return out, lse
    for g in range(Hkv):
        K = gather_rows(k_pool, page_row, idx, g)
        V = gather_rows(v_pool, page_row, idx, g)
        for j in range(G):
            h = g * G + j
            s = alpha * (K @ q[h])
            m = s.max()
            e = np.exp(s - m)
            Z = e.sum()
            out[h] = (e @ V) / Z
            lse[h] = m + math.log(Z)
    return out, lse


def dense_attention(q, k_pool, v_pool, page_row, n, scale=None):
    """O: the same attention over every cached token (TS-notes, equation for O)."""
    return sparse_attention(q, k_pool, v_pool, page_row, np.arange(n), scale)


# ---------------------------------------------------------- selection cache

def cosine(a: np.ndarray, b: np.ndarray) -> float:
    """cos(a, b) over the flattened vectors; 0-norm gives nan."""
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na = math.sqrt(float(a @ a))
    nb = math.sqrt(float(b @ b))
    if na == 0.0 or nb == 0.0:
        return float("nan")
    return float(a @ b) / (na * nb)


@dataclass
class CacheState:
    """Selection Cache of one (sequence, layer): first-query flag, C_Q, C_T."""

    first: bool = True
    cq: Optional[np.ndarray] = None
    ct: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))


def cache_decision(state: CacheState, q: np.ndarray, theta: float):
    """(hit, cos) of Algorithm 1 (TS-notes Appendix Algorithm 1; TS-review 3.2).

    Miss when this is the first query or cos(Q, C_Q) < theta; a hit otherwise
    (equality is a hit). Reading R6.
    """
    if state.first:
        return False, float("nan")
    c = cosine(q, state.cq)
    if math.isnan(c):
        return False, c
    return c >= theta, c


def decode_step(state: CacheState, q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                page_row: np.ndarray, n: int, *, mode: str = "topk", k: int = 2048,
                n_sink: int = 4, n_local: int = 512, top_p: float = 0.9,
                theta: float = 0.9, scale: Optional[float] = None,
                score_fn: str = "soft_vote") -> dict:
    """One decode step of one (sequence, layer): cache check, score, select, attend.

    TS-notes, "TokenSelect overall flow" (paged dot product -> head soft vote
    -> paged attention over the selected tokens) wrapped in Algorithm 1. On a
    miss the cache takes the new selected part and the query; on a hit the
    cached part is reused. score_fn selects the selection function: the head soft
    vote (default) or one of the ablations (logit_sum, hard_vote; top-k only).
    """
    q = np.asarray(q, dtype=np.float64)
    if score_fn != "soft_vote" and mode != "topk":
        raise ValueError("the ablation selection functions are defined for top-k only")
    hit, c = cache_decision(state, q, theta)
    res = {"hit": hit, "cos": c}
    if hit:
        part = state.ct
        idx = refresh_hit(part, n, n_sink, n_local)
    else:
        logits = head_logits(q, k_pool, page_row, n, scale)
        vote = selection_scores(logits, score_fn, n, k, n_sink, n_local)
        if mode == "topk":
            idx, part = select_topk(vote, n, k, n_sink, n_local)
        elif mode == "topp":
            idx, part = select_topp(vote, n, top_p, float(q.shape[0]), n_sink, n_local)
        else:
            raise ValueError(mode)
        state.first = False
        state.cq = q.copy()
        state.ct = part
        res["vote"] = vote
        res["logits_L"] = log_normalisers(logits)
    out, lse = sparse_attention(q, k_pool, v_pool, page_row, idx, scale)
    res.update(idx=idx, part=part, out=out, lse=lse)
    return res


# ---------------------------------------------------- chunk-wise prefill (R12)

def prefill_chunk(q_chunk: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, page_row: np.ndarray,
                  n: int, *, k: int = 2048, n_sink: int = 4, n_local: int = 512,
                  scale: Optional[float] = None) -> dict:
    """One chunk of c prefill queries: one selection from their mean, causal sparse attention.

    TS-notes, "Optimising the selection frequency of the prefill stage": the c
    queries of a chunk Q_C are averaged, (1/c) sum_i (Q_C)_i, and that mean
    query goes through the selection function once; the chunk shares the
    result. TS-review section 3.2 (closing paragraph): prefill uses no
    Selection Cache. Reading R12 places the chunk at the end of the n cached
    tokens and masks each query causally. Returns the index set (ascending),
    out [c, H, d], lse [c, H] and the mean query's vote.
    """
    q_chunk = np.asarray(q_chunk, dtype=np.float64)
    c = q_chunk.shape[0]
    if not 1 <= c <= n:
        raise ValueError("the chunk must hold 1..n queries")
    q_mean = q_chunk.sum(axis=0) / c
    vote = soft_vote(head_logits(q_mean, k_pool, page_row, n, scale))
    idx, part = select_topk(vote, n, k, n_sink, n_local)
    H, d = q_chunk.shape[1], q_chunk.shape[2]
    out = np.zeros((c, H, d))
    lse = np.full((c, H), -np.inf)
    for i in range(c):
        visible = idx[idx <= n - c + i]
        out[i], lse[i] = sparse_attention(q_chunk[i], k_pool, v_pool, page_row, visible, scale)
    return {"idx": idx, "part": part, "out": out, "lse": lse, "vote": vote, "q_mean": q_mean}


# ---------------------------------------- Selection Cache rationale (R13, figure 3(b))

def lemma1_epsilon(q1: np.ndarray, keys: np.ndarray, k: int) -> float:
    """Sufficient cosine above which TopK_k(q . K^T) equals TopK_k(q1 . K^T) (reading R13).

    TS-notes, "Selection Cache" (the lemma: consecutive queries with cosine above
    a threshold select the same top-k keys) and Appendix C (the proof by the
    orthogonal decomposition q2 = q1 cos t + p sin t). keys [n, d], 0 < k < n.
    Returns eps = 2R / sqrt(D^2 + 4R^2); 1.0 when the k-th and (k+1)-th scores tie.
    """
    keys = np.asarray(keys, dtype=np.float64)
    q1 = np.asarray(q1, dtype=np.float64)
    s1 = keys @ (q1 / math.sqrt(float(q1 @ q1)))
    srt = np.sort(s1)[::-1]
    gap = float(srt[k - 1] - srt[k])
    R = float(np.sqrt((keys * keys).sum(axis=1)).max())
    if gap <= 0.0:
        return 1.0
    return 2.0 * R / math.sqrt(gap * gap + 4.0 * R * R)


def selection_overlap(a: np.ndarray, b: np.ndarray) -> float:
    """|A n B| / |A|: the overlap rate of two selections (TS-review, figure 3(b))."""
    a = np.asarray(a)
    if a.size == 0:
        return 1.0
    return float(np.intersect1d(a, np.asarray(b)).size) / float(a.size)


# ------------------------------------------- block-level selection contrast (R14)

def select_blocks(vote: np.ndarray, n: int, budget: int, block: int) -> np.ndarray:
    """Tokens of the budget // block best blocks of `block` tokens by their largest vote (R14).

    TS-review, figure 2(b) and observation 1 (block-level methods such as InfLLM
    take whole blocks; selection granularity 1 is token-level selection).
    Returns the selected token indices, ascending.
    """
    vote = np.asarray(vote, dtype=np.float64)[:n]
    nb = -(-n // block)
    scores = np.array([vote[j * block:min(n, (j + 1) * block)].max() for j in range(nb)])
    take = min(nb, max(0, budget // block))
    blocks = np.argsort(-scores, kind="stable")[:take]
    toks = [np.arange(j * block, min(n, (j + 1) * block)) for j in sorted(blocks.tolist())]
    return np.concatenate(toks).astype(np.int64) if toks else np.zeros(0, dtype=np.int64)


def recall_at(selected: np.ndarray, vote: np.ndarray, n: int, m: int) -> float:
    """|selected n TopM(vote)| / m, ties to the lower index (R14; TS-review figure 2(b))."""
    top = _order_desc(np.asarray(vote, dtype=np.float64), np.arange(n))[:m]
    return float(np.intersect1d(top, np.asarray(selected)).size) / float(m)
