"""Seeded synthetic decode workloads for token-level KV selection.

This module only draws inputs. It holds none of the method's arithmetic (no
logits, no softmax, no selection, no attention): both the CUDA path and the
CPU oracle read what it produces, and neither imports the other.

The pages the method comes from evaluate on long-context benchmarks with real
models (InfiniteBench, RULER, LongBench with Qwen2-7B / Llama-3-8B). Neither
the data nor the weights are available here, so these generators stand in for
them with the models' attention geometry only:

* keys    K = N(0,1) * s_g, one scale per KV head, s_g = 10**U(-2, 1)
          (three decades; the TokenSelect deep notes, "attention is sparse,
          non-contiguous and head-distinctive", report per-head logit L1 norms
          spanning about three orders of magnitude), or s_g = 1 for the tiny
          fp32 case;
* values  V = N(0,1);
* queries an AR(1) walk q_{t+1} = rho_t q_t + sqrt(1 - rho_t^2) eps, so
          consecutive cosines sit near rho_t (the TokenSelect review, figure
          3(a): consecutive-query cosine medians near 0.945);
* needles planted high-dot-product keys in the middle of the context, at
          distinct positions, with a fixed logit at step 0;
* pages   16-token pages, physical pages a seeded random permutation (one
          shared, interleaved pool when the batch has several sequences).

Pool layout (what the C ABI reads): ``pool[page][kv_head][slot][d]``, with
token ``i`` of a sequence at ``pool[page_table[i // P], :, i % P, :]``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

PAGE_SIZE = 16


@dataclass(frozen=True)
class Spec:
    """Shape and selection parameters of one synthetic decode workload."""

    name: str
    batch: int
    layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    kv_dtype: str                  # "f32" or "bf16"
    n0: tuple                      # per-sequence cache length at step 0 (None: drawn)
    n0_range: Optional[tuple]      # (lo, hi) for log-uniform draws when n0 is None
    steps: int
    mode: str                      # "topk" or "topp"
    k: int
    n_sink: int
    n_local: int
    top_p: float
    theta: float
    rho: Optional[float]           # fixed AR(1) coefficient, or None for U(rho_lo, rho_hi)
    rho_range: tuple
    key_scale: str                 # "unit" or "logu3"
    needles: str                   # "unit4", "lnN2", "topp_mix"
    q_bf16: bool                   # round queries to bf16 values (held as fp32)
    seed: int
    page_size: int = PAGE_SIZE


def _spec(**kw) -> Spec:
    base = dict(batch=1, layers=1, n_q_heads=32, n_kv_heads=8, head_dim=128,
                kv_dtype="bf16", n0_range=None, steps=64, mode="topk", k=2048,
                n_sink=4, n_local=512, top_p=0.0, theta=0.9, rho=None,
                rho_range=(0.85, 0.99), key_scale="logu3", needles="lnN2",
                q_bf16=True)
    base.update(kw)
    return Spec(**base)


# The five workloads. Index i uses seed 20260 + i.
CONFIGS = {
    0: _spec(name="tiny-mha-fp32-n1024", n_q_heads=4, n_kv_heads=4, head_dim=64,
             kv_dtype="f32", n0=(1024,), steps=8, k=64, n_sink=4, n_local=16,
             rho=0.95, key_scale="unit", needles="unit4", q_bf16=False, seed=20260),
    1: _spec(name="llama3-8b-gqa-n128k", n0=(131072,), steps=64, seed=20261),
    2: _spec(name="qwen2-7b-cb8-n32k-256k", batch=8, n_q_heads=28, n_kv_heads=4,
             n0=None, n0_range=(32768, 262144), steps=32, seed=20262),
    3: _spec(name="llama3-8b-8layer-n1m", layers=8, n0=(1048576,), steps=16,
             seed=20263),
    4: _spec(name="llama3-8b-topp-b4-n256k", batch=4, n0=(262144,) * 4, steps=32,
             mode="topp", top_p=0.9, needles="topp_mix", seed=20264),
}


def spec(cfg: int, **overrides) -> Spec:
    """The spec of workload ``cfg`` with optional field overrides (for small cases)."""
    return replace(CONFIGS[cfg], **overrides)


@dataclass
class Workload:
    """All inputs of a decode trajectory, on one device.

    q[t][l]          fp32 [B][H][d] query of step t, layer l
    k_pool[l]        [num_pages][H_kv][P][d] (fp32, or bf16)
    v_pool[l]        same layout as k_pool
    page_table       int32 [B][max_pages], -1 past a sequence's pages
    n0               int list, cache length of each sequence at step 0
    needle_pos[l][b] int64 [H][n_needles] logical positions of planted needles
    """

    spec: Spec
    q: List[List[torch.Tensor]]
    k_pool: List[torch.Tensor]
    v_pool: List[torch.Tensor]
    page_table: torch.Tensor
    n0: List[int]
    needle_pos: List[List[torch.Tensor]] = field(default_factory=list)
    key_scales: List[torch.Tensor] = field(default_factory=list)
    rho: Optional[torch.Tensor] = None

    def seq_lens(self, t: int) -> torch.Tensor:
        """int32 [B]: cache length of every sequence at decode step t (N_t = N0 + t)."""
        return torch.tensor([n + t for n in self.n0], dtype=torch.int32,
                            device=self.page_table.device)

    @property
    def num_pages(self) -> int:
        return self.k_pool[0].shape[0]

    @property
    def max_tokens(self) -> int:
        return self.page_table.shape[1] * self.spec.page_size


def _round_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).to(torch.float32)


def generate(sp: Spec, device="cpu", extra_steps: int = 0) -> Workload:
    """Draw the whole trajectory of ``sp`` (steps + extra_steps decode steps)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(sp.seed)
    gcpu = torch.Generator(device="cpu")
    gcpu.manual_seed(sp.seed + 7919)
    T = sp.steps + extra_steps
    B, L, H, Hkv, d, P = sp.batch, sp.layers, sp.n_q_heads, sp.n_kv_heads, sp.head_dim, sp.page_size
    assert H % Hkv == 0
    G = H // Hkv

    # cache lengths at step 0
    if sp.n0 is not None:
        n0 = [int(x) for x in sp.n0]
        assert len(n0) == B
    else:
        lo, hi = sp.n0_range
        u = torch.rand(B, generator=gcpu, dtype=torch.float64)
        n0 = [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]

    # pages: one pool for all sequences, a seeded permutation interleaves them
    pages_per_seq = [-(-(n + T) // P) for n in n0]
    total_pages = sum(pages_per_seq)
    perm = torch.randperm(total_pages, generator=gcpu).to(torch.int32)
    max_pages = max(pages_per_seq)
    pt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, np_ in enumerate(pages_per_seq):
        pt[b, :np_] = perm[off:off + np_]
        off += np_
    page_table = pt.to(dev)

    kv_torch = torch.float32 if sp.kv_dtype == "f32" else torch.bfloat16

    # queries: q[t][l] = [B][H][d]
    q0 = torch.randn(L, B, H, d, generator=g, device=dev, dtype=torch.float32)
    if sp.q_bf16:
        q0 = _round_bf16(q0)
    if sp.rho is not None:
        rho = torch.full((T, B), sp.rho, dtype=torch.float32)
    else:
        lo, hi = sp.rho_range
        rho = lo + (hi - lo) * torch.rand(T, B, generator=gcpu, dtype=torch.float32)
    qs = [q0]
    for t in range(1, T):
        eps = torch.randn(L, B, H, d, generator=g, device=dev, dtype=torch.float32)
        r = rho[t].to(dev).view(1, B, 1, 1)
        nxt = r * qs[-1] + torch.sqrt(1.0 - r * r) * eps
        if sp.q_bf16:
            nxt = _round_bf16(nxt)
        qs.append(nxt)
    q = [[qs[t][l].contiguous() for l in range(L)] for t in range(T)]

    k_pools, v_pools, needle_pos, key_scales = [], [], [], []
    for l in range(L):
        kp = torch.randn(total_pages, Hkv, P, d, generator=g, device=dev, dtype=torch.float32)
        if sp.key_scale == "logu3":
            sc = torch.pow(10.0, -2.0 + 3.0 * torch.rand(Hkv, generator=gcpu, dtype=torch.float64)).to(torch.float32)
        else:
            sc = torch.ones(Hkv, dtype=torch.float32)
        key_scales.append(sc)
        kp.mul_(sc.to(dev).view(1, Hkv, 1, 1))
        kp = kp.to(kv_torch)
        vp = torch.randn(total_pages, Hkv, P, d, generator=g, device=dev, dtype=torch.float32).to(kv_torch)

        # needles, planted against the step-0 query of this layer
        per_seq = []
        for b in range(B):
            n_cand_lo, n_cand_hi = min(sp.n_sink, n0[b]), max(min(sp.n_sink, n0[b]), n0[b] - sp.n_local)
            n_needle, logit_of = _needle_plan(sp, b, n0[b])
            pos_bh = torch.zeros(H, n_needle, dtype=torch.int64)
            if n_needle > 0 and n_cand_hi - n_cand_lo >= G * n_needle:
                for gk in range(Hkv):
                    choice = torch.randperm(n_cand_hi - n_cand_lo, generator=gcpu)[: G * n_needle] + n_cand_lo
                    for j in range(G):
                        h = gk * G + j
                        pos = choice[j * n_needle:(j + 1) * n_needle]
                        pos_bh[h] = pos
                        qh = q[0][l][b, h].to(torch.float32)
                        # std of this head's random step-0 logits: s_g |q_h| / sqrt(d)
                        sigma = float(sc[gk]) * float(qh.norm()) / math.sqrt(d)
                        key = logit_of(qh, d, sigma, n0[b])   # [d] fp32
                        pages = page_table[b, (pos // P).to(dev)].to(torch.int64)
                        slots = (pos % P).to(dev)
                        kp[pages, gk, slots, :] = key.to(kv_torch).view(1, d).expand(len(pos), d)
            per_seq.append(pos_bh)
        needle_pos.append(per_seq)
        k_pools.append(kp.contiguous())
        v_pools.append(vp.contiguous())

    return Workload(spec=sp, q=q, k_pool=k_pools, v_pool=v_pools, page_table=page_table,
                    n0=n0, needle_pos=needle_pos, key_scales=key_scales, rho=rho)


def _needle_plan(sp: Spec, b: int, n0: int):
    """(needles per query head, key builder) for sequence b.

    The key builders only scale the step-0 query direction; the logit the key
    reaches at step 0 (softmax scale 1/sqrt(d)) is stated beside each. Outside
    the tiny case the logit is set against the head's own logit spread: the
    expected largest of n0 random logits of std sigma is about
    sigma*sqrt(2 ln n0), and the needle sits a margin above it, so it stands out
    in heads of every key scale.
    """
    sqd = math.sqrt(sp.head_dim)

    def unit4(qh, d, sigma, n):            # key = 4 q/|q|   -> logit 4|q|/sqrt(d)
        return 4.0 * qh / qh.norm()

    def with_logit(margin):                # key = c sqrt(d) q/|q|^2 -> logit exactly c
        def build(qh, d, sigma, n):
            c = margin(n) + sigma * math.sqrt(2.0 * math.log(n))
            return (c * sqd) * qh / (qh.norm() ** 2)
        return build

    if sp.needles == "unit4":              # eight needle keys in all, spread over the heads
        return max(1, 8 // sp.n_q_heads), unit4
    if sp.needles == "lnN2":               # 32 per head, margin ln n0 + 2
        return 32, with_logit(lambda n: math.log(n) + 2.0)
    if sp.needles == "topp_mix":
        if b % 4 < 2:                      # 2 dominant needles, margin ln n0 + 6
            return 2, with_logit(lambda n: math.log(n) + 6.0)
        # 4096 mild needles, margin ln(n0/4096) + 2
        return 4096, with_logit(lambda n: math.log(n / 4096.0) + 2.0)
    raise ValueError(sp.needles)


def host_copy(x: torch.Tensor):
    """numpy view of a tensor on the host; bf16 tensors come back as uint16 bit patterns."""
    x = x.detach().to("cpu")
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    return x.numpy()
