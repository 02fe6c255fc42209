"""GPU decode path against the CPU oracle, through the C ABI, on seeded inputs.

Small sizes check every output of every step (several score CTAs, ragged last
pages, several selection chunks); the full sizes of the 128K, batched and
top-p workloads run the same comparison on fewer steps (both cache settings,
both top-p masses), and the 1M-token workload at its stated shape of 8 layers
with the cache off and at theta 0.9. Multi-layer cases check that every layer
keeps its own Selection Cache entry.
"""
import pytest
import torch

import workloads as W
from parity import run_trajectory

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(sp, steps, wl=None, **kw):
    wl = wl if wl is not None else W.generate(sp, DEV)
    rep = run_trajectory(wl, steps, **kw)
    print(f"{sp.name}: steps={rep.steps} hits={rep.hits} replays={rep.replays} "
          f"band_swaps={rep.band_swaps} worst_vote_rel={rep.worst_vote_rel:.2e} "
          f"near_tau_err={rep.near_err:.2e} margin={rep.margin:.2e} at_risk={rep.at_risk}")
    return rep


def test_tiny_fp32_trajectory_with_cache():
    rep = _run(W.spec(0), 8)
    assert rep.steps == 8


@pytest.mark.parametrize("multi", [False, True])
def test_llama_small_both_paths(multi):
    sp = W.spec(1, n0=(9001,), steps=4, k=512, n_local=128)
    _run(sp, 4, multi_kernel=multi)


@pytest.mark.parametrize("multi", [False, True])
def test_qwen_batched_small_both_paths(multi):
    sp = W.spec(2, n0=(700, 5000, 3100, 40), n0_range=None, batch=4, steps=3, k=256, n_local=64)
    _run(sp, 3, multi_kernel=multi)


@pytest.mark.parametrize("scan", ["tensor", "tensor-claim", "cuda"])
def test_llama_scan_paths(scan, monkeypatch):
    # bf16 pages of 8 KV heads scan on the tensor cores unless TOKENSELECT_NO_TC=1; with
    # TOKENSELECT_SCAN_CLAIM=1 the CTAs claim pages from a shared counter
    if scan == "cuda":
        monkeypatch.setenv("TOKENSELECT_NO_TC", "1")
    if scan == "tensor-claim":
        monkeypatch.setenv("TOKENSELECT_SCAN_CLAIM", "1")
    sp = W.spec(1, n0=(20011,), steps=3, k=1024, n_local=128)
    _run(sp, 3)


@pytest.mark.parametrize("claim", [False, True])
def test_llama_batched_two_sequences_per_cta(claim, monkeypatch):
    # two sequences: every CTA range meets at most two of them (or, claiming pages, every CTA
    # holds both query images and takes pages of either)
    if claim:
        monkeypatch.setenv("TOKENSELECT_SCAN_CLAIM", "1")
    sp = W.spec(1, n0=(40000, 33001), n0_range=None, batch=2, steps=2, k=512, n_local=64)
    _run(sp, 2, theta=2.0)


def test_llama_batched_many_short_sequences():
    # a CTA range meets three or more sequences: the CUDA-core scan takes over
    sp = W.spec(1, n0=(300, 17, 2000, 45, 999, 5), n0_range=None, batch=6, steps=2, k=128, n_local=32)
    _run(sp, 2, theta=2.0)


@pytest.mark.parametrize("multi", [False, True])
def test_llama_three_layers_with_cache(multi):
    # every layer keeps its own Selection Cache entry (C_Q, C_T, counts): layers > 0 read and
    # write at their own offsets, on the persistent kernel and on the multi-kernel path
    sp = W.spec(1, n0=(6007,), layers=3, steps=4, k=384, n_local=96)
    rep = _run(sp, 4, layers=(0, 1, 2), multi_kernel=multi)
    assert rep.steps == 4 * 3      # (step, layer) pairs


def test_qwen_batched_layers_with_cache():
    sp = W.spec(2, n0=(1800, 3333, 950), n0_range=None, batch=3, layers=2, steps=3, k=200, n_local=40)
    _run(sp, 3, layers=(0, 1))


def test_tiny_fp32_separate_calls_all_miss():
    _run(W.spec(0), 4, separate_calls=True, theta=2.0)


@pytest.mark.parametrize("overrides", [
    dict(n0=(3001,), steps=3, k=256, n_local=64),                              # GQA 32/8, ragged
    dict(n0=(5000,), steps=2, k=2048),                                         # k close to |C|
    dict(n0=(70,), steps=3, k=2048),                                           # N < k+s+w: all tokens
])
def test_llama_geometry_small(overrides):
    sp = W.spec(1, **overrides)
    _run(sp, sp.steps, theta=2.0)
    _run(sp, sp.steps)


def test_qwen_geometry_batched_small():
    sp = W.spec(2, n0=(1000, 4099, 2500), n0_range=None, batch=3, steps=3, k=300, n_local=50)
    _run(sp, 3)
    _run(sp, 2, theta=2.0)


@pytest.mark.parametrize("geom", [
    dict(n_q_heads=8, n_kv_heads=2, head_dim=64, kv_dtype="f32"),
    dict(n_q_heads=32, n_kv_heads=8, head_dim=128, kv_dtype="f32"),
    dict(n_q_heads=8, n_kv_heads=8, head_dim=128, kv_dtype="bf16"),
    dict(n_q_heads=8, n_kv_heads=4, head_dim=64, kv_dtype="bf16"),
    dict(n_q_heads=16, n_kv_heads=2, head_dim=128, kv_dtype="bf16"),
])
def test_other_geometries(geom):
    sp = W.spec(1, n0=(2300,), steps=2, k=200, n_local=32, key_scale="logu3", needles="lnN2", **geom)
    _run(sp, 2, theta=2.0)


def test_topp_small():
    for p in (0.9, 0.99):
        sp = W.spec(4, n0=(6000, 6000, 7000, 9000), steps=3, top_p=p)
        _run(sp, 3)
        _run(sp, 2, theta=2.0)


def test_topp_all_tokens_when_p_is_one():
    sp = W.spec(4, n0=(300,) * 4, steps=1, top_p=1.0, needles="lnN2")
    _run(sp, 1, theta=2.0)


# ------------------------------------------------------------ full sizes

def test_llama_128k_full():
    sp = W.spec(1, steps=6)
    _run(sp, 6)


@pytest.mark.parametrize("theta", [2.0, 0.9])
def test_qwen_batched_full(theta):
    sp = W.spec(2, steps=3)
    _run(sp, 3 if theta <= 1.0 else 2, theta=theta)


@pytest.mark.parametrize("p", [0.9, 0.99])
def test_topp_256k_full(p):
    sp = W.spec(4, steps=2, top_p=p)
    _run(sp, 2)


def test_llama_1m_8layers_full():
    # the 1M-token workload at its stated shape: 8 layers of 1M tokens (4 GB of K+V each), every
    # layer with its own Selection Cache entry; two steps with the cache off, then two with
    # theta 0.9 on the same inputs
    sp = W.spec(3, steps=2)
    wl = W.generate(sp, DEV)
    layers = tuple(range(sp.layers))
    r0 = _run(sp, 2, wl=wl, layers=layers, theta=2.0)
    assert r0.steps == 2 * sp.layers and r0.hits == 0      # (step, layer) pairs
    r1 = _run(sp, 2, wl=wl, layers=layers, theta=0.9)
    assert r1.steps == 2 * sp.layers
    del wl
    torch.cuda.empty_cache()
