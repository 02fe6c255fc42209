"""Planted mistakes in the oracle must each fail at least one pin.

Every case copies the oracle, changes one line the way a plausible slip would
(wrong GQA index, dropped scale, off-by-one window, ...), and runs the pin
suite against the copy in a separate process. Mistakes are planted only in a
temporary copy of the CPU oracle.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "gqa index h % G": ("h = g * G + j\n            out[h] = alpha", "h = j * Hkv + g\n            out[h] = alpha"),
    "vote without scale": ('out[h] = alpha * np.einsum("nd,d->n", K, q[h])',
                           'out[h] = np.einsum("nd,d->n", K, q[h])'),
    "normaliser drops max": ("m + np.log(np.exp(logits - m[:, None]).sum(axis=1))",
                             "np.log(np.exp(logits - m[:, None]).sum(axis=1))"),
    "vote not normalised": ("v += np.exp(logits[h] - L[h])", "v += np.exp(logits[h])"),
    "top-k over all tokens": ("cand = np.arange(s_end, local_start)", "cand = np.arange(0, n)"),
    "window off by one": ("local_start = max(s_end, n - n_local)", "local_start = max(s_end, n - n_local + 1)"),
    "top-p drops crossing token": ("take = min(n, j + 1)", "take = min(n, j)"),
    "cache hit needs strict >": ("return c >= theta, c", "return c > theta, c"),
    "C_Q written on hits": ('    res = {"hit": hit, "cos": c}\n',
                            '    res = {"hit": hit, "cos": c}\n    if hit:\n        state.cq = q.copy()\n'),
    "hit window not rebuilt": ("idx = refresh_hit(part, n, n_sink, n_local)",
                               "idx = refresh_hit(part, n - 1, n_sink, n_local)"),
    "lse drops max": ("lse[h] = m + math.log(Z)", "lse[h] = math.log(Z)"),
    "attention reads K as V": ("V = gather_rows(v_pool, page_row, idx, g)", "V = gather_rows(k_pool, page_row, idx, g)"),
    "page slot index": ("return as_f64(pool[pages, g, tokens % P, :])",
                        "return as_f64(pool[pages, g, (tokens // P) % P, :])"),
    "cosine normalisation": ("return float(a @ b) / (na * nb)", "return float(a @ b) / (na * na)"),
    "bf16 widening shift": ("<< np.uint32(16)", "<< np.uint32(15)"),
    "hard vote over all tokens": ("top = _order_desc(logits[h], cand)[:max(0, k)]",
                                  "top = _order_desc(logits[h], np.arange(n))[:max(0, k)]"),
    "hard vote takes k + 1": ("top = _order_desc(logits[h], cand)[:max(0, k)]",
                              "top = _order_desc(logits[h], cand)[:max(0, k + 1)]"),
    "prefill mean drops a query": ("q_mean = q_chunk.sum(axis=0) / c", "q_mean = q_chunk[1:].sum(axis=0) / c"),
    "prefill not causal": ("visible = idx[idx <= n - c + i]", "visible = idx"),
    "prefill causal off by one": ("visible = idx[idx <= n - c + i]", "visible = idx[idx < n - c + i]"),
    "logit sum as max": ("return np.asarray(logits, dtype=np.float64).sum(axis=0)",
                         "return np.asarray(logits, dtype=np.float64).max(axis=0)"),
    "page size fixed at 16": ("    P = pool.shape[2]\n", "    P = 16\n"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    a, b = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "tokenselect_oracle.py")).read()
    assert a in src, f"mutation anchor for {name!r} no longer in the oracle"
    for sub in ("tests", "workloads"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py"))
    (tmp_path / "oracle").mkdir()
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), tmp_path / "oracle")
    (tmp_path / "oracle" / "tokenselect_oracle.py").write_text(src.replace(a, b, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"planted mistake {name!r} passed every pin"
