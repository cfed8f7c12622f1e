"""The algorithmic work counts behind every roofline fraction bench.py
reports, against their closed forms and a brute-force count (CPU)."""
import importlib.util
import os

import pytest

from learned_token_pruning_09_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_attention_flops_count_the_causal_triangle(bench):
    # brute force: every (i, j <= i) pair costs D multiply-adds in Q K^T and D in P V, per query head
    for lens, hq, d in (([5], 2, 8), ([3, 7, 1], 4, 16)):
        brute = sum(hq * 2 * (2 * d) for t in lens for i in range(t) for j in range(i + 1))
        assert bench.attention_flops(lens, hq, d) == brute
    # the 128k workload: 8,256 kept tokens, 16 heads of 128
    assert bench.attention_flops([8256], 16, 128) == 2.0 * 16 * 128 * 8256 * 8257 == 279223468032.0


def test_gate_topk_gather_bytes(bench):
    shape = synth.ALL_SHAPES["long-128k"]()
    n, t, d = shape.n_rows, shape.n_kept, shape.d
    assert (n, t, d) == (131072, 8256, 2048)
    # residuals read once, scores written and read, kept ids written and read,
    # kept rows read and written, kept positions and scores written
    assert bench.path_bytes(shape) == n * 2 * d + n * (4 + 4) + t * (4 + 4) + t * 2 * (2 * d) + t * (4 + 4)
    assert bench.path_bytes(shape) == 605684736.0
    # the prunable-span path reads the per-row mask twice more
    assert bench.masked_path_bytes(shape, t) == bench.path_bytes(shape) + 2 * n


def test_projection_flops(bench):
    shape = synth.ALL_SHAPES["long-128k"]()
    t, d, hq, hkv, dh = shape.n_kept, shape.d, shape.hq, shape.hkv, shape.head_dim
    qkv = 2.0 * t * d * (hq * dh + 2 * hkv * dh)
    out = 2.0 * t * (hq * dh) * d
    assert bench.proj_flops(shape) == qkv + out
    assert abs(bench.proj_flops(shape) / 1e9 - 207.8) < 0.1
