"""Host-side logic of the benchmark (no GPU): algorithmic bytes, workload
selection, host-tier sizing and the L2 note."""
import importlib.util
import os

import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_of_the_headline_config(bench):
    w = syn.qwen3_8b_decode()
    ab = bench.algorithmic_bytes(w, attended_per_head=38.0)
    blocks = 32 * 8 * 2048
    assert ab["score"] == blocks * 16 * 128 * 2 + 32 * 4 * 32 * 128 * 2 + blocks * 8
    assert ab["attn"] == int(32 * 8 * 38.0 * 16 * 128 * 2 * 2) + 32 * 32 * 128 * (2 + 4)
    assert ab["gather_hbm"] == 32 * 8 * 2 * 16 * 128 * 2 * 2
    assert ab["total"] == ab["score"] + ab["topk"] + ab["attn"] + ab["gather_hbm"]
    pooled = bench.algorithmic_bytes(w, attended_per_head=38.0, scoring="pooled")
    assert pooled["score"] == blocks * 512 + 32 * 4 * 32 * 128 * 2 + blocks * 8  # 512 B of pooled keys per block


def test_workload_selection(bench):
    import argparse

    ns = argparse.Namespace(workload="qwen3_32b", ratio="all", batch=32, layers=36, ctx=32768)
    w = bench.workload(ns)
    assert (w.L, w.B, w.Hq, w.Kb, w.C) == (64, 16, 64, 128, 128)
    ns.ratio = "0.05"
    assert bench.workload(ns).C == 6
    ns.workload = "long_output"
    w = bench.workload(ns)
    assert w.B == 128 and min(w.ctx) < max(w.ctx)
    ns.workload = "qwen3_8b_decode"
    w = bench.workload(ns)
    assert (w.L, w.B, w.ctx[0], w.C) == (36, 32, 32768, 2)


def test_host_layers_respect_request_and_model(bench):
    w = syn.qwen3_8b_decode()
    assert 1 <= bench.host_layers_for(w, 8) <= 8
    assert 1 <= bench.host_layers_for(w, 0) <= w.L
    assert bench.host_layers_for(w, 100) <= w.L


def test_l2_note(bench):
    assert bench.l2_note(syn.qwen3_8b_decode(), "maxdot").startswith("inputs larger than L2 (2.00 GiB of keys")
    assert "pooled keys" in bench.l2_note(syn.qwen3_8b_decode(), "pooled")
    assert "smaller than" in bench.l2_note(syn.tiny(), "maxdot")
