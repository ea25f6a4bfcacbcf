"""Host-side logic of the benchmark (no GPU): algorithmic bytes, workload
selection, host-tier sizing, the L2 note, the --impl flag and the CPU
baseline's reporting rule."""
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


def test_impl_flag_parsing(bench, monkeypatch):
    for argv, want in [(["bench.py"], None), (["bench.py", "--impl", "reference"], "reference"),
                       (["bench.py", "--steps", "2", "--impl=reference"], "reference"),
                       (["bench.py", "--impl", "gb300"], "gb300")]:
        monkeypatch.setattr(bench.sys, "argv", argv)
        assert bench._impl_from_argv() == want


@pytest.mark.parametrize("one,allc,faster", [(0.5, 2.0, "one"), (3.0, 1.5, "all")])
def test_cpu_baseline_reports_the_faster_thread_setting(bench, monkeypatch, one, allc, faster):
    """`value` is the faster of the one-thread and all-cores timings, `cores` the
    threads it used; both values are reported and scaled by the pairs per layer."""
    import argparse

    calls = []

    def fake(args, heads, threads):
        calls.append((heads, threads))
        return one if threads == 1 else allc

    monkeypatch.setattr(bench, "_cpu_worker_sec_per_head", fake)
    monkeypatch.setattr(bench.os, "cpu_count", lambda: 16)
    ns = argparse.Namespace(workload="qwen3_8b_decode", ratio="0.01", batch=32, layers=36, ctx=32768)
    r = bench.cpu_baseline(ns, 12)
    per = 32 * 8
    assert calls == [(48, 1), (4, 16)]
    assert r["value_1_thread"] == pytest.approx(1.0 / (one * per))
    assert r["value_16_threads"] == pytest.approx(1.0 / (allc * per))
    assert r["cores"] == (1 if faster == "one" else 16)
    assert r["value"] == max(r["value_1_thread"], r["value_16_threads"])
    assert r["kind"] == "oracle" and r["unit"] == bench.UNIT


def test_reference_arm_line_says_what_it_timed(bench, monkeypatch, capsys):
    """The reference arm's line: the measured time of each timed step (so steps x
    ms_per_step fits the run), the extrapolated layer-step time beside it, the
    pairs it timed, and the same config as the GPU arm's line."""
    monkeypatch.setattr(bench.sys, "argv", ["bench.py", "--impl", "reference", "--workload", "tiny",
                                            "--steps", "2", "--warmup", "1"])
    args = bench.parse()
    bench.run_reference(args, 0)
    import json

    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["extrapolated"] is True
    assert line["pairs_timed"] == 2 and line["pairs_per_step"] == 1
    assert line["steps"] * line["ms_per_step"] / 1000.0 <= line["run_wall_s"]
    w = bench.workload(args)
    assert line["ms_per_step_extrapolated"] == pytest.approx(1000.0 * w.L / line["value"])
    l_phys, l_host = bench.planned_layers(args, w)
    assert line["config"] == bench.config_dict(args, w, l_phys, l_host, 0)
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_workload_description_names_the_drifting_hot_set(bench):
    assert "drifting through 256 planted blocks" in bench.workload_desc(syn.long_output())
    assert "64 planted hot blocks" in bench.workload_desc(syn.qwen3_8b_decode())


def test_span_summary_of_a_hand_made_overlap_timeline(bench):
    """Two layers, one step, in ns: score 0-300us, select 302-322, gather 324-350
    (side), attention of layer 0 runs 324-340 beside layer 1's gather; the gaps of
    the critical path follow from these numbers alone."""
    import numpy as np

    us = lambda *v: np.array([int(x * 1000) for x in v], dtype=np.int64)  # noqa: E731
    sp = {
        "score": (us(0, 352), us(300, 652)),
        "select": (us(302, 654), us(322, 674)),
        "gather": (us(324, 676), us(350, 700)),
        "attn": (us(676, 702), us(690, 716)),
        "score_pooled": (us(), us()), "copy": (us(), us()), "append": (us(), us()),
    }
    out = bench.summarize_spans(sp, L=2, steps=1, copy="overlap", gather_bytes=4_194_304, link_gbs=200.0)
    k = out["kernel_us"]
    assert k["score"]["p50"] == 300.0 and k["select"]["p50"] == 20.0 and k["gather"]["mean"] == 25.0
    assert out["layer_period_us"]["p50"] == 352.0
    g = out["gaps_us"]
    assert g["score_end_to_select_start"]["p50"] == 2.0
    assert g["select_end_to_gather_start"]["p50"] == 2.0
    assert g["gather_end_to_next_score_start"]["p50"] == 2.0
    assert g["select_end_to_attn_prev_start"]["p50"] == 2.0  # attention of layer 0 after layer 1's select
    assert g["next_score_start_after_gather_and_attn_prev"] is None  # no layer after layer 1 here
    # 4 MiB in 26 and 24 us: 161.3 and 174.8 GB/s
    assert abs(out["decode_gather_gbs"]["p50"] - (4_194_304 / 26000 + 4_194_304 / 24000) / 2) < 0.1
