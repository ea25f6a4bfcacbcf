"""Parity on the shapes of the other workloads: long input (128K context, span and
sink/recent hot blocks), GQA 8 with the fetch-ratio sweep, long output (growing
context with token appends), and the full-size Qwen3-8B decode shape sampled
head by head in the pipelined launch configuration the benchmark times."""
import math

import numpy as np
import pytest

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn

from gpu_helpers import Case, _check_out, _dev_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()


def test_llama_long_input_shape_128k_context():
    w = syn.llama31_8b_long(B=1, L=1)
    assert w.nb_max == 8192 and w.C == 6
    c = Case(w)
    c.step(0)
    c.step(1)


@pytest.mark.parametrize("ratio", [0.01, 0.02, 0.05, 0.10, 0.20, None])
def test_qwen3_32b_shape_fetch_ratio_sweep(ratio):
    w = syn.qwen3_32b(ratio=ratio, B=1, L=1, ctx=32768)
    c = Case(w)
    for step in range(2):
        c.step(step)


def test_long_output_growing_context_with_appends():
    ctx = [1000, 1531, 2047, 2048]
    w = syn.Workload("long_output", L=1, B=4, Hq=32, Hkv=8, ctx=list(ctx), Kb=32, C=2, n_hot=16,
                     nb_max=-(-(max(ctx) + 40) // 16))
    c = Case(w)
    for step in range(6):
        c.step(step, append=True)
    c.compare_caches()
    assert w.ctx == [x + 6 for x in ctx]


def test_full_size_qwen3_8b_sampled_heads_pipelined():
    """36 layers x batch 32 x ctx 32K on the GPU; sampled (layer, request, head) against the oracle."""
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    w = syn.qwen3_8b_decode()
    dev = torch.device("cuda", 0)
    st = DecodeState(w, device=dev, l_phys=w.L, l_host=4)
    st.fill_synthetic()
    qs = [syn.QueryStream(w, l) for l in range(w.L)]
    out = torch.empty((w.L, w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(dev)
    rng = np.random.default_rng(11)
    samples = [(int(rng.integers(0, 4)), int(rng.integers(w.B)), int(rng.integers(w.Hkv))) for _ in range(3)]
    samples.append((3, w.B - 1, w.Hkv - 1))
    oracle_state = {}
    for (l, b, h) in samples:
        K, V = syn.head_kv(w, l, b, h)
        sub = syn.Workload("sub", L=1, B=1, Hq=w.G, Hkv=1, ctx=[w.ctx[b]], Kb=w.Kb, C=w.C, nb_max=w.nb_max)
        host = syn.host_tier_from_kv(sub, K[None, None], V[None, None])
        b2s, s2b, lu = [t[b:b + 1, h:h + 1].copy() for t in syn.initial_tables(w, l)]
        kp, vp = syn.pools_from_tables(sub, host, s2b)
        oracle_state[(l, b, h)] = (K[None, None], host, b2s, s2b, lu, kp, vp)
    for step in range(2):
        qla_l, q_l = [], []
        for l in range(w.L):
            qb, qlab = qs[l].next()
            q_l.append(_dev_bits(qb))
            qla_l.append(_dev_bits(qlab))
        st.decode_step(step, qla_l, q_l, out_layers=out, side=side)
        torch.cuda.synchronize()
        assert int(st.scratch.err.item()) == 0 and int(st.scratch2.err.item()) == 0
        for (l, b, h), (K, host, b2s, s2b, lu, kp, vp) in oracle_state.items():
            qh, qlah = syn.head_queries(w, l, b, h, step)
            r = ref.layer_step(K, qlah[None], qh[None], [w.ctx[b]], host, kp, vp, b2s, s2b, lu,
                               w.Kb, w.C, step)
            np.testing.assert_array_equal(st.blk2slot[l, b, h].cpu().numpy(), b2s[0, 0])
            np.testing.assert_array_equal(st.slot2blk[l, b, h].cpu().numpy(), s2b[0, 0])
            np.testing.assert_array_equal(st.last_used[l, b, h].cpu().numpy(), lu[0, 0])
            got = out[l, b, h * w.G:(h + 1) * w.G].cpu().numpy().astype(np.float64)
            _check_out(got, r["out"][0], f"layer {l} request {b} head {h} step {step}")
