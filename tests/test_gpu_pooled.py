"""Pooled-key scoring (min/max compressed keys, f1) on the GPU against the oracle.

Same bar as the max-dot path: pooled keys equal to the oracle's pooling, block
scores inside their certified interval around the exact pooled score, selected
and fetched blocks, tables and pools bit-exact, attention within tolerance."""
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


@pytest.mark.parametrize("gather", ["fused", "carry"])
def test_tiny_workload_pooled(gather):
    w = syn.tiny()
    c = Case(w, scoring="pooled")
    c.compare_pooled()
    for step in range(3):
        c.step(step, gather=gather)


def test_ragged_contexts_pooled():
    w = syn.Workload("ragged", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=4, n_hot=16)
    c = Case(w, scoring="pooled")
    c.compare_pooled()
    for step in range(2):
        c.step(step)


@pytest.mark.parametrize("Hq,n_la", [(64, 4), (8, 4), (16, 3)])
def test_gqa_groups_pooled(Hq, n_la):
    w = syn.Workload("gqa", L=1, B=2, Hq=Hq, Hkv=8, ctx=[2048, 1531], Kb=32, C=6, n_hot=16, n_la=n_la)
    c = Case(w, scoring="pooled")
    c.step(0)
    c.step(1, gather="carry")


def test_duplicate_blocks_tie_pooled():
    """Copies of one block have equal pooled scores: ties go to the lower index."""
    w = syn.Workload("ties", L=1, B=1, Hq=32, Hkv=8, ctx=[2048], Kb=32, C=8, n_hot=16)
    K, V = syn.layer_kv(w, 0)
    for h in range(w.Hkv):
        src = K[0, h, 16 * 5:16 * 6].copy()
        for x in range(20, 120, 3):
            K[0, h, 16 * x:16 * (x + 1)] = src
    c = Case(w, K=K, V=V, scoring="pooled")
    c.step(0)
    c.step(1)


def test_long_output_appends_keep_pooled_keys_current():
    ctx = [1000, 1531, 2047, 2048]
    w = syn.Workload("long_output", L=1, B=4, Hq=32, Hkv=8, ctx=list(ctx), Kb=32, C=2, n_hot=16,
                     nb_max=-(-(max(ctx) + 40) // 16))
    c = Case(w, scoring="pooled")
    for step in range(6):
        c.step(step, append=True)
    c.compare_pooled()
    c.compare_caches()


def test_multi_layer_decode_step_pooled_carry():
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    L = 3
    w = syn.Workload("layers", L=L, B=2, Hq=32, Hkv=8, ctx=[3000, 1777], Kb=32, C=3, n_hot=16)
    st = DecodeState(w, l_phys=L, l_host=L, scoring="pooled")
    layers = []
    for l in range(L):
        K, V = syn.layer_kv(w, l)
        host = syn.host_tier_from_kv(w, K, V)
        b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, l)]
        kp, vp = syn.pools_from_tables(w, host, s2b)
        st.fill_layer_numpy(l, K, V, b2s, s2b, lu)
        layers.append([K, host, b2s, s2b, lu, kp, vp])
    out = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device="cuda")
    for step in range(3):
        qs = [syn.layer_queries(w, l, step) for l in range(L)]
        st.decode_step(step, [_dev_bits(qla) for _, qla in qs], [_dev_bits(q) for q, _ in qs], out_layers=out)
        torch.cuda.synchronize()
        assert int(st.scratch.err.item()) == 0 and int(st.scratch2.err.item()) == 0
        for l in range(L):
            K, host, b2s, s2b, lu, kp, vp = layers[l]
            q, qla = qs[l]
            r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step, scoring="pooled")
            np.testing.assert_array_equal(st.blk2slot[l].cpu().numpy(), b2s)
            np.testing.assert_array_equal(st.slot2blk[l].cpu().numpy(), s2b)
            _check_out(out[l].cpu().numpy().astype(np.float64), r["out"], f"layer {l} step {step}")
