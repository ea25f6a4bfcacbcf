"""Pins of the oracle's fused look-ahead attention output (Figure 7, right).

Each lookahead row is checked against textbook softmax attention (scipy) over the
whole context when the budget covers it and everything is fetched, and a
lookahead query equal to the true query must give the true query's output."""
import numpy as np
from scipy.special import softmax

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn


def test_lookahead_rows_equal_dense_attention_at_full_budget():
    w = syn.Workload("dense", L=1, B=2, Hq=8, Hkv=2, ctx=[200, 77], Kb=16, C=16, n_hot=2, n_la=3)
    K, V = syn.layer_kv(w, 0)
    host = syn.host_tier_from_kv(w, K, V)
    b2s, s2b, lu = [np.full_like(np.array(t), -1) for t in syn.initial_tables(w, 0)]
    kp, vp = syn.pools_from_tables(w, host, s2b)
    q, qla = syn.layer_queries(w, 0, 0)
    r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 0, lookahead_out=True)
    for b in range(w.B):
        for h in range(w.Hkv):
            Kt = ref.bf16_to_f64(K[b, h, :w.ctx[b]])
            Vt = ref.bf16_to_f64(V[b, h, :w.ctx[b]])
            for j in range(w.n_la):
                for g in range(w.G):
                    qq = ref.bf16_to_f64(qla[b, j, h * w.G + g])
                    want = softmax(Kt @ qq / np.sqrt(w.d)) @ Vt
                    np.testing.assert_allclose(r["out_la"][b, j, h * w.G + g], want, rtol=1e-11, atol=1e-12)


def test_lookahead_row_equal_to_the_true_query_gives_its_output():
    w = syn.Workload("same", L=1, B=1, Hq=8, Hkv=2, ctx=[500], Kb=8, C=2, n_hot=4, n_la=2)
    K, V = syn.layer_kv(w, 0)
    host = syn.host_tier_from_kv(w, K, V)
    b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, 0)]
    kp, vp = syn.pools_from_tables(w, host, s2b)
    q, qla = syn.layer_queries(w, 0, 0)
    qla = qla.copy()
    qla[:, 1] = q
    r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 0, lookahead_out=True)
    np.testing.assert_array_equal(r["out_la"][:, 1], r["out"])
    assert not np.array_equal(r["out_la"][:, 0], r["out"])
