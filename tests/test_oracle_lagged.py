"""Pins of the oracle's cross-step pipeline (Figure 8): attention at step t+1 over
the blocks the lookahead queries of step t selected.

Checked against textbook softmax attention over exactly those blocks (fetch-all
makes them all resident), a hand example where the lag changes the attended
block, and the identity that the lag changes no table or pool."""
import numpy as np
from scipy.special import softmax

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn


def _bits(x):
    return syn.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _setup(w, layer=0):
    K, V = syn.layer_kv(w, layer)
    host = syn.host_tier_from_kv(w, K, V)
    b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, layer)]
    kp, vp = syn.pools_from_tables(w, host, s2b)
    return K, V, host, b2s, s2b, lu, kp, vp


def test_lagged_attention_is_softmax_over_the_previous_selection():
    w = syn.Workload("lag", L=1, B=2, Hq=8, Hkv=2, ctx=[700, 333], Kb=8, C=8, n_hot=4)
    K, V, host, b2s, s2b, lu, kp, vp = _setup(w)
    q0, qla0 = syn.layer_queries(w, 0, 0)
    r0 = ref.layer_step(K, qla0, q0, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 0)
    q1, qla1 = syn.layer_queries(w, 0, 1)
    r1 = ref.layer_step(K, qla1, q1, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 1, prev_S=r0["S"])
    G, d = w.G, w.d
    for (b, h), S in r0["S"].items():
        assert r1["A"][(b, h)] == S  # fetch-all: every block of S is resident
        toks = [t for x in S for t in range(16 * x, 16 * x + 16) if t < w.ctx[b]]
        Kt = ref.bf16_to_f64(K[b, h, toks])
        Vt = ref.bf16_to_f64(V[b, h, toks])
        for g in range(G):
            q = ref.bf16_to_f64(q1[b, h * G + g])
            want = softmax(Kt @ q / np.sqrt(d)) @ Vt
            np.testing.assert_allclose(r1["out"][b, h * G + g], want, rtol=1e-12, atol=1e-12)


def test_lag_changes_no_table_or_pool():
    w = syn.Workload("lag", L=1, B=2, Hq=8, Hkv=2, ctx=[900, 500], Kb=8, C=2, n_hot=4)
    a = _setup(w)
    b = [x.copy() for x in a]

    def run(state, q, qla, step, prev=None):
        K, V, host, b2s, s2b, lu, kp, vp = state
        return ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step, prev_S=prev)

    q0, qla0 = syn.layer_queries(w, 0, 0)
    r0 = run(a, q0, qla0, 0)
    run(b, q0, qla0, 0)
    for step in (1, 2):
        q, qla = syn.layer_queries(w, 0, step)
        r = run(a, q, qla, step, r0["S"])
        u = run(b, q, qla, step)
        assert r["S"] == u["S"] and r["F"] == u["F"]
        for x, y in zip(a[3:], b[3:]):
            np.testing.assert_array_equal(x, y)
        r0 = r


def test_hand_example_lag_attends_the_earlier_choice():
    """Two one-token blocks; the step-0 lookahead picks block 0, the step-1 one
    picks block 1.  With Kb = 1 and the lag, step 1 attends block 0 (output =
    its value); without the lag it attends block 1."""
    d, bs = 2, 1
    K = _bits([[1, 0], [0, 1]]).reshape(1, 1, 2, d)
    V = _bits([[3, 0], [0, 5]]).reshape(1, 1, 2, d)
    host = np.stack([K.reshape(1, 1, 2, bs, d), V.reshape(1, 1, 2, bs, d)], axis=3)

    def fresh():
        return (np.full((1, 1, 2), -1, np.int32), np.full((1, 1, 2), -1, np.int32),
                np.full((1, 1, 2), -1, np.int32), np.zeros((1, 1, 2, bs, d), np.uint16),
                np.zeros((1, 1, 2, bs, d), np.uint16))

    qa = _bits([[1, 0]]).reshape(1, 1, 1, d)
    qb = _bits([[0, 1]]).reshape(1, 1, 1, d)
    q = _bits([[1, 1]]).reshape(1, 1, d)
    b2s, s2b, lu, kp, vp = fresh()
    r0 = ref.layer_step(K, qa, q, [2], host, kp, vp, b2s, s2b, lu, 1, 1, 0, bs=bs)
    assert r0["S"][(0, 0)] == [0]
    r1 = ref.layer_step(K, qb, q, [2], host, kp, vp, b2s, s2b, lu, 1, 1, 1, bs=bs, prev_S=r0["S"])
    np.testing.assert_allclose(r1["out"][0, 0], [3, 0])
    assert r1["S"][(0, 0)] == [1]
    b2s, s2b, lu, kp, vp = fresh()
    ref.layer_step(K, qa, q, [2], host, kp, vp, b2s, s2b, lu, 1, 1, 0, bs=bs)
    u1 = ref.layer_step(K, qb, q, [2], host, kp, vp, b2s, s2b, lu, 1, 1, 1, bs=bs)
    np.testing.assert_allclose(u1["out"][0, 0], [0, 5])


def test_lagged_attention_precedes_the_steps_own_gather():
    """A block of the previous selection that was capped out is not attended even
    when this step's gather brings it in: the lagged attention reads the blocks
    resident on entry.  Step 0 selects {0, 1} and fetches only 0 (cap 1); step 1
    selects {1, 2} and fetches 1; its attention covers block 0 alone."""
    d, bs = 3, 1
    K = _bits([[1, 0, 0], [0.5, 1, 0], [0, 0.5, 0]]).reshape(1, 1, 3, d)
    V = _bits([[3, 0, 0], [0, 5, 0], [0, 0, 7]]).reshape(1, 1, 3, d)
    host = np.stack([K.reshape(1, 1, 3, bs, d), V.reshape(1, 1, 3, bs, d)], axis=3)
    b2s = np.full((1, 1, 3), -1, np.int32)
    s2b = np.full((1, 1, 2), -1, np.int32)
    lu = np.full((1, 1, 2), -1, np.int32)
    kp = np.zeros((1, 1, 2, bs, d), np.uint16)
    vp = np.zeros_like(kp)
    q = _bits([[1, 1, 1]]).reshape(1, 1, d)
    r0 = ref.layer_step(K, _bits([[1, 0, 0]]).reshape(1, 1, 1, d), q, [3], host, kp, vp, b2s, s2b, lu, 2, 1, 0,
                        bs=bs)
    assert r0["S"][(0, 0)] == [0, 1] and r0["F"][(0, 0)] == [0]
    r1 = ref.layer_step(K, _bits([[0, 1, 0]]).reshape(1, 1, 1, d), q, [3], host, kp, vp, b2s, s2b, lu, 2, 1, 1,
                        bs=bs, prev_S=r0["S"])
    assert r1["S"][(0, 0)] == [1, 2] and r1["F"][(0, 0)] == [1]
    assert r1["A"][(0, 0)] == [0]
    np.testing.assert_allclose(r1["out"][0, 0], [3, 0, 0])
