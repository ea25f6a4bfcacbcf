"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a hand-derived example, a brute-force
enumeration in exact rational arithmetic, a closed form, a textbook routine
(dense softmax attention), or an invariant that the definitions fix.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    return syn.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- golden
def test_golden_hand_two_steps():
    g = json.load(open(os.path.join(GOLDEN, "hand_two_steps.json")))
    sh = g["shape"]
    bs, d = sh["bs"], sh["d"]
    K = _bits(g["keys"]).reshape(1, 1, -1, d)
    V = _bits(g["values"]).reshape(1, 1, -1, d)
    qla = _bits(g["q_la"]).reshape(1, 1, 1, d)
    q = _bits(g["q"]).reshape(1, 1, d)
    ctx = [g["ctx"]]
    nbm = sh["nb_max"]
    host = np.stack([K.reshape(1, 1, nbm, bs, d), V.reshape(1, 1, nbm, bs, d)], axis=3)
    b2s = np.array([g["initial"]["blk2slot"]], np.int32).reshape(1, 1, -1)
    s2b = np.array([g["initial"]["slot2blk"]], np.int32).reshape(1, 1, -1)
    lu = np.array([g["initial"]["last_used"]], np.int32).reshape(1, 1, -1)
    kp = np.zeros((1, 1, sh["P"], bs, d), np.uint16)
    vp = np.zeros_like(kp)
    for p, x in enumerate(s2b[0, 0]):
        if x >= 0:
            kp[0, 0, p] = host[0, 0, x, 0]
            vp[0, 0, p] = host[0, 0, x, 1]
    for tag in ("step5", "step6"):
        exp = g[tag]
        r = ref.layer_step(K, qla, q, ctx, host, kp, vp, b2s, s2b, lu, sh["Kb"], sh["C"],
                           exp["step"], bs=bs)
        if "block_scores_unscaled" in exp:
            sc, key = r["score"][(0, 0)]
            np.testing.assert_array_equal(sc * math.sqrt(d), exp["block_scores_unscaled"])
        assert r["S"][(0, 0)] == exp["S"]
        assert r["F"][(0, 0)] == exp["F"]
        assert r["A"][(0, 0)] == exp["A"]
        assert b2s[0, 0].tolist() == exp["blk2slot"]
        assert s2b[0, 0].tolist() == exp["slot2blk"]
        assert lu[0, 0].tolist() == exp["last_used"]
        np.testing.assert_allclose(r["out"][0], exp["out"], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- a1 brute force
def _frac(bits):
    return Fraction(float(ref.bf16_to_f64(np.uint16(bits))))


def _brute_scores(Kbits, qlabits, ctx, bs):
    """max over (j, g, t) of q.k in exact rationals, by explicit loops."""
    B, Hkv, T, d = Kbits.shape
    n_la, Hq = qlabits.shape[1], qlabits.shape[2]
    G = Hq // Hkv
    out = {}
    for b in range(B):
        for h in range(Hkv):
            nb = -(-ctx[b] // bs)
            res = []
            for blk in range(nb):
                best = None
                for j in range(n_la):
                    for g in range(G):
                        for t in range(blk * bs, min(ctx[b], (blk + 1) * bs)):
                            v = sum(_frac(qlabits[b, j, h * G + g, i]) * _frac(Kbits[b, h, t, i])
                                    for i in range(d))
                            best = v if best is None or v > best else best
                res.append(best)
            out[(b, h)] = res
    return out


@pytest.mark.parametrize("extreme", [False, True])
def test_block_scores_match_bruteforce(extreme):
    rng = np.random.default_rng(7)
    B, Hkv, G, n_la, d, bs = 2, 2, 2, 3, 8, 4
    ctx = [13, 9]
    T = 16
    Kf = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
    Q = rng.standard_normal((B, n_la, Hkv * G, d)).astype(np.float32)
    if extreme:
        # exponent spread beyond float64's 53 bits forces the exact integer path
        Kf[0, 1, 2, 3] = 2.0 ** -100
        Kf[0, 1, 2, 4] = 2.0 ** 40
        Q[0, 1, 2, 3] = 2.0 ** -90
        Kf[1, 0, 5, :] = 2.0 ** -120
        Kf[1, 0, 5, 0] = 2.0 ** 60
    Kb, Qb = _bits(Kf), _bits(Q)
    got = ref.block_scores(Kb, Qb, ctx, bs)
    want = _brute_scores(Kb, Qb, ctx, bs)
    for key in want:
        sc, exact = got[key]
        assert len(exact) == len(want[key])
        for blk, w in enumerate(want[key]):
            assert Fraction(exact[blk], 2 ** 266) == w
            assert sc[blk] == pytest.approx(float(w) / math.sqrt(d), rel=1e-12, abs=1e-300)


def test_scores_use_hG_plus_g_query_heads():
    """Only query heads hG..hG+G-1 of the lookahead queries score KV head h."""
    B, Hkv, G, n_la, d, bs = 1, 2, 2, 1, 4, 2
    K = np.zeros((B, Hkv, 4, d), np.float32)
    K[0, 0, 0, 0] = 1.0      # head 0, block 0
    K[0, 0, 2, 1] = 1.0      # head 0, block 1
    K[0, 1, 0, 2] = 1.0      # head 1, block 0
    K[0, 1, 2, 3] = 1.0      # head 1, block 1
    Q = np.zeros((B, n_la, Hkv * G, d), np.float32)
    Q[0, 0, 0, 0] = 3.0      # q-head 0 (group of KV head 0) likes dim 0
    Q[0, 0, 1, 1] = 5.0      # q-head 1 (group of KV head 0) likes dim 1
    Q[0, 0, 2, 3] = 7.0      # q-head 2 (group of KV head 1) likes dim 3
    Q[0, 0, 3, 2] = 2.0      # q-head 3 (group of KV head 1) likes dim 2
    got = ref.block_scores(_bits(K), _bits(Q), [4], bs)
    s = math.sqrt(d)
    np.testing.assert_allclose(got[(0, 0)][0] * s, [3.0, 5.0])
    np.testing.assert_allclose(got[(0, 1)][0] * s, [2.0, 7.0])


# ---------------------------------------------------------------- a2
def _assert_topk_valid(key, S, Kb):
    nb = len(key)
    assert S == sorted(S)
    assert len(S) == min(Kb, nb)
    out = set(range(nb)) - set(S)
    for i in S:
        for j in out:
            assert key[i] > key[j] or (key[i] == key[j] and i < j)


def test_topk_invariants_random_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(200):
        nb = int(rng.integers(1, 40))
        Kb = int(rng.integers(1, 45))
        key = [int(v) for v in rng.integers(-5, 6, nb)]   # many exact ties
        S = ref.topk_select(key, Kb)
        _assert_topk_valid(key, S, Kb)


def test_topk_bruteforce_subsets():
    """S is the unique subset whose sorted (-key, index) list is lexicographically least."""
    rng = np.random.default_rng(4)
    for trial in range(50):
        nb = int(rng.integers(1, 8))
        Kb = int(rng.integers(1, 8))
        key = [int(v) for v in rng.integers(-2, 3, nb)]
        k = min(Kb, nb)
        best = min(itertools.combinations(range(nb), k),
                   key=lambda c: sorted((-key[i], i) for i in c))
        assert ref.topk_select(key, Kb) == sorted(best)


def test_duplicate_blocks_tie_to_lower_index():
    rng = np.random.default_rng(5)
    d, bs, nb = 8, 4, 6
    K = (0.01 * rng.standard_normal((1, 1, nb * bs, d))).astype(np.float32)
    K[0, 0, 1 * bs:2 * bs] = 1.0 + rng.random((bs, d)).astype(np.float32)
    K[0, 0, 4 * bs:5 * bs] = K[0, 0, 1 * bs:2 * bs]         # exact duplicate of block 1
    Q = np.ones((1, 1, 1, d), np.float32)
    r = ref.block_scores(_bits(K), _bits(Q), [nb * bs], bs)
    sc, key = r[(0, 0)]
    assert key[1] == key[4]
    assert ref.topk_select(key, 1) == [1]
    assert ref.topk_select(key, 2) == [1, 4]


def test_planted_blocks_rank_top():
    rng = np.random.default_rng(6)
    d, bs, nb, n_hot = 32, 16, 40, 8
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    K = 0.1 * rng.standard_normal((nb * bs, d))
    hot = sorted(rng.choice(nb, n_hot, replace=False).tolist())
    for x in hot:
        K[x * bs:(x + 1) * bs] += 10 * u
    Q = (u + 0.05 * rng.standard_normal((2, d)))[None, :, None, :]
    r = ref.block_scores(_bits(K[None, None]), _bits(Q), [nb * bs], bs)
    assert ref.topk_select(r[(0, 0)][1], n_hot) == hot


# ---------------------------------------------------------------- a3 / a4
def test_fetch_list_is_highest_missing():
    rng = np.random.default_rng(8)
    for trial in range(200):
        nb = int(rng.integers(1, 30))
        key = [int(v) for v in rng.integers(-4, 5, nb)]
        S = ref.topk_select(key, int(rng.integers(1, 20)))
        b2s = np.full(nb, -1, np.int32)
        for x in rng.choice(nb, int(rng.integers(0, nb + 1)), replace=False):
            b2s[x] = 0
        C = int(rng.integers(0, 8))
        F = ref.fetch_diff_capped(S, b2s, C, key)
        M = [x for x in S if b2s[x] < 0]
        assert F == sorted(F) and set(F) <= set(M)
        assert len(F) == min(C, len(M))
        for x in F:
            for y in set(M) - set(F):
                assert key[x] > key[y] or (key[x] == key[y] and x < y)


def test_lru_victims_by_hand():
    # slots:        0   1   2   3   4   5
    s2b = np.array([10, 11, -1, 12, 13, 14], np.int32)
    lu = np.array([3, 1, -1, 1, 0, 0], np.int32)
    b2s = np.full(32, -1, np.int32)
    for p, x in enumerate(s2b):
        if x >= 0:
            b2s[x] = p
    S = [11, 14, 20, 21, 22, 23]
    F = [20, 21, 22, 23]
    copies = ref.assign_slots(S, F, b2s, s2b, lu, step=7)
    # candidates: free slot 2; victims outside S by (last_used, block): 13 (0) @4, 12 (1) @3, 10 (3) @0
    assert copies == [(20, 2), (21, 4), (22, 3), (23, 0)]
    assert s2b.tolist() == [23, 11, 20, 22, 21, 14]
    assert b2s[10] == b2s[12] == b2s[13] == -1
    assert lu.tolist() == [7, 7, 7, 7, 7, 7]


def test_lru_equal_last_used_evicts_lower_block():
    s2b = np.array([9, 4, 7], np.int32)
    lu = np.array([2, 2, 2], np.int32)
    b2s = np.full(16, -1, np.int32)
    for p, x in enumerate(s2b):
        b2s[x] = p
    copies = ref.assign_slots([1], [1], b2s, s2b, lu, step=3)
    assert copies == [(1, 1)]                    # block 4 (lowest) is evicted first
    assert s2b.tolist() == [9, 1, 7] and lu.tolist() == [2, 3, 2]


def _tiny_state(w, layer=0):
    K, V = syn.layer_kv(w, layer)
    host = syn.host_tier_from_kv(w, K, V)
    b2s, s2b, lu = syn.initial_tables(w, layer)
    kp, vp = syn.pools_from_tables(w, host, s2b)
    return K, V, host, b2s, s2b, lu, kp, vp


def _small_workload(**kw):
    base = dict(name="small", L=1, B=2, Hq=8, Hkv=2, ctx=[700, 333], Kb=8, C=3,
                n_hot=4, d=32, steps=4)
    base.update(kw)
    return syn.Workload(**base)


def test_cap_zero_with_empty_resident_set_changes_nothing():
    w = _small_workload(C=0)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    b2s[:] = -1
    s2b[:] = -1
    q, qla = syn.layer_queries(w, 0, 0)
    r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, 0, 0, bs=w.bs)
    assert (b2s == -1).all() and (s2b == -1).all() and (lu == -1).all()
    for key in r["F"]:
        assert r["F"][key] == [] and r["A"][key] == []
    assert (r["out"] == 0).all()


def test_fetch_all_from_empty_makes_resident_equal_selected():
    w = _small_workload(C=8)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    b2s[:] = -1
    s2b[:] = -1
    q, qla = syn.layer_queries(w, 0, 0)
    r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.Kb, 4, bs=w.bs)
    for (b, h), S in r["S"].items():
        resident = sorted(int(x) for x in s2b[b, h] if x >= 0)
        assert resident == S == r["A"][(b, h)]
        for x in S:
            assert (kp[b, h, b2s[b, h, x]] == host[b, h, x, 0]).all()


def test_full_budget_fetch_all_equals_dense_attention():
    w = _small_workload(ctx=[333, 97], Kb=64, C=64, P=64)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    q, qla = syn.layer_queries(w, 0, 0)
    r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 1, bs=w.bs)
    G = w.G
    for b in range(w.B):
        for hq in range(w.Hq):
            h = hq // G
            k = ref.bf16_to_f64(K[b, h, : w.ctx[b]])
            v = ref.bf16_to_f64(V[b, h, : w.ctx[b]])
            qq = ref.bf16_to_f64(q[b, hq])
            dense = softmax(k @ qq / math.sqrt(w.d)) @ v
            np.testing.assert_allclose(r["out"][b, hq], dense, rtol=1e-12, atol=1e-12)


def test_single_token_context_returns_its_value():
    w = _small_workload(ctx=[1, 1], Kb=4, C=4)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    q, qla = syn.layer_queries(w, 0, 0)
    r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 0, bs=w.bs)
    for b in range(w.B):
        for hq in range(w.Hq):
            np.testing.assert_array_equal(r["out"][b, hq], ref.bf16_to_f64(V[b, hq // w.G, 0]))


def test_two_token_closed_form_with_scale():
    q = _bits([[1.0, 0.0, 0.0, 0.0]])
    kp = np.zeros((1, 2, 4), np.uint16)
    vp = np.zeros((1, 2, 4), np.uint16)
    kp[0, 0] = _bits([2.0, 0, 0, 0])
    kp[0, 1] = _bits([-1.0, 0, 0, 0])
    vp[0, 0] = _bits([1.0, 0, 0, 0])
    vp[0, 1] = _bits([0.0, 1, 0, 0])
    b2s = np.array([0], np.int32)
    o = ref.head_sparse_attention(q, kp, vp, [0], b2s, ctx=2, scale=0.5, bs=2)
    p = 1.0 / (1.0 + math.exp(-0.5 * 3.0))       # logits 1.0 and -0.5
    np.testing.assert_allclose(o[0], [p, 1 - p, 0, 0], rtol=0, atol=1e-15)


def test_multistep_table_invariants():
    w = _small_workload(steps=5)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    for step in range(w.steps):
        q, qla = syn.layer_queries(w, 0, step)
        before = {(b, h): set(int(x) for x in s2b[b, h] if x >= 0)
                  for b in range(w.B) for h in range(w.Hkv)}
        r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step, bs=w.bs)
        for (b, h), S in r["S"].items():
            R0 = before[(b, h)]
            R1 = set(int(x) for x in s2b[b, h] if x >= 0)
            F = r["F"][(b, h)]
            assert set(F) <= set(S) - R0
            assert len(F) == min(w.C, len(set(S) - R0))
            assert len(R1) <= w.P
            assert R1 == (R0 - (R0 - R1)) | set(F)
            assert (R0 - R1) <= (R0 - set(S))
            assert set(r["A"][(b, h)]) == set(S) & R1
            for p in range(w.P):
                x = s2b[b, h, p]
                if x >= 0:
                    assert b2s[b, h, x] == p
                    assert (kp[b, h, p] == host[b, h, x, 0]).all()
                    assert (vp[b, h, p] == host[b, h, x, 1]).all()
            assert (b2s[b, h] >= 0).sum() == len(R1)
            for x in r["A"][(b, h)]:
                assert lu[b, h, b2s[b, h, x]] == step


# ---------------------------------------------------------------- token append
def test_append_then_full_budget_attention_is_dense_over_the_new_context():
    w = _small_workload(ctx=[333, 96], Kb=64, C=64, P=64, nb_max=24)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    ctx = list(w.ctx)
    kn, vn = syn.append_tokens(w, 0, 0)
    ref.append_token(K, host, kp, vp, b2s, ctx, kn, vn, bs=w.bs)
    assert ctx == [334, 97]
    for b in range(w.B):
        t = ctx[b] - 1
        assert (K[b, :, t] == kn[b]).all() and (V[b, :, t] == 0).all()   # V lives in the host tier
        assert (host[b, :, t // 16, 0, t % 16] == kn[b]).all()
        assert (host[b, :, t // 16, 1, t % 16] == vn[b]).all()
        for h in range(w.Hkv):
            p = b2s[b, h, t // 16]
            if p >= 0:
                assert (kp[b, h, p, t % 16] == kn[b, h]).all() and (vp[b, h, p, t % 16] == vn[b, h]).all()
    V2 = V.copy()
    for b in range(w.B):
        V2[b, :, ctx[b] - 1] = vn[b]
    q, qla = syn.layer_queries(w, 0, 0)
    r = ref.layer_step(K, qla, q, ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, 1, bs=w.bs)
    for b in range(w.B):
        for hq in range(w.Hq):
            h = hq // w.G
            k = ref.bf16_to_f64(K[b, h, :ctx[b]])
            v = ref.bf16_to_f64(V2[b, h, :ctx[b]])
            dense = softmax(k @ ref.bf16_to_f64(q[b, hq]) / math.sqrt(w.d)) @ v
            np.testing.assert_allclose(r["out"][b, hq], dense, rtol=1e-12, atol=1e-12)


def test_append_to_a_full_cache_changes_nothing():
    w = _small_workload(ctx=[64, 10], nb_max=4)
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    ctx = list(w.ctx)
    K0, host0 = K.copy(), host.copy()
    kn, vn = syn.append_tokens(w, 0, 0)
    ref.append_token(K, host, kp, vp, b2s, ctx, kn, vn, bs=w.bs)
    assert ctx == [64, 11]
    assert (K[0] == K0[0]).all() and (host[0] == host0[0]).all()


def test_append_without_advance_keeps_the_length():
    w = _small_workload(ctx=[40, 10])
    K, V, host, b2s, s2b, lu, kp, vp = _tiny_state(w)
    ctx = list(w.ctx)
    kn, vn = syn.append_tokens(w, 0, 3)
    ref.append_token(K, host, kp, vp, b2s, ctx, kn, vn, bs=w.bs, advance=False)
    assert ctx == [40, 10] and (K[0, :, 40] == kn[0]).all()
