"""Pins of the oracle's agreement counters (Figure 6 / Figure 4 analogue).

The exact top-K of the true query is checked against a brute-force enumeration in
exact rationals over (g, t) with the true query heads hG+g, ranked by value with
ties to the lower block; the counts against a hand example and set identities."""
from fractions import Fraction

import numpy as np

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn


def _bits(x):
    return syn.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _frac(bits):
    return Fraction(float(ref.bf16_to_f64(np.uint16(bits))))


def test_exact_topk_of_true_query_matches_bruteforce():
    rng = np.random.default_rng(3)
    B, Hkv, G, d, bs, Kb = 2, 2, 2, 8, 4, 2
    ctx = [15, 10]
    T = 16
    Kbits = _bits(rng.standard_normal((B, Hkv, T, d)))
    qbits = _bits(rng.standard_normal((B, Hkv * G, d)))
    got = ref.exact_topk_true_query(Kbits, qbits, ctx, Kb, bs)
    for b in range(B):
        for h in range(Hkv):
            nb = -(-ctx[b] // bs)
            val = []
            for blk in range(nb):
                best = None
                for g in range(G):
                    for t in range(blk * bs, min(ctx[b], (blk + 1) * bs)):
                        v = sum(_frac(qbits[b, h * G + g, i]) * _frac(Kbits[b, h, t, i]) for i in range(d))
                        best = v if best is None or v > best else best
                val.append(best)
            order = sorted(range(nb), key=lambda x: (-val[x], x))
            assert got[(b, h)] == sorted(order[:min(Kb, nb)])


def test_exact_topk_uses_only_the_group_heads():
    """Changing a query head outside KV head h's group leaves h's exact set unchanged."""
    rng = np.random.default_rng(5)
    B, Hkv, G, d, bs, Kb = 1, 2, 2, 8, 4, 2
    Kbits = _bits(rng.standard_normal((B, Hkv, 16, d)))
    q = rng.standard_normal((B, Hkv * G, d)).astype(np.float32)
    a = ref.exact_topk_true_query(Kbits, _bits(q), [16], Kb, bs)
    q2 = q.copy()
    q2[0, 2:] = -q2[0, 2:]  # heads of KV head 1 only
    b_ = ref.exact_topk_true_query(Kbits, _bits(q2), [16], Kb, bs)
    assert a[(0, 0)] == b_[(0, 0)]


def test_agreement_counts_by_hand():
    b2s = np.full(10, -1, np.int32)
    b2s[[3, 7]] = [0, 1]
    assert ref.set_agreement([1, 3, 5, 7], [3, 4, 7, 9], b2s) == (2, 2, 4)
    assert ref.set_agreement([1, 3, 5, 7], [3, 4, 5, 9], b2s) == (2, 1, 4)
    assert ref.set_agreement([], [3, 4], b2s) == (0, 0, 2)


def test_agreement_identities():
    rng = np.random.default_rng(9)
    for _ in range(20):
        E = sorted(rng.choice(64, size=16, replace=False).tolist())
        P = sorted(rng.choice(64, size=16, replace=False).tolist())
        b2s = np.where(rng.random(64) < 0.5, 0, -1).astype(np.int32)
        hit, res, n = ref.set_agreement(P, E, b2s)
        assert ref.set_agreement(E, E, b2s)[0] == n == 16
        assert hit == len(set(P) & set(E)) and 0 <= res <= hit
        assert ref.set_agreement(P, E, np.zeros(64, np.int32))[1] == hit
        disjoint = [x for x in range(64) if x not in E][:16]
        assert ref.set_agreement(disjoint, E, b2s)[0] == 0


def test_planted_true_query_exact_set_is_the_hot_blocks():
    """Keys 0.1 N(0,1) plus 3u on Kb hot blocks, true query 2u + 0.1 N(0,1): the
    exact set is the hot set (hot scores ~6, the others well below 1)."""
    rng = np.random.default_rng(4)
    B, Hkv, G, d, bs, Kb, nb = 1, 2, 2, 128, 16, 8, 40
    K = 0.1 * rng.standard_normal((B, Hkv, nb * bs, d))
    q = 0.1 * rng.standard_normal((B, Hkv * G, d))
    hot = {}
    for h in range(Hkv):
        u = rng.standard_normal(d)
        u /= np.linalg.norm(u)
        hot[h] = sorted(rng.choice(nb, size=Kb, replace=False).tolist())
        for x in hot[h]:
            K[0, h, x * bs:(x + 1) * bs] += 3 * u
        q[0, h * G:(h + 1) * G] += 2 * u
    got = ref.exact_topk_true_query(_bits(K), _bits(q), [nb * bs], Kb, bs)
    for h in range(Hkv):
        assert got[(0, h)] == hot[h]
