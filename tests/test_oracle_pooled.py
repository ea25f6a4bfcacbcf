"""Pins of the oracle's min/max pooled-key scoring (Figure 7, left).

Pooling against its definition (per-dimension extremes of the valid tokens only);
pooled scores against brute-force enumeration in exact rationals; the upper-bound
property over the max-dot score, its equality case (one valid token), a hand
example where the two scores rank blocks differently, and planted blocks."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn


def _bits(x):
    return syn.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _frac(bits):
    return Fraction(float(ref.bf16_to_f64(np.uint16(bits))))


def test_pool_keys_extremes_of_valid_tokens_only():
    rng = np.random.default_rng(1)
    bs, d, nb_max, ctx = 4, 8, 5, 14
    K = rng.standard_normal((nb_max * bs, d)).astype(np.float32)
    K[ctx:] = 1e6  # tokens past ctx must not count
    hi, lo = ref.pool_keys(_bits(K), ctx, nb_max, bs)
    Kv = ref.bf16_to_f64(_bits(K))
    for x in range(nb_max):
        rows = [t for t in range(x * bs, (x + 1) * bs) if t < ctx]
        if not rows:
            assert (hi[x] == 0).all() and (lo[x] == 0).all()
            continue
        np.testing.assert_array_equal(ref.bf16_to_f64(hi[x]), Kv[rows].max(axis=0))
        np.testing.assert_array_equal(ref.bf16_to_f64(lo[x]), Kv[rows].min(axis=0))


@pytest.mark.parametrize("extreme", [False, True])
def test_pooled_scores_match_bruteforce(extreme):
    rng = np.random.default_rng(2)
    bs, d, nb, N = 4, 8, 4, 3
    K = rng.standard_normal((nb * bs, d)).astype(np.float32)
    Q = rng.standard_normal((N, d)).astype(np.float32)
    if extreme:  # exponent spread beyond float64's 53 bits forces the exact integer path
        K[5, 2] = 2.0 ** 50
        K[6, 3] = 2.0 ** -80
        Q[1, 3] = 2.0 ** -70
    hi, lo = ref.pool_keys(_bits(K), nb * bs, nb, bs)
    Qf = ref.bf16_to_f64(_bits(Q))
    score, key = ref.head_block_scores_pooled(hi, lo, Qf, nb)
    for x in range(nb):
        best = None
        for n in range(N):
            v = sum(max(_frac(_bits(Q)[n, i]) * _frac(hi[x, i]), _frac(_bits(Q)[n, i]) * _frac(lo[x, i]))
                    for i in range(d))
            best = v if best is None or v > best else best
        assert Fraction(key[x], 2 ** 266) == best


def test_pooled_score_bounds_max_dot_and_is_tight_for_one_token():
    rng = np.random.default_rng(3)
    bs, d = 16, 32
    for seed in range(4):
        ctx = 16 * 5 + 1  # the last block holds one valid token
        K = _bits(rng.standard_normal((16 * 6, d)))
        Q = ref.bf16_to_f64(_bits(rng.standard_normal((4, d))))
        hi, lo = ref.pool_keys(K, ctx, 6, bs)
        nb = -(-ctx // bs)
        _, kp = ref.head_block_scores_pooled(hi, lo, Q, nb)
        _, km = ref.head_block_scores(ref.bf16_to_f64(K), Q, ctx, bs)
        assert all(a >= b for a, b in zip(kp, km))
        assert kp[nb - 1] == km[nb - 1]
        assert any(a > b for a, b in zip(kp, km))


def test_hand_example_pooled_and_max_dot_rank_differently():
    """Block 0 keys (1,0) and (0,1): max-dot with q=(1,1) is 1, pooled box corner
    (1,1) gives 2.  Block 1 key (0.875,0.875): both give 1.75.  With Kb = 1 the
    max-dot score keeps block 1, the pooled score keeps block 0."""
    d, bs = 2, 2
    K = _bits([[1, 0], [0, 1], [0.875, 0.875], [0.875, 0.875]]).reshape(1, 1, 4, d)
    q = _bits([[1, 1]]).reshape(1, 1, d)
    qla = q.reshape(1, 1, 1, d)
    V = np.zeros_like(K)
    host = np.stack([K.reshape(1, 1, 2, bs, d), V.reshape(1, 1, 2, bs, d)], axis=3)
    for scoring, want in (("maxdot", [1]), ("pooled", [0])):
        b2s = np.full((1, 1, 2), -1, np.int32)
        s2b = np.full((1, 1, 1), -1, np.int32)
        lu = np.full((1, 1, 1), -1, np.int32)
        kp = np.zeros((1, 1, 1, bs, d), np.uint16)
        vp = np.zeros_like(kp)
        r = ref.layer_step(K, qla, q, [4], host, kp, vp, b2s, s2b, lu, 1, 1, 0, bs=bs, scoring=scoring)
        assert r["S"][(0, 0)] == want
        sc, key = r["score"][(0, 0)]
        exp = {"maxdot": [1.0, 1.75], "pooled": [2.0, 1.75]}[scoring]
        np.testing.assert_allclose(sc * np.sqrt(d), exp)


def test_planted_blocks_rank_top_under_pooling():
    rng = np.random.default_rng(4)
    bs, d, nb, n_hot = 16, 128, 40, 8
    K = 0.05 * rng.standard_normal((nb * bs, d))
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    hot = sorted(rng.choice(nb, size=n_hot, replace=False).tolist())
    for x in hot:
        K[x * bs:(x + 1) * bs] += 3 * u
    q = 2 * u + 0.05 * rng.standard_normal(d)
    hi, lo = ref.pool_keys(_bits(K), nb * bs, nb, bs)
    _, key = ref.head_block_scores_pooled(hi, lo, ref.bf16_to_f64(_bits(q[None])), nb)
    assert ref.topk_select(key, n_hot) == hot
