"""The seeded input generator: host (numpy) and device (torch) draws are the same bits."""
import numpy as np
import pytest
import torch

from sparse_decode_attention_oasis_gb300 import synthetic as syn


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _w():
    return syn.Workload("t", L=2, B=3, Hq=16, Hkv=4, ctx=[100, 77, 300], Kb=8, C=2, n_hot=3, steps=4)


def test_hash_normals_numpy_equals_torch():
    a = syn.hash_normals(3, syn.STREAM_K, 1, 2, 3, 17, 5000)
    b = syn.hash_normals_torch(3, syn.STREAM_K, 1, 2, 3, 17, 5000, "cpu").numpy()
    assert (a.view(np.uint32) == b.view(np.uint32)).all()


def test_normal_draws_have_unit_moments():
    x = syn.hash_normals(0, syn.STREAM_V, 0, 0, 0, 0, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.var() - 1.0) < 1e-2
    assert len(np.unique(syn.hash_normals(0, 0, 0, 0, 1, 0, 1 << 16))) > 30000


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40], np.float32)
    assert syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(x)).tolist() == \
        torch.from_numpy(x).to(torch.bfloat16).float().tolist()


def test_keys_values_numpy_equals_torch():
    w = _w()
    for layer in range(2):
        for b in range(w.B):
            K, V = syn.kv_request_torch(w, layer, b, "cpu")
            for h in range(w.Hkv):
                Kn, Vn = syn.head_kv(w, layer, b, h)
                assert (_bits(K[h]) == Kn).all() and (_bits(V[h]) == Vn).all()
                Kh, Vh = syn.head_kv_torch(w, layer, b, h, "cpu")
                assert (_bits(Kh) == Kn).all() and (_bits(Vh) == Vn).all()


def test_query_streams_equal_the_per_step_draws():
    w = _w()
    for layer in range(2):
        a = syn.QueryStream(w, layer)
        t = syn.QueryStreamTorch(w, layer, "cpu")
        for s in range(4):
            q, qla = syn.layer_queries(w, layer, s)
            qa, la = a.next()
            qt, lt = t.next()
            assert (qa == q).all() and (la == qla).all()
            assert (_bits(qt) == q).all() and (_bits(lt) == qla).all()


def test_planted_blocks_carry_the_shift():
    w = _w()
    Kf, _ = syn.head_kv_f32(w, 0, 2, 1)
    base = syn.hash_normals(w.seed, syn.STREAM_K, 0, 2, 1, 0, w.ctx[2] * w.d).reshape(w.ctx[2], w.d)
    u = syn.unit_dir(w, 0, 2, 1)
    hot = syn.hot_blocks(w, 0, 2, 1)
    for x in range(w.nb(2)):
        rows = slice(x * 16, min(w.ctx[2], (x + 1) * 16))
        want = base[rows] + (np.float32(3.0) * u) if x in hot else base[rows]
        assert (Kf[rows] == want.astype(np.float32)).all()


def _wd():
    return syn.Workload("d", L=2, B=3, Hq=16, Hkv=4, ctx=[700, 77, 300], Kb=8, C=2, n_hot=8, steps=6,
                        hot_mode="drift", n_pool=24, rho_u=0.99)


def test_drift_keys_and_queries_numpy_equal_torch():
    w = _wd()
    for layer in range(2):
        for b in range(w.B):
            K, V = syn.kv_request_torch(w, layer, b, "cpu")
            for h in range(w.Hkv):
                Kn, Vn = syn.head_kv(w, layer, b, h)
                assert (_bits(K[h]) == Kn).all() and (_bits(V[h]) == Vn).all()
        a, t = syn.QueryStream(w, layer), syn.QueryStreamTorch(w, layer, "cpu")
        for s in range(5):
            q, qla = syn.layer_queries(w, layer, s)
            qa, la = a.next()
            qt, lt = t.next()
            assert (qa == q).all() and (la == qla).all()
            assert (_bits(qt) == q).all() and (_bits(lt) == qla).all()


def test_drift_pool_blocks_carry_their_own_directions():
    w = _wd()
    b, h = 0, 2
    Kf, _ = syn.head_kv_f32(w, 1, b, h)
    base = syn.hash_normals(w.seed, syn.STREAM_K, 1, b, h, 0, w.ctx[b] * w.d).reshape(w.ctx[b], w.d)
    pool = syn.pool_blocks(w, 1, b, h)
    a, c = syn.drift_plane(w, 1, b, h)
    assert abs(a @ a - 1) < 1e-12 and abs(c @ c - 1) < 1e-12 and abs(a @ c) < 1e-12
    assert len(set(pool.tolist())) == w.n_pool and pool.max() < w.nb(b)
    for i, x in enumerate(pool):
        phi = 2 * np.pi * i / w.n_pool
        v = np.cos(phi) * a + np.sin(phi) * c
        rows = slice(x * 16, min(w.ctx[b], (x + 1) * 16))
        assert (Kf[rows] == base[rows] + (3.0 * v).astype(np.float32)).all()
    others = np.setdiff1d(np.arange(w.nb(b)), pool)
    for x in others[:10]:
        rows = slice(x * 16, min(w.ctx[b], (x + 1) * 16))
        assert (Kf[rows] == base[rows]).all()


def test_drift_hot_set_is_an_arc_of_the_pool_that_moves():
    w = _wd()
    pool = syn.pool_blocks(w, 0, 0, 1).tolist()
    moved = 0
    prev = None
    for s in range(6):
        hot = syn.hot_set(w, 0, 0, 1, s)
        idx = sorted(pool.index(x) for x in hot)
        assert len(hot) == w.n_hot
        # consecutive pool indices modulo n_pool (one arc of the circle)
        gaps = [(idx[(k + 1) % len(idx)] - idx[k]) % w.n_pool for k in range(len(idx))]
        assert sorted(gaps)[:-1] == [1] * (len(idx) - 1)
        u = syn.query_dir(w, 0, 0, 1, s)
        al = syn.pool_dirs(w, 0, 0, 1) @ u
        assert min(al[pool.index(x)] for x in hot) >= max(al[i] for i in range(w.n_pool) if pool[i] not in hot)
        if prev is not None:
            moved += len(set(hot) - set(prev))
        prev = hot
    assert moved > 0


def test_long_output_hot_set_turns_over_about_five_percent_per_step():
    w = syn.long_output(B=8, L=1)
    assert w.hot_mode == "drift" and w.n_pool == 256 and w.n_hot == 64 and w.rho_u == 0.997
    t = syn.hot_set_turnover(w, 0, 64)
    assert 0.035 <= t <= 0.065, t
    # the fixed-set workloads never move
    assert syn.hot_set_turnover(syn.tiny(), 0, 8) == 0.0
