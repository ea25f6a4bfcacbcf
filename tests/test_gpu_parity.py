"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bar: selected blocks, fetch lists, block tables and pool contents bit-exact;
block scores inside their certified interval; attention outputs within
abs 2e-3 or rel 1e-2 per element (bf16 inputs, fp32 accumulation).
"""
import math

import numpy as np
import pytest

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn

from gpu_helpers import Case, _check_out

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()


def test_tiny_workload_three_steps():
    w = syn.tiny()
    c = Case(w)
    for step in range(3):
        c.step(step)


def test_ragged_contexts_partial_blocks():
    w = syn.Workload("ragged", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=4, n_hot=16)
    c = Case(w)
    for step in range(2):
        c.step(step)


@pytest.mark.parametrize("Hq,n_la", [(64, 4), (8, 4), (16, 3)])
def test_gqa_groups(Hq, n_la):
    w = syn.Workload("gqa", L=1, B=2, Hq=Hq, Hkv=8, ctx=[2048, 1531], Kb=32, C=6, n_hot=16, n_la=n_la)
    c = Case(w)
    c.step(0)
    c.step(1)


def test_budget_covers_context_and_fetch_all_is_dense():
    w = syn.Workload("dense", L=1, B=2, Hq=32, Hkv=8, ctx=[500, 77], Kb=32, C=32, n_hot=4)
    blank = tuple(np.full_like(t, -1) for t in syn.initial_tables(w, 0))
    c = Case(w, tables=blank)
    r, sc = c.step(0)
    out = sc.out.cpu().numpy().astype(np.float64)
    q, _ = syn.layer_queries(w, 0, 0)
    for b in range(w.B):
        for hq in range(w.Hq):
            h = hq // w.G
            k = ref.bf16_to_f64(c.K[b, h, :w.ctx[b]])
            v = ref.bf16_to_f64(c.V[b, h, :w.ctx[b]])
            lg = k @ ref.bf16_to_f64(q[b, hq]) / math.sqrt(w.d)
            p = np.exp(lg - lg.max())
            _check_out(out[b, hq], p @ v / p.sum(), "dense")


def test_cap_zero_empty_resident_set():
    w = syn.Workload("cap0", L=1, B=1, Hq=32, Hkv=8, ctx=[3000], Kb=32, C=0, n_hot=8)
    blank = tuple(np.full_like(t, -1) for t in syn.initial_tables(w, 0))
    c = Case(w, tables=blank)
    r, sc = c.step(0)
    assert (c.st.blk2slot[0].cpu().numpy() == -1).all()
    assert (sc.out.cpu().numpy() == 0).all()


@pytest.mark.parametrize("ctx", [2048, 8192])
def test_duplicate_blocks_force_exact_ties(ctx):
    """48 identical top blocks straddle the rank-32 boundary: ties go to the lower index.

    128 blocks take the rank-count bracket; 512 take the histogram pass with the
    tied blocks inside the bin that holds the threshold."""
    w = syn.Workload("ties", L=1, B=1, Hq=32, Hkv=8, ctx=[ctx], Kb=32, C=8, n_hot=0)
    K, V = syn.layer_kv(w, 0)
    Kf = syn.bf16_bits_to_f32(K) * np.float32(1.0 / 64)     # power-of-two scaling is exact
    for h in range(w.Hkv):
        u = syn.unit_dir(w, 0, 0, h)
        Kf[0, h, 40 * 16:88 * 16] = 3.0 * u[None, :]
    K = syn.f32_to_bf16_bits(Kf)
    c = Case(w, K=K, V=V)
    r, _ = c.step(0)
    for h in range(w.Hkv):
        assert r["S"][(0, h)] == list(range(40, 72))
    c.step(1)


@pytest.mark.parametrize("ctx", [1024, 4800])
def test_all_zero_keys(ctx):
    """Every score ties at 0 and every block is uncertain (more than Kb: the batched
    refine).  300 blocks also put more than 256 entries in one histogram bin (the
    second histogram pass)."""
    w = syn.Workload("zeros", L=1, B=1, Hq=32, Hkv=8, ctx=[ctx], Kb=32, C=4, n_hot=0)
    K, V = syn.layer_kv(w, 0)
    K[:] = 0
    c = Case(w, K=K, V=V)
    r, _ = c.step(0)
    assert r["S"][(0, 0)] == list(range(32))


def test_difference_below_fp32_resolution_is_resolved_exactly():
    """Two blocks whose dots differ by 2^-24 of their value: fp32 ties them, exact does not."""
    w = syn.Workload("ulp", L=1, B=1, Hq=8, Hkv=8, ctx=[64 * 16], Kb=1, C=1, n_hot=0, n_la=1)
    K = np.zeros((1, 8, w.T_max, w.d), np.uint16)
    V = syn.f32_to_bf16_bits(np.random.default_rng(0).standard_normal((1, 8, w.T_max, w.d)).astype(np.float32))
    one = syn.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    for h in range(8):
        K[0, h, 3 * 16, 0] = one                 # block 3: q.k = 1
        K[0, h, 9 * 16 + 4, 0] = one             # block 9: q.k = 1 + 2^-24
        K[0, h, 9 * 16 + 4, 1] = one
    qla = np.zeros((1, 1, 8, w.d), np.float32)
    qla[..., 0] = 1.0
    qla[..., 1] = 2.0 ** -24
    q = np.ones((1, 8, w.d), np.float32)
    c = Case(w, K=K, V=V)
    r, sc = c.step(0, q=syn.f32_to_bf16_bits(q), qla=syn.f32_to_bf16_bits(qla))
    for h in range(8):
        assert r["S"][(0, h)] == [9]


def test_device_query_generator_matches_host():
    w = syn.qwen3_8b_decode(B=4, L=1)
    a = syn.QueryStream(w, 0)
    t = syn.QueryStreamTorch(w, 0, "cuda")
    for s in range(3):
        qa, la = a.next()
        qt, lt = t.next()
        assert (qt.cpu().view(torch.int16).numpy().view(np.uint16) == qa).all()
        assert (lt.cpu().view(torch.int16).numpy().view(np.uint16) == la).all()
    K, V = syn.kv_request_torch(w, 0, 1, "cuda")
    Kn, Vn = syn.head_kv(w, 0, 1, 3)
    assert (K[3].cpu().view(torch.int16).numpy().view(np.uint16) == Kn).all()


@pytest.mark.parametrize("scoring", ["maxdot", "pooled"])
def test_separate_topk_and_diff_kernels(scoring):
    """The decode path runs top-K and the diff as one launch; the two separate
    calls must give the same (oracle) results."""
    w = syn.Workload("ragged", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=4, n_hot=16)
    c = Case(w, scoring=scoring)
    c.st.fused_select = False
    for step in range(2):
        c.step(step)


def _two_block_case(k_rows, q_vals, want):
    """Keys zero except the given (block, token, dim) -> value entries; one lookahead
    query per head with the given (dim -> value); Kb = 1: the kept block must be want."""
    w = syn.Workload("exact", L=1, B=1, Hq=8, Hkv=8, ctx=[64 * 16], Kb=1, C=1, n_hot=0, n_la=1)
    K = np.zeros((1, 8, w.T_max, w.d), np.float32)
    for (blk, tok, dim), val in k_rows.items():
        K[0, :, blk * 16 + tok, dim] = val
    V = syn.f32_to_bf16_bits(np.random.default_rng(0).standard_normal((1, 8, w.T_max, w.d)).astype(np.float32))
    qla = np.zeros((1, 1, 8, w.d), np.float32)
    for dim, val in q_vals.items():
        qla[..., dim] = val
    q = np.ones((1, 8, w.d), np.float32)
    c = Case(w, K=syn.f32_to_bf16_bits(K), V=V)
    r, sc = c.step(0, q=syn.f32_to_bf16_bits(q), qla=syn.f32_to_bf16_bits(qla))
    for h in range(8):
        assert r["S"][(0, h)] == [want]


def test_exact_sum_beyond_fp64_resolution_uses_the_limb_path():
    """Dots 2^60 + 2^-60 (block 9) and 2^60 (block 3): 120 bits apart, so the fp64
    certificate fails and the 544-bit sum decides; block 9 must win."""
    _two_block_case({(3, 0, 0): 2.0 ** 30, (9, 5, 0): 2.0 ** 30, (9, 5, 1): 2.0 ** -30},
                    {0: 2.0 ** 30, 1: 2.0 ** -30}, 9)


def test_exact_negative_dots_compare_correctly():
    """All dots negative: -1 (block 4) beats -1 - 2^-20 (block 11) and -2 (the others);
    the exact sums are negative, so their limb encoding is two's complement."""
    rows = {}
    for blk in range(64):
        for tok in range(16):  # every token of a block negative, so its max-dot is negative
            rows[(blk, tok, 0)] = -1.0 if blk in (4, 11) else -2.0
            if blk == 11:
                rows[(blk, tok, 1)] = -(2.0 ** -20)
    _two_block_case(rows, {0: 1.0, 1: 1.0}, 4)


@pytest.mark.parametrize("C,scoring", [(256, "maxdot"), (7, "maxdot"), (7, "pooled")])
def test_largest_budget_slots_and_query_rows(C, scoring):
    """The largest shapes the ABI accepts in the per-head dimensions: a 256-block
    (4,096-token) budget, 1,024 slots per head and 32 query rows per KV head (GQA 8 x
    4 lookahead queries), over ragged contexts with more blocks than slots;
    fetch-all (C = Kb) and a small cap, three steps each."""
    w = syn.Workload("maxdims", L=1, B=2, Hq=16, Hkv=2, ctx=[32768 - 3, 20000], Kb=256, C=C, n_hot=64,
                     n_la=4, P=1024)
    # more blocks than slots, so the resident sets are partial and blocks are fetched
    assert w.Kb == 256 and w.P == 1024 and w.n_la * w.G == 32 and min(w.nb(b) for b in range(w.B)) > w.P
    c = Case(w, scoring=scoring)
    for step in range(3):
        c.step(step)
