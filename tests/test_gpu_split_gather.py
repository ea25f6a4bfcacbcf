"""The gather in two halves (oasis_assign_slots + oasis_copy_fetched) and the copy
carried by a scoring launch (oasis_score_blocks_copy), against the oracle.

Tables and pools must come out bit-identical to the one-call gather's, which the
oracle fixes; the multi-layer decode step is checked layer by layer in both of
its launch orders (copy carried by the next layer's scoring, or the whole gather
after each selection)."""
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


@pytest.mark.parametrize("gather", ["split", "carry"])
def test_tiny_workload_split_gather(gather):
    w = syn.tiny()
    c = Case(w)
    for step in range(3):
        c.step(step, gather=gather)


@pytest.mark.parametrize("gather", ["split", "carry"])
def test_ragged_and_fetch_all_split_gather(gather):
    w = syn.Workload("ragged", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=32, n_hot=16)
    c = Case(w)
    for step in range(2):
        c.step(step, gather=gather)


def test_cap_zero_copy_is_a_no_op():
    w = syn.Workload("cap0", L=1, B=2, Hq=32, Hkv=8, ctx=[2048, 999], Kb=32, C=0, n_hot=16)
    c = Case(w)
    c.step(0, gather="carry")


def _multi_layer(copy, L=3, steps=3, host_alloc="cuda", dynamic=False):
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    w = syn.Workload("layers", L=L, B=2, Hq=32, Hkv=8, ctx=[3000, 1777], Kb=32, C=3, n_hot=16)
    st = DecodeState(w, l_phys=L, l_host=L, host_alloc=host_alloc)
    st.dynamic_scorer = dynamic
    layers = []
    for l in range(L):
        K, V = syn.layer_kv(w, l)
        host = syn.host_tier_from_kv(w, K, V)
        b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, l)]
        kp, vp = syn.pools_from_tables(w, host, s2b)
        st.fill_layer_numpy(l, K, V, b2s, s2b, lu)
        layers.append([K, host, b2s, s2b, lu, kp, vp])
    out = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device="cuda")
    for step in range(steps):
        qs = [syn.layer_queries(w, l, step) for l in range(L)]
        st.decode_step(step, [_dev_bits(qla) for _, qla in qs], [_dev_bits(q) for q, _ in qs],
                       out_layers=out, copy=copy)
        torch.cuda.synchronize()
        assert st.error_word() == 0
        for l in range(L):
            K, host, b2s, s2b, lu, kp, vp = layers[l]
            q, qla = qs[l]
            r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step)
            np.testing.assert_array_equal(st.blk2slot[l].cpu().numpy(), b2s)
            np.testing.assert_array_equal(st.slot2blk[l].cpu().numpy(), s2b)
            np.testing.assert_array_equal(st.last_used[l].cpu().numpy(), lu)
            kpool = st.k_pool[l].cpu().view(torch.int16).numpy().view(np.uint16)
            vpool = st.v_pool[l].cpu().view(torch.int16).numpy().view(np.uint16)
            occ = s2b >= 0
            np.testing.assert_array_equal(kpool[occ], kp[occ])
            np.testing.assert_array_equal(vpool[occ], vp[occ])
            _check_out(out[l].cpu().numpy().astype(np.float64), r["out"], f"layer {l} step {step}")


@pytest.mark.parametrize("copy", ["carry", "gather", "overlap", "fork", "pipe"])
def test_multi_layer_decode_step_all_orders(copy):
    _multi_layer(copy, L=6 if copy == "pipe" else 3)


def test_multi_layer_decode_step_with_the_dynamic_scorer():
    _multi_layer("overlap", L=4, dynamic=True)


def test_dynamic_scorer_equals_the_static_one_and_leaves_its_counter_at_zero():
    """oasis_score_blocks_dynamic writes the same (approximation, bound) pairs as
    oasis_score_blocks with the mma.sync kernel, call after call, and leaves its
    work counter at zero."""
    from sparse_decode_attention_oasis_gb300 import binding as B
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    w = syn.Workload("dyn", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=4, n_hot=16)
    st = DecodeState(w, l_phys=1)
    K, V = syn.layer_kv(w, 0)
    st.fill_layer_numpy(0, K, V, *[np.array(t) for t in syn.initial_tables(w, 0)])
    _, qla = syn.layer_queries(w, 0, 0)
    q = _dev_bits(qla)
    s = st.shape
    ref_scores = torch.zeros((w.B, w.Hkv, w.nb_max, 2), dtype=torch.float32, device="cuda")
    B.oasis_set_option(B.OPT_SCORE_KERNEL, B.SCORE_KERNEL_MMA)  # the dynamic scorer is the mma.sync kernel
    try:
        B.oasis_score_blocks(s, st.K[0], st.ctx, q, ref_scores)
    finally:
        B.oasis_set_option(B.OPT_SCORE_KERNEL, B.SCORE_KERNEL_TC)
    work = torch.zeros(2, dtype=torch.int32, device="cuda")
    try:
        for share in (750, 0, 500, 1000):  # per mille of the blocks in fixed shares
            B.oasis_set_option(B.OPT_SCORE_STATIC_SHARE, share)
            for reserve in (0, 16, 0):
                got = torch.zeros_like(ref_scores)
                B.oasis_score_blocks_dynamic(s, st.K[0], st.ctx, q, got, work, reserve)
                torch.cuda.synchronize()
                for b in range(w.B):
                    nb = w.nb(b)
                    assert torch.equal(got[b, :, :nb], ref_scores[b, :, :nb]), (share, reserve)
                assert work.tolist() == [0, 0]
    finally:
        B.oasis_set_option(B.OPT_SCORE_STATIC_SHARE, 750)


@pytest.mark.parametrize("host_alloc", ["thp", "thp_layers", "cuda_layers"])
def test_host_tier_allocations(host_alloc):
    _multi_layer("overlap", L=2, steps=2, host_alloc=host_alloc)


def test_pipe_order_with_fewer_scorer_ctas():
    from sparse_decode_attention_oasis_gb300 import binding as B

    B.oasis_set_option(B.OPT_SCORE_CTAS_PER_SM, 1)
    try:
        _multi_layer("pipe", L=5, steps=2)
    finally:
        B.oasis_set_option(B.OPT_SCORE_CTAS_PER_SM, 0)


def test_copy_reports_out_of_range_fetch_entry():
    """A fetch entry naming a block past nb_max is skipped and flagged; nothing else changes."""
    from sparse_decode_attention_oasis_gb300 import binding as B
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    w = syn.Workload("bad", L=1, B=1, Hq=32, Hkv=8, ctx=[1024], Kb=16, C=2, n_hot=4)
    st = DecodeState(w, l_phys=1)
    K, V = syn.layer_kv(w, 0)
    st.fill_layer_numpy(0, K, V, *[np.array(t) for t in syn.initial_tables(w, 0)])
    s = st.shape
    fetch = torch.full((w.B, w.Hkv, w.Kb), -1, dtype=torch.int32, device="cuda")
    nfetch = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device="cuda")
    fetch[0, 3, 0] = w.nb_max + 5
    nfetch[0, 3] = 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp0, vp0 = st.k_pool.clone(), st.v_pool.clone()
    B.oasis_copy_fetched(s, st.host[0], fetch, nfetch, st.blk2slot[0], st.k_pool[0], st.v_pool[0], err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.EW_BAD_BLOCK
    assert torch.equal(st.k_pool, kp0) and torch.equal(st.v_pool, vp0)


@pytest.mark.parametrize("call", ["gather", "assign"])
def test_out_of_range_sel_entry_leaves_resident_selected_blocks_alone(call):
    """An out-of-range last entry of S (still ascending) is flagged; every resident
    block of S keeps its slot and its LRU clock, as the oracle gives for S without
    that entry (the bad entry must not make a selected block a victim)."""
    from sparse_decode_attention_oasis_gb300 import binding as B
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    w = syn.Workload("badsel", L=1, B=1, Hq=32, Hkv=8, ctx=[1024], Kb=16, C=4, n_hot=4)
    st = DecodeState(w, l_phys=1)
    K, V = syn.layer_kv(w, 0)
    b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, 0)]
    rng = np.random.default_rng(5)
    lu[...] = rng.integers(-1, 3, size=lu.shape).astype(np.int32)
    st.fill_layer_numpy(0, K, V, b2s, s2b, lu)
    sel = np.full((w.B, w.Hkv, w.Kb), -1, np.int32)
    nsel = np.zeros((w.B, w.Hkv), np.int32)
    fetch = np.full((w.B, w.Hkv, w.Kb), -1, np.int32)
    nfetch = np.zeros((w.B, w.Hkv), np.int32)
    want = {}
    for h in range(w.Hkv):
        res = sorted(int(x) for x in s2b[0, h] if x >= 0)
        missing = sorted(set(range(w.nb(0))) - set(res))
        # the 11 largest resident blocks (the end of S, where the bad entry sits) and 4 missing ones
        S = sorted(res[-11:] + [int(x) for x in rng.choice(missing, 4, replace=False)])
        F = sorted(x for x in S if b2s[0, h, x] < 0)
        bad = S + [w.nb_max + 3] if h % 2 == 0 else S   # half of the heads carry the bad entry
        sel[0, h, :len(bad)] = bad
        nsel[0, h] = len(bad)
        fetch[0, h, :len(F)] = F
        nfetch[0, h] = len(F)
        want[h] = (S, F)
    step = 7
    for h, (S, F) in want.items():
        ref.assign_slots(S, F, b2s[0, h], s2b[0, h], lu[0, h], step)
    dev = lambda a: torch.from_numpy(a).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stepd = torch.full((1,), step, dtype=torch.int32, device="cuda")
    s = st.shape
    if call == "gather":
        B.oasis_gather_h2d(s, st.host[0], dev(sel), dev(nsel), dev(fetch), dev(nfetch), st.blk2slot[0],
                           st.slot2blk[0], st.last_used[0], stepd, st.k_pool[0], st.v_pool[0], err)
    else:
        B.oasis_assign_slots(s, dev(sel), dev(nsel), dev(fetch), dev(nfetch), st.blk2slot[0], st.slot2blk[0],
                             st.last_used[0], stepd, err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.EW_BAD_BLOCK
    np.testing.assert_array_equal(st.blk2slot[0].cpu().numpy(), b2s)
    np.testing.assert_array_equal(st.slot2blk[0].cpu().numpy(), s2b)
    np.testing.assert_array_equal(st.last_used[0].cpu().numpy(), lu)


def test_cross_step_pipeline_matches_oracle():
    """copy="lag": step 0 selects, gathers and attends; later steps attend the
    previous step's selection first (oracle prev_S), then select and gather."""
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    L = 2
    w = syn.Workload("lag", L=L, B=2, Hq=32, Hkv=8, ctx=[2500, 1234], Kb=32, C=3, n_hot=16)
    st = DecodeState(w, l_phys=L, l_host=L)
    layers = []
    for l in range(L):
        K, V = syn.layer_kv(w, l)
        host = syn.host_tier_from_kv(w, K, V)
        b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, l)]
        kp, vp = syn.pools_from_tables(w, host, s2b)
        st.fill_layer_numpy(l, K, V, b2s, s2b, lu)
        layers.append([K, host, b2s, s2b, lu, kp, vp, None])
    out = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device="cuda")
    for step in range(4):
        qs = [syn.layer_queries(w, l, step) for l in range(L)]
        st.decode_step(step, [_dev_bits(qla) for _, qla in qs], [_dev_bits(q) for q, _ in qs],
                       out_layers=out, copy="lag")
        torch.cuda.synchronize()
        assert int(st.scratch.err.item()) == 0 and int(st.scratch2.err.item()) == 0
        for l in range(L):
            K, host, b2s, s2b, lu, kp, vp, prev = layers[l]
            q, qla = qs[l]
            r = ref.layer_step(K, qla, q, w.ctx, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step, prev_S=prev)
            layers[l][7] = r["S"]
            np.testing.assert_array_equal(st.blk2slot[l].cpu().numpy(), b2s)
            np.testing.assert_array_equal(st.slot2blk[l].cpu().numpy(), s2b)
            np.testing.assert_array_equal(st.last_used[l].cpu().numpy(), lu)
            _check_out(out[l].cpu().numpy().astype(np.float64), r["out"], f"layer {l} step {step}")


def test_touch_host_reads_a_pinned_range():
    from sparse_decode_attention_oasis_gb300 import binding as B

    host = torch.arange(1 << 20, dtype=torch.int32).pin_memory()
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.oasis_touch_host(host, sink=sink)
    B.oasis_touch_host(host, nbytes=4096 + 16)
    torch.cuda.synchronize()
    assert int(sink.item()) == 0
    with pytest.raises(B.OasisError):
        B.oasis_touch_host(host, nbytes=100)  # not a multiple of 16


@pytest.mark.parametrize("scoring", ["maxdot", "pooled"])
def test_decode_steps_with_appends_in_every_layer(scoring):
    """append_step (every layer gets the step's token, ctx advances once) then a
    decode step, against the oracle's per-layer appends and layer steps."""
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    L = 3
    ctx0 = [1000, 1531, 2047]
    w = syn.Workload("grow", L=L, B=3, Hq=32, Hkv=8, ctx=list(ctx0), Kb=32, C=2, n_hot=16,
                     nb_max=-(-(max(ctx0) + 20) // 16))
    st = DecodeState(w, l_phys=L, l_host=L, scoring=scoring)
    layers = []
    for l in range(L):
        K, V = syn.layer_kv(w, l)
        host = syn.host_tier_from_kv(w, K, V)
        b2s, s2b, lu = [np.array(t) for t in syn.initial_tables(w, l)]
        kp, vp = syn.pools_from_tables(w, host, s2b)
        st.fill_layer_numpy(l, K, V, b2s, s2b, lu)
        layers.append([K, host, b2s, s2b, lu, kp, vp])
    out = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device="cuda")
    ctx_ref = list(ctx0)
    for step in range(4):
        news = [syn.append_tokens(w, l, step) for l in range(L)]
        st.append_step(torch.stack([_dev_bits(k) for k, _ in news]), torch.stack([_dev_bits(v) for _, v in news]))
        for l in range(L):
            K, host, b2s, s2b, lu, kp, vp = layers[l]
            ref.append_token(K, host, kp, vp, b2s, ctx_ref, news[l][0], news[l][1], advance=(l == L - 1))
        w.ctx = list(ctx_ref)
        qs = [syn.layer_queries(w, l, step) for l in range(L)]
        st.decode_step(step, [_dev_bits(qla) for _, qla in qs], [_dev_bits(q) for q, _ in qs], out_layers=out,
                       copy="overlap")
        torch.cuda.synchronize()
        assert st.error_word() == 0
        np.testing.assert_array_equal(st.ctx.cpu().numpy(), np.array(ctx_ref))
        for l in range(L):
            K, host, b2s, s2b, lu, kp, vp = layers[l]
            q, qla = qs[l]
            r = ref.layer_step(K, qla, q, ctx_ref, host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step, scoring=scoring)
            np.testing.assert_array_equal(st.blk2slot[l].cpu().numpy(), b2s)
            np.testing.assert_array_equal(st.slot2blk[l].cpu().numpy(), s2b)
            _check_out(out[l].cpu().numpy().astype(np.float64), r["out"], f"layer {l} step {step}")
