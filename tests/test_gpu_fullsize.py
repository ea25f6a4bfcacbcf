"""Full-size parity: whole decode steps of the benchmark's workloads, replayed as
the benchmark replays them (one captured CUDA graph per decode step, `overlap`
launch order unless stated), against the oracle head by head.

Compared after every step:
  * every KV head of the last layer: the selected blocks, the fetch list (the
    decode step's last two layers keep their selection buffers), the block
    tables, the contents of every occupied slot and the attention output;
  * two (request, KV head) pairs of every other layer: tables, slot contents and
    attention output (selection and fetch list are fixed by the tables: the
    fetched blocks are the new mappings and the attended set is the blocks whose
    LRU clock is the step).
The host tier holds fewer layers than the model (layer l reads host buffer
l mod l_host, as the benchmark does); the oracle is given exactly those inputs.
"""
import numpy as np
import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

from gpu_helpers import _check_out

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()


class FullState:
    """A DecodeState filled on the device, with a snapshot of its tables and pools
    so that several launch orders can start from the same state."""

    def __init__(self, w, l_host):
        from sparse_decode_attention_oasis_gb300.engine import DecodeState

        self.w, self.l_host = w, l_host
        self.st = DecodeState(w, device="cuda:0", l_phys=w.L, l_host=l_host)
        self.st.fill_synthetic()
        self.st.warm_host_tier()
        st = self.st
        self.snap = [t.clone() for t in (st.blk2slot, st.slot2blk, st.last_used, st.k_pool, st.v_pool)]

    def reset(self, scoring):
        st, w_ = self.st, self.w
        for t, s in zip((st.blk2slot, st.slot2blk, st.last_used, st.k_pool, st.v_pool), self.snap):
            t.copy_(s)
        # the cross-step order's per-layer selection buffers, made outside any capture
        st._lag_sel = torch.full((st.L_phys, w_.B, w_.Hkv, w_.Kb), -1, dtype=torch.int32, device=st.device)
        st._lag_nsel = torch.zeros((st.L_phys, w_.B, w_.Hkv), dtype=torch.int32, device=st.device)
        st._lag_ready = False
        st.set_scoring(scoring)
        torch.cuda.synchronize()

    def sample(self, per_layer=2, seed=3):
        """Every head of the last layer (of every layer when there are at most two),
        `per_layer` heads of every other layer."""
        w = self.w
        rng = np.random.default_rng(seed)
        full = range(w.L) if w.L <= 2 else [w.L - 1]
        heads = [(l, b, h) for l in full for b in range(w.B) for h in range(w.Hkv)]
        for l in range(w.L - 1 if w.L > 2 else 0):
            for _ in range(per_layer):
                heads.append((l, int(rng.integers(w.B)), int(rng.integers(w.Hkv))))
        return sorted(set(heads))


def _pool_digests(kp_head, vp_head, s2b_head):
    import oracle_pool

    k = kp_head.cpu().view(torch.int16).numpy().view(np.uint16)
    v = vp_head.cpu().view(torch.int16).numpy().view(np.uint16)
    return oracle_pool.slot_digests(k, v, s2b_head)


def run_and_compare(fs, scoring="maxdot", copy="overlap", steps=2):
    from sparse_decode_attention_oasis_gb300.engine import StepGraph

    import oracle_pool

    w, st = fs.w, fs.st
    fs.reset(scoring)
    heads = fs.sample()
    lag = copy == "lag"
    want = oracle_pool.head_histories([(w, l, b, h, fs.l_host, steps, scoring, lag) for (l, b, h) in heads])
    dev = st.device
    qs = [syn.QueryStreamTorch(w, l, dev) for l in range(w.L)]
    out = torch.empty((w.L, w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
    # the layers whose selection buffers survive a decode step: the last two share the
    # two alternating scratch sets; the cross-step order keeps every layer's selection
    kept = {w.L - 1, w.L - 2} - {-1}
    for s in range(steps):
        q_l, qla_l = [], []
        for l in range(w.L):
            q, qla = qs[l].next()
            q_l.append(q)
            qla_l.append(qla)
        g = StepGraph(st, s, [qla_l], [q_l], [out], copy=copy)
        with torch.cuda.stream(g.stream):
            g.replay()
        torch.cuda.synchronize()
        del g
        assert st.error_word() == 0
        lists = {}
        for l in kept:
            sc = st.scratch2 if l % 2 else st.scratch
            lists[l] = ((st._lag_sel[l] if lag else sc.sel).cpu().numpy(),
                        (st._lag_nsel[l] if lag else sc.nsel).cpu().numpy(),
                        sc.fetch.cpu().numpy(), sc.nfetch.cpu().numpy())
        b2s_all, s2b_all, lu_all = st.blk2slot.cpu().numpy(), st.slot2blk.cpu().numpy(), st.last_used.cpu().numpy()
        out_all = out.cpu().numpy().astype(np.float64)
        for (l, b, h), hist in zip(heads, want):
            r = hist[s]
            where = f"step {s} layer {l} request {b} head {h} ({scoring}, {copy})"
            if l in lists:
                sel, nsel, fetch, nfetch = lists[l]
                S, F = r["S"], r["F"]
                assert nsel[b, h] == len(S) and sel[b, h, :len(S)].tolist() == S, where
                assert nfetch[b, h] == len(F) and fetch[b, h, :len(F)].tolist() == F, where
            np.testing.assert_array_equal(b2s_all[l, b, h], r["b2s"], err_msg=where)
            np.testing.assert_array_equal(s2b_all[l, b, h], r["s2b"], err_msg=where)
            np.testing.assert_array_equal(lu_all[l, b, h], r["lu"], err_msg=where)
            assert _pool_digests(st.k_pool[l, b, h], st.v_pool[l, b, h], r["s2b"]) == r["pool"], where
            _check_out(out_all[l, b, h * w.G:(h + 1) * w.G], r["out"], where)
    return heads


@pytest.fixture(scope="module")
def qwen3_8b():
    fs = FullState(syn.qwen3_8b_decode(), l_host=4)
    yield fs
    del fs.st, fs.snap
    torch.cuda.empty_cache()


def test_qwen3_8b_full_size_overlap_order(qwen3_8b):
    """36 layers x batch 32 x ctx 32K, max-dot scoring, the benchmark's order."""
    heads = run_and_compare(qwen3_8b, "maxdot", "overlap")
    assert len(heads) >= 256 + 36


def test_qwen3_8b_full_size_pooled_scoring(qwen3_8b):
    run_and_compare(qwen3_8b, "pooled", "overlap")


def test_qwen3_8b_full_size_cross_step_pipeline(qwen3_8b):
    """copy="lag": attention over the previous step's selection (three steps so
    that two of them attend a lagged selection)."""
    run_and_compare(qwen3_8b, "maxdot", "lag", steps=3)


def test_llama_long_input_full_8192_blocks_whole_batch():
    """Batch 8 x 128K context (8,192 blocks per head), span + sink/recent hot set,
    cap 6, two layers: every head of both layers is compared."""
    w = syn.llama31_8b_long(L=2)
    assert w.nb_max == 8192 and w.B == 8
    fs = FullState(w, l_host=2)
    run_and_compare(fs, "maxdot", "overlap")


def test_qwen3_32b_gqa8_full_batch():
    """GQA 8 (64 query heads, 32 lookahead rows per KV head), batch 16 x 32K, cap
    at fetch ratio 0.05, two layers."""
    w = syn.qwen3_32b(ratio=0.05, L=2)
    assert w.G == 8 and w.B == 16
    fs = FullState(w, l_host=2)
    run_and_compare(fs, "maxdot", "overlap")
