"""Agreement counters (f3) on the GPU against the oracle: the exact top-K of the
true query, the lookahead prediction and the previous-token prediction, counted
per head through oasis_set_agreement; counts must be identical."""
import numpy as np
import pytest

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn

from gpu_helpers import Case, _dev_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()


def _check(w, c, probe, step, q, qla, q_prev, S):
    got = probe.run(0, _dev_bits(qla), _dev_bits(q), None if q_prev is None else _dev_bits(q_prev))
    torch.cuda.synchronize()
    assert int(probe.err.item()) == 0
    K = probe.K
    exact = ref.exact_topk_true_query(c.K, q, w.ctx, K)

    def predicted(rows):  # top-K under the decode path's scoring, rows [B][n][Hq][d]
        if c.scoring == "pooled":
            pooled = {(b, h): ref.pool_keys(c.K[b, h], w.ctx[b], w.nb_max) for b in range(w.B)
                      for h in range(w.Hkv)}
            sc = ref.block_scores_pooled(pooled, rows, w.ctx, w.d)
        else:
            sc = ref.block_scores(c.K, rows, w.ctx)
        return {bh: ref.topk_select(key, K) for bh, (_, key) in sc.items()}

    la = predicted(qla)
    if K == w.Kb:
        assert la == S  # the probe's lookahead set is the decode step's S
    preds = {"la": la}
    if q_prev is not None:
        preds["prev"] = predicted(q_prev[:, None])
    for which, pred in preds.items():
        counts = got[which].cpu().numpy()
        for (b, h), E in exact.items():
            want = ref.set_agreement(pred[(b, h)], E, c.b2s[b, h])
            assert tuple(counts[b, h].tolist()) == want, (which, b, h)


@pytest.mark.parametrize("K,scoring", [(None, "maxdot"), (20, "maxdot"), (None, "pooled")])
def test_agreement_counts_match_oracle(K, scoring):
    from sparse_decode_attention_oasis_gb300.engine import AgreementProbe

    w = syn.Workload("agree", L=1, B=2, Hq=32, Hkv=8, ctx=[4096, 1500], Kb=32, C=4, n_hot=16)
    c = Case(w, scoring=scoring)
    probe = AgreementProbe(c.st, K=K)
    q_prev = None
    for step in range(3):
        q, qla = syn.layer_queries(w, 0, step)
        r, _ = c.step(step, q=q, qla=qla)
        _check(w, c, probe, step, q, qla, q_prev, r["S"])
        q_prev = q


def test_agreement_without_table_reports_minus_one():
    from sparse_decode_attention_oasis_gb300 import binding as B

    w = syn.tiny()
    s = B.Shape.from_workload(w)
    sel = torch.arange(w.Kb, dtype=torch.int32, device="cuda").repeat(w.B, w.Hkv, 1)
    n = torch.full((w.B, w.Hkv), w.Kb, dtype=torch.int32, device="cuda")
    ex = sel.clone() + 5
    counts = torch.empty((w.B, w.Hkv, 3), dtype=torch.int32, device="cuda")
    B.oasis_set_agreement(s, sel, n, ex, n, None, counts)
    torch.cuda.synchronize()
    assert (counts[..., 0] == w.Kb - 5).all() and (counts[..., 1] == -1).all() and (counts[..., 2] == w.Kb).all()
