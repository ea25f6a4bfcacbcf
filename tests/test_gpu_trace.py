"""The kernel span trace (oasis_trace_set): a traced decode step computes exactly
what an untraced one does, and records one span per launch, in stream order."""
import numpy as np
import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()


def _run(st, snap, w, steps, trace=None):
    from sparse_decode_attention_oasis_gb300.engine import StepGraph

    for t, v in zip((st.blk2slot, st.slot2blk, st.last_used, st.k_pool, st.v_pool), snap):
        t.copy_(v)
    torch.cuda.synchronize()
    dev = st.device
    qs = [syn.QueryStreamTorch(w, l, dev) for l in range(w.L)]
    q_steps, qla_steps = [], []
    for _ in range(steps):
        q_l, qla_l = zip(*(qs[l].next() for l in range(w.L)))
        q_steps.append(list(q_l))
        qla_steps.append(list(qla_l))
    outs = [torch.zeros((w.L, w.B, w.Hq, w.d), dtype=torch.float32, device=dev) for _ in range(steps)]
    if trace is not None:
        trace.start()
    try:
        g = StepGraph(st, 0, qla_steps, q_steps, outs, copy="overlap")
    finally:
        if trace is not None:
            trace.stop()
    with torch.cuda.stream(g.stream):
        g.replay()
    torch.cuda.synchronize()
    assert st.error_word() == 0
    return [o.cpu() for o in outs], [t.cpu() for t in (st.blk2slot, st.slot2blk, st.last_used)]


def test_traced_step_is_identical_and_records_every_launch():
    from sparse_decode_attention_oasis_gb300.engine import DecodeState, KernelTrace

    w = syn.qwen3_8b_decode(B=2, L=3, ctx=4096)
    st = DecodeState(w, device="cuda:0", l_phys=w.L, l_host=w.L)
    st.fill_synthetic()
    st.warm_host_tier()
    snap = [t.clone() for t in (st.blk2slot, st.slot2blk, st.last_used, st.k_pool, st.v_pool)]
    steps = 2
    out_a, tab_a = _run(st, snap, w, steps)
    tr = KernelTrace(capacity=64)
    out_b, tab_b = _run(st, snap, w, steps, trace=tr)
    for a, b in zip(out_a + tab_a, out_b + tab_b):
        assert torch.equal(a, b)
    sp = tr.spans()
    n = w.L * steps
    for kind in ("score", "select", "gather", "attn"):
        a, b = sp[kind]
        assert len(a) == n, kind
        d = b - a
        assert (d > 0).all() and (d < 10**9).all(), kind
    assert len(sp["score_pooled"][0]) == 0 and len(sp["copy"][0]) == 0
    S0, S1 = sp["score"]
    T0, T1 = sp["select"]
    G0, G1 = sp["gather"]
    A0, A1 = sp["attn"]
    # stream order: scorer, then selection (main); the gather (side stream) after the
    # selection; the next scorer after the gather
    assert (T0 >= S1).all() and (G0 >= T1).all()
    assert (S0[1:] >= G1[:-1]).all()
    # attention of layer l: after its own gather; attention of the last layer after all
    assert (A0 >= G1).all()
    # launches made after the trace was stopped do not record
    before = tr.buf.clone()
    _run(st, snap, w, 1)
    assert torch.equal(before, tr.buf)
