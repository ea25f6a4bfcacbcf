"""A copy that waits for a host-written ready flag gives up after a bounded number
of polls: the error word gets OASIS_EW_TIMEOUT, oasis_error_word_status reports
OASIS_ERR_TIMEOUT, nothing is copied, no kernel is left waiting, and the next
calls run normally.  The failure is made on the host (a flag nothing sets);
nothing faults, traps or hangs."""
import threading
import time

import numpy as np
import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import binding, build

    build.build()
    return binding


def _prepared(B):
    """A layer whose fetch lists are mapped to slots (table half done), data not copied."""
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    w = syn.Workload("wait", L=1, B=2, Hq=32, Hkv=8, ctx=[1024, 700], Kb=16, C=3, n_hot=4)
    st = DecodeState(w, l_phys=1)
    K, V = syn.layer_kv(w, 0)
    st.fill_layer_numpy(0, K, V, *[np.array(t) for t in syn.initial_tables(w, 0)])
    q, qla = syn.layer_queries(w, 0, 0)
    from gpu_helpers import _dev_bits

    sc = st.scratch
    main = torch.cuda.current_stream()
    st._select(0, _dev_bits(qla), 0, sc, main)
    st._assign(0, st._step_tensor(0, main), sc, main)
    torch.cuda.synchronize()
    assert int(sc.nfetch.sum().item()) > 0
    return w, st, sc


def _expected_pools(w, st, sc):
    """Pools after a successful copy: each fetched block's host data in its slot."""
    kp, vp = st.k_pool[0].clone(), st.v_pool[0].clone()
    fetch, nfetch, b2s = sc.fetch.cpu().numpy(), sc.nfetch.cpu().numpy(), st.blk2slot[0].cpu().numpy()
    host = st.host[0]
    for b in range(w.B):
        for h in range(w.Hkv):
            for x in fetch[b, h, :nfetch[b, h]]:
                p = b2s[b, h, x]
                kp[b, h, p] = host[b, h, x, 0].cuda()
                vp[b, h, p] = host[b, h, x, 1].cuda()
    return kp, vp


def _copy_wait(B, st, sc, flag, value, polls, err):
    B.oasis_copy_fetched_wait(st.shape, st.host[0], sc.fetch, sc.nfetch, st.blk2slot[0], st.k_pool[0],
                              st.v_pool[0], flag, value, polls, err)


def test_wait_gives_up_then_the_gpu_answers(B):
    w, st, sc = _prepared(B)
    flag = torch.zeros(1, dtype=torch.int32).pin_memory()   # nothing sets it
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp0, vp0 = st.k_pool.clone(), st.v_pool.clone()
    want_k, want_v = _expected_pools(w, st, sc)
    t0 = time.perf_counter()
    _copy_wait(B, st, sc, flag, 1, 4000, err)
    status, bits = B.oasis_error_word_status(err)
    waited = time.perf_counter() - t0
    assert status == 3 and bits == B.EW_TIMEOUT          # OASIS_ERR_TIMEOUT
    assert "gave up" in B.oasis_last_error()
    assert waited < 5.0
    assert torch.equal(st.k_pool, kp0) and torch.equal(st.v_pool, vp0)   # nothing copied
    # the GPU answers normal calls afterwards: the same copy once the flag is set
    flag[0] = 1
    err.zero_()
    _copy_wait(B, st, sc, flag, 1, 4000, err)
    assert B.oasis_error_word_status(err) == (0, 0)
    assert torch.equal(st.k_pool[0], want_k) and torch.equal(st.v_pool[0], want_v)


def test_wait_sees_a_flag_the_host_sets_while_it_polls(B):
    w, st, sc = _prepared(B)
    want_k, want_v = _expected_pools(w, st, sc)
    flag = torch.zeros(1, dtype=torch.int32).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def producer():
        time.sleep(0.02)
        flag[0] = 7

    t = threading.Thread(target=producer)
    t.start()
    _copy_wait(B, st, sc, flag, 7, 1 << 22, err)   # at most about one to two seconds of polls
    status, bits = B.oasis_error_word_status(err)
    t.join()
    assert (status, bits) == (0, 0)
    assert torch.equal(st.k_pool[0], want_k) and torch.equal(st.v_pool[0], want_v)


def test_wait_argument_checks(B):
    w, st, sc = _prepared(B)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pageable = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(B.OasisError):
        _copy_wait(B, st, sc, pageable, 1, 10, err)          # not page-locked mapped memory
    flag = torch.zeros(1, dtype=torch.int32).pin_memory()
    for polls in (0, (1 << 22) + 1):
        with pytest.raises(B.OasisError):
            _copy_wait(B, st, sc, flag, 1, polls, err)
