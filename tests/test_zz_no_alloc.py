"""The allocation-free attention call, checked against the oracle and the workspace call.

Callers that cannot allocate device memory when they call - a serving loop whose
device-memory budget is fixed at start-up, or host code that must not call
cudaMalloc on its decode path - use oasis_sparse_decode_attn_noalloc, which keeps
its scratch in a device array built into the library.  Its output must match
the oracle's attention over the same selection, and oasis_sparse_decode_attn's,
call after call (the array is shared and reused).
"""
import ctypes

import numpy as np
import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import binding, build

    build.build()
    return binding


def _state(w, step):
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    K, V = syn.layer_kv(w, 0)
    b2s, s2b, lu = syn.initial_tables(w, 0)
    st = DecodeState(w, device="cuda:0", l_phys=1)
    st.fill_layer_numpy(0, K, V, b2s, s2b, lu)
    q, qla = syn.layer_queries(w, 0, step)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    qd = dev(q)
    sc = st.layer_step(0, dev(qla), qd, step)
    torch.cuda.synchronize()
    return st, sc, qd


def _close(a, b):
    err = (a - b).abs()
    return bool(((err <= ATOL) | (err <= RTOL * b.abs())).all())


def test_noalloc_matches_the_workspace_call_on_two_calls_in_a_row(lib):
    for w, step in ((syn.tiny(), 0),
                    (syn.Workload("ragged", L=1, B=3, Hq=64, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=4,
                                  n_hot=16), 1)):
        st, sc, q = _state(w, step)
        s = st.shape
        ref = torch.empty_like(sc.out)
        lib.oasis_sparse_decode_attn(s, q, st.k_pool[0], st.v_pool[0], sc.sel, sc.nsel, st.blk2slot[0],
                                     st.ctx, st.scale, sc.ws, sc.ws_bytes, ref)
        for _ in range(2):
            out = torch.full_like(sc.out, float("nan"))
            lib.oasis_sparse_decode_attn_noalloc(s, q, st.k_pool[0], st.v_pool[0], sc.sel, sc.nsel,
                                                 st.blk2slot[0], st.ctx, st.scale, out)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all()
            assert _close(out, ref)


@pytest.mark.parametrize("w", [
    syn.Workload("ragged", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=4, n_hot=16),
    syn.Workload("gqa8", L=1, B=2, Hq=64, Hkv=8, n_la=4, ctx=[3000, 2048], Kb=24, C=3, n_hot=12),
], ids=["ragged", "gqa8"])
def test_noalloc_matches_the_oracle(lib, w):
    """The oracle's decode step (selection, gather, attention over the attended
    blocks) against the allocation-free call run on the device's selection, which
    the harness has checked index for index against the oracle's."""
    from gpu_helpers import Case, _check_out, _dev_bits

    case = Case(w)
    q, qla = syn.layer_queries(w, 0, 0)
    r, sc = case.step(0, q=q, qla=qla)
    st = case.st
    out = torch.full_like(sc.out, float("nan"))
    lib.oasis_sparse_decode_attn_noalloc(st.shape, _dev_bits(q), st.k_pool[0], st.v_pool[0], sc.sel, sc.nsel,
                                         st.blk2slot[0], st.ctx, st.scale, out)
    torch.cuda.synchronize()
    _check_out(out.cpu().numpy().astype(np.float64), r["out"], f"allocation-free attention ({w.name})")


def test_noalloc_rejects_shapes_beyond_its_array(lib):
    big = lib.Shape.of(B=4096, Hq=64, Hkv=8, nb_max=2048, n_la=4, Kb=256, P=256)
    assert lib.oasis_attn_workspace_bytes(big) > 8 << 20
    dummy = torch.empty(64, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    st = lib.load().oasis_sparse_decode_attn_noalloc(ctypes.byref(big), p, p, p, p, p, p, p, 0.1, p, None)
    assert st == 4
    assert "bytes" in lib.oasis_last_error()


def test_noalloc_rejects_what_the_workspace_call_rejects(lib):
    """n_la * G > 32 is outside the supported range for both attention calls."""
    s = lib.Shape.of(B=2, Hq=64, Hkv=8, nb_max=256, n_la=5, Kb=32, P=32)
    dummy = torch.empty(64, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    raw = lib.load()
    a = raw.oasis_sparse_decode_attn(ctypes.byref(s), p, p, p, p, p, p, p, 0.1, p, 1 << 20, p, None)
    b = raw.oasis_sparse_decode_attn_noalloc(ctypes.byref(s), p, p, p, p, p, p, p, 0.1, p, None)
    assert a == b == 4
    assert "n_la * G" in lib.oasis_last_error()
