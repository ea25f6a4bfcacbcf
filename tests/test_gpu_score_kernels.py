"""The two scoring kernels: the mma.sync one (the alternative to the default TMA +
tcgen05 kernel) checked like the default (bound, selection, full step), and the
two against each other."""
import numpy as np
import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

from gpu_helpers import Case

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _use(kernel):
    from sparse_decode_attention_oasis_gb300 import binding as B

    B.oasis_set_option(B.OPT_SCORE_KERNEL, B.SCORE_KERNEL_TC if kernel == "tc" else B.SCORE_KERNEL_MMA)


@pytest.fixture(autouse=True)
def _mma_kernel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()
    _use("mma")
    yield
    _use("tc")  # the process-wide default for the tests that follow


def test_mma_tiny_workload_two_steps():
    c = Case(syn.tiny())
    c.step(0)
    c.step(1)


@pytest.mark.parametrize("Hq,n_la,ctx", [(32, 4, [4096, 1000, 17]), (64, 4, [2048, 1531]),
                                        (16, 3, [1024, 700]), (8, 4, [3000, 129])])
def test_mma_shapes(Hq, n_la, ctx):
    w = syn.Workload("mma", L=1, B=len(ctx), Hq=Hq, Hkv=8, ctx=ctx, Kb=32, C=5, n_hot=16, n_la=n_la)
    c = Case(w)
    c.step(0)


def test_tc_matches_the_mma_kernel_within_bounds():
    _use("tc")
    w = syn.Workload("cmp", L=1, B=2, Hq=32, Hkv=8, ctx=[4096, 2500], Kb=32, C=4, n_hot=16)
    c = Case(w)
    r, sc = c.step(0)
    tc_scores = sc.scores.cpu().numpy().copy()
    _use("mma")
    c2 = Case(w)
    r2, sc2 = c2.step(0)
    mma_scores = sc2.scores.cpu().numpy()
    for b in range(w.B):
        nb = w.nb(b)
        a, e = tc_scores[b, :, :nb, 0], tc_scores[b, :, :nb, 1]
        m, e2 = mma_scores[b, :, :nb, 0], mma_scores[b, :, :nb, 1]
        assert (np.abs(a - m) <= e + e2).all()
        np.testing.assert_allclose(e, e2, rtol=1e-5)
