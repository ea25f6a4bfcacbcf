"""Fused look-ahead attention (f2) on the GPU against the oracle: the true-query
rows and every lookahead row within the attention tolerance, over the same
resident selected blocks as a5, for group sizes whose (1 + n_la) G rows fill one,
two or three 16-row tiles."""
import pytest

from sparse_decode_attention_oasis_gb300 import synthetic as syn

from gpu_helpers import Case

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_decode_attention_oasis_gb300 import build

    build.build()


def test_tiny_workload_lookahead_rows():
    w = syn.tiny()
    c = Case(w)
    for step in range(2):
        c.step(step, lookahead=True)


@pytest.mark.parametrize("Hq,n_la", [(8, 4), (16, 3), (64, 4), (64, 1), (32, 7)])
def test_group_sizes_and_row_tiles(Hq, n_la):
    w = syn.Workload("la", L=1, B=2, Hq=Hq, Hkv=8, ctx=[2048, 999], Kb=32, C=6, n_hot=16, n_la=n_la)
    c = Case(w)
    c.step(0, lookahead=True)
    c.step(1, lookahead=True)


def test_ragged_and_empty_attended_set():
    w = syn.Workload("ragged", L=1, B=3, Hq=32, Hkv=8, ctx=[4096, 1000, 17], Kb=32, C=0, n_hot=16)
    import numpy as np

    blank = tuple(np.full_like(t, -1) for t in syn.initial_tables(w, 0))
    c = Case(w, tables=blank)  # nothing resident and a cap of 0: A is empty, outputs are zero
    c.step(0, lookahead=True)
