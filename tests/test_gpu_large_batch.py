"""More requests than the scorers' per-CTA prefix holds (512): both scorers then
give every KV head nb_max positions of their work sequence and skip the ones
past its context.  600 short ragged requests (some empty, some a single token,
block boundaries) against the oracle: certified scores, selection, fetch list,
tables, slot contents and attention output of every head."""
import numpy as np
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


def _workload():
    rng = np.random.default_rng(5)
    ctx = [int(x) for x in rng.integers(0, 600, size=600)]
    ctx[0], ctx[1], ctx[2], ctx[3], ctx[599] = 0, 1, 16, 17, 599
    w = syn.Workload("b600", L=1, B=600, Hq=8, Hkv=2, ctx=ctx, Kb=8, C=2, n_hot=4)
    assert w.B > 512 and w.nb_max > w.Kb
    return w


@pytest.mark.parametrize("scoring", ["maxdot", "pooled"])
def test_more_requests_than_the_prefix_holds(scoring):
    c = Case(_workload(), scoring=scoring)
    if scoring == "pooled":
        c.compare_pooled()
    c.step(0)
    c.step(1)
