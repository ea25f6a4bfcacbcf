"""Parity on the shapes of the other workloads: long input (128K context, span and
sink/recent hot blocks), GQA 8 with the fetch-ratio sweep, long output (growing
context with token appends, the drifting hot set).  Whole full-size decode steps
are in test_gpu_fullsize.py."""
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


@pytest.mark.parametrize("scoring", ["maxdot", "pooled"])
def test_llama_long_input_shape_128k_context(scoring):
    """8,192 blocks per head over few heads: the selection runs 16 warps per head."""
    w = syn.llama31_8b_long(B=1, L=1)
    assert w.nb_max == 8192 and w.C == 6
    c = Case(w, scoring=scoring)
    c.step(0)
    c.step(1)


@pytest.mark.parametrize("ratio", [0.01, 0.02, 0.05, 0.10, 0.20, None])
def test_qwen3_32b_shape_fetch_ratio_sweep(ratio):
    w = syn.qwen3_32b(ratio=ratio, B=1, L=1, ctx=32768)
    c = Case(w)
    for step in range(2):
        c.step(step)


def test_long_output_growing_context_with_appends():
    ctx = [1000, 1531, 2047, 2048]
    w = syn.Workload("long_output", L=1, B=4, Hq=32, Hkv=8, ctx=list(ctx), Kb=32, C=2, n_hot=16,
                     nb_max=-(-(max(ctx) + 40) // 16))
    c = Case(w)
    for step in range(6):
        c.step(step, append=True)
    c.compare_caches()
    assert w.ctx == [x + 6 for x in ctx]


@pytest.mark.parametrize("scoring", ["maxdot", "pooled"])
def test_long_output_drifting_hot_set_batch2_ctx_8k_to_32k_with_appends(scoring):
    """The long-output workload itself: contexts 8,192 and 32,512 tokens (nb_max
    2,048), budget 128 blocks, cap 2, the hot set drifting through 256 planted
    blocks per head, one token appended per request every step, eight steps,
    everything compared with the oracle after every step."""
    w = syn.long_output(B=2, L=1)
    assert w.ctx == [8192, 32512] and w.hot_mode == "drift" and w.C == 2 and w.Kb == 128
    c = Case(w, scoring=scoring)
    fetched = 0
    for step in range(8):
        r, sc = c.step(step, append=True)
        fetched += sum(len(f) for f in r["F"].values())
    c.compare_caches()
    if scoring == "pooled":
        c.compare_pooled()
    assert w.ctx == [8200, 32520]
    assert fetched > 0
    moved = sum(len(set(syn.hot_set(w, 0, b, h, 7)) - set(syn.hot_set(w, 0, b, h, 0)))
                for b in range(w.B) for h in range(w.Hkv))
    assert moved > 0
