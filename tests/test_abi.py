"""The C-ABI library builds, loads without a GPU and exports every declared call."""
import ctypes
import os
import re

import pytest

from sparse_decode_attention_oasis_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "oasis.h")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"OASIS_API\s+[\w\s\*]+?\b(oasis_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("oasis_score_blocks", "oasis_topk_select", "oasis_fetch_diff_capped",
              "oasis_gather_h2d", "oasis_sparse_decode_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(binding.LIB_PATH)
    for n in declared_functions():
        assert hasattr(raw, n), n
    assert binding.oasis_version().startswith("oasis-gb300")


def test_binding_exposes_the_same_names():
    for n in declared_functions():
        assert hasattr(binding, n), n


def _shape(**kw):
    base = dict(B=2, Hq=32, Hkv=8, nb_max=256, n_la=4, Kb=32, P=32)
    base.update(kw)
    return binding.Shape.of(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=30), 1), (dict(d=64), 4), (dict(bs=32), 4), (dict(Kb=300, P=300), 4),
    (dict(P=16), 4), (dict(nb_max=9000), 4), (dict(n_la=9), 4), (dict(Hq=24, Hkv=8), 4),
])
def test_shape_validation_rejects_before_launch(lib, kw, status):
    s = _shape(**kw)
    st = lib.oasis_score_blocks(ctypes.byref(s), 16, 16, 16, 16, None, None)
    assert st == status
    assert lib.oasis_last_error()


def test_null_and_misaligned_pointers_are_invalid(lib):
    s = _shape()
    assert lib.oasis_score_blocks(ctypes.byref(s), None, 16, 16, 16, None, None) == 1
    assert lib.oasis_score_blocks(ctypes.byref(s), 18, 16, 16, 16, None, None) == 1
    assert lib.oasis_score_blocks(ctypes.byref(s), 16, 16, 16, 16, 18, None) == 1
    assert lib.oasis_fetch_diff_capped(ctypes.byref(s), 16, 16, 16, 16, 16, 16, 16, 33, 16, 16, None) == 1
    assert lib.oasis_sparse_decode_attn(ctypes.byref(s), 16, 16, 16, 16, 16, 16, 16, 0.1, 16, 0, 16, None) == 1
    with pytest.raises(binding.OasisError):
        binding.oasis_score_blocks(s, None, 16, 16, 16, None, stream=0)


def test_workspace_size_formula(lib):
    s = _shape()
    # splits x (2 requests * 8 KV heads * 4 query heads) rows of (128 + 2) floats;
    # the split count (1 .. Kb/4) follows the device's SM count
    row = 2 * 8 * 4 * 130 * 4
    ws = binding.oasis_attn_workspace_bytes(s)
    assert ws % row == 0 and 1 <= ws // row <= 32 // 4
    assert binding.oasis_attn_workspace_bytes(_shape(d=64)) == 0


def test_new_calls_validate_before_launch(lib):
    s = _shape()
    # fetch cap beyond Kb, misaligned pointers, NULL outputs: rejected without a launch
    assert lib.oasis_topk_select_diff(ctypes.byref(s), 16, 16, 16, 16, 16, 33, 16, 16, 16, 16, None, None) == 1
    assert lib.oasis_topk_select_diff_pooled(ctypes.byref(s), 16, 18, 16, 16, 16, 2, 16, 16, 16, 16, None,
                                             None) == 1
    assert lib.oasis_topk_select_diff(ctypes.byref(s), 16, 16, 16, 16, 16, 2, 16, 16, 16, 16, 24, None) == 1
    assert lib.oasis_copy_fetched(ctypes.byref(s), 16, 16, 16, 16, 16, 16, None, None) == 1
    assert lib.oasis_assign_slots(ctypes.byref(s), 16, 16, 16, 16, 16, 16, 16, 18, 16, None) == 1
    assert lib.oasis_score_blocks_pooled(ctypes.byref(s), 16, 16, 16, 12, None, None, None, None, None, None,
                                         None, None) == 1
    assert lib.oasis_sparse_decode_attn_lookahead(ctypes.byref(s), 16, 16, 16, 16, 16, 16, 16, 16, 0.1, 16, 0,
                                                  16, 16, None) == 1
    assert lib.oasis_set_agreement(ctypes.byref(s), 16, 16, 16, 16, None, None, None, None) == 1
    assert lib.oasis_touch_host(None, 16, None, None) == 1
    assert lib.oasis_touch_host(16, 15, None, None) == 1


def test_lookahead_workspace_size_formula(lib):
    s = _shape()
    # splits x row tiles of 16 rows of (128 + 2) floats; (1 + n_la) G = 20 rows -> 2 tiles
    tile = 2 * 8 * 2 * 16 * 130 * 4
    ws = binding.oasis_attn_lookahead_workspace_bytes(s)
    assert ws % tile == 0 and 1 <= ws // tile <= 32 // 4


def test_set_option_validates(lib):
    assert lib.oasis_set_option(1, -1) == 1
    assert lib.oasis_set_option(99, 0) == 1
    assert lib.oasis_set_option(1, 0) == 0
    assert lib.oasis_set_option(2, 2) == 1        # OASIS_OPT_SCORE_KERNEL: only MMA (0) or TC (1)
    assert lib.oasis_set_option(2, 1) == 0
    assert lib.oasis_set_option(2, 0) == 0


def _header_signatures():
    """{name: (return type, [parameter types])} from the declarations in oasis.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    sigs = {}
    for ret, name, params in re.findall(r"OASIS_API\s+([\w\s\*]+?)\b(oasis_\w+)\s*\(([^;]*?)\)\s*;", text, flags=re.S):
        ps = [] if params.strip() in ("", "void") else [p.strip() for p in params.split(",")]
        types = [re.sub(r"\s+", " ", p if p.endswith("*") else re.sub(r"\b\w+$", "", p)).strip() for p in ps]
        sigs[name] = (re.sub(r"\s+", " ", ret).strip(), types)
    return sigs


def _ctypes_kind(t):
    if t is ctypes.c_void_p or t is ctypes.c_char_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "pointer"
    return {ctypes.c_int32: "int32", ctypes.c_int: "int32", ctypes.c_uint32: "int32", ctypes.c_size_t: "size",
            ctypes.c_float: "float"}[t]


def _c_kind(t):
    if t.endswith("*") or t == "oasis_stream_t":
        return "pointer"
    return {"int32_t": "int32", "oasis_status": "int32", "size_t": "size", "float": "float",
            "uint32_t": "int32"}[t]


def test_binding_signatures_match_the_header():
    """Every call's ctypes argument list has the header's arity and argument kinds
    (pointer, 32-bit integer, size, float), and the same kind of return value: a
    mismatch would pass every CPU test and corrupt arguments on the GPU."""
    sigs = _header_signatures()
    assert len(sigs) == len(declared_functions())
    for name, (ret, params) in sigs.items():
        argtypes, restype = binding._SIGS[name]
        assert len(argtypes) == len(params), (name, params)
        assert [_ctypes_kind(a) for a in argtypes] == [_c_kind(p) for p in params], name
        assert _ctypes_kind(restype) == _c_kind(ret), (name, ret)


@pytest.mark.parametrize("kw,ptr,status", [
    (dict(Hq=64, Hkv=8, n_la=5), 16, 4),   # n_la * G = 40 > 32
    (dict(Hq=30), 16, 1), (dict(d=64), 16, 4), (dict(nb_max=9000), 16, 4),
    ({}, 8, 1),                            # a q pointer that is not 16-byte aligned
])
def test_noalloc_attention_validates_like_the_workspace_call(lib, kw, ptr, status):
    """Both attention entry points share their shape and argument checks: the same
    status and message (after the function name) for every rejected call; nothing
    is launched, so no GPU is needed."""
    s = _shape(**kw)
    a = lib.oasis_sparse_decode_attn(ctypes.byref(s), ptr, 16, 16, 16, 16, 16, 16, 0.1, 16, 1 << 30, 16, None)
    ea = lib.oasis_last_error().decode()
    b = lib.oasis_sparse_decode_attn_noalloc(ctypes.byref(s), ptr, 16, 16, 16, 16, 16, 16, 0.1, 16, None)
    eb = lib.oasis_last_error().decode()
    assert a == b == status
    assert ea.startswith("oasis_sparse_decode_attn: ") and eb.startswith("oasis_sparse_decode_attn_noalloc: ")
    assert ea.split(": ", 1)[1] == eb.split(": ", 1)[1]
