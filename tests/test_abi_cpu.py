"""CPU-only checks of the C-ABI library: it builds, loads, exports every symbol
that include/talker.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from kv_cached_qwen3_gb300 import build, talker
    build.build()
    return talker.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(talker_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("talker_create", "talker_destroy", "talker_prefill", "talker_decode", "talker_kv_rewind",
                 "talker_kv_init_batched", "talker_cur_len", "talker_kv_import", "talker_kv_export"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def declared_arity():
    """Function name -> number of parameters, from the prototypes in include/*.h."""
    arity = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            for name, params in re.findall(r"\b(talker_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
                params = params.strip()
                arity[name] = 0 if params in ("", "void") else params.count(",") + 1
    return arity


def test_binding_signatures_match_header(lib):
    """Every prototype the ctypes binding sets has as many arguments as the header declares."""
    arity = declared_arity()
    checked = 0
    for name in declared_functions():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert name in arity, name
        assert len(fn.argtypes) == arity[name], (name, len(fn.argtypes), arity[name])
        checked += 1
    assert checked >= 20


def test_status_strings(lib):
    assert lib.talker_status_str(0) == b"ok"
    assert lib.talker_status_str(2) == b"KV cache overflow"
    assert lib.talker_kernel_launches(None) == 0


def test_create_rejects_bad_geometry_without_gpu(lib):
    from kv_cached_qwen3_gb300 import inputs, talker
    h = ctypes.c_void_p()
    # null config / null out pointer
    assert lib.talker_create(None, None, None, ctypes.byref(h)) == 1
    assert lib.talker_create(None, None, None, None) == 1
    bad = [
        dict(head_dim=96),                  # unsupported head_dim
        dict(n_q_heads=6, n_kv_heads=4),    # not a multiple
        dict(n_q_heads=32, n_kv_heads=2),   # group > 8
        dict(hidden=100),                   # not a multiple of 64
        dict(vocab=3),                      # not a multiple of 8
        dict(intermediate=0),
    ]
    for change in bad:
        g = inputs.Geometry(**{**inputs.TINY.__dict__, **change})
        cfg = talker.make_config(g)
        assert lib.talker_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == 1, change
        assert not h.value
    # a valid geometry with no weights is still rejected before any device work
    cfg = talker.make_config(inputs.TALKER)
    assert lib.talker_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == 1


def test_calls_on_null_handle_are_rejected(lib):
    out = ctypes.c_int()
    assert lib.talker_kv_init_batched(None, 1, 16) == 1
    assert lib.talker_kv_rewind(None, 0, 0) == 1
    assert lib.talker_cur_len(None, 0, ctypes.byref(out)) == 1
    assert lib.talker_prefill(None, 0, None, 1, None, None, None) == 1
    assert lib.talker_decode(None, None, 1, None, None, None) == 1
    assert lib.talker_sync_status(None, None) == 1
    lib.talker_destroy(None)


def test_later_entry_points_reject_null_handles_and_off_grid_shapes(lib):
    """Every entry point added for chunked / batched prefill, the TTS loop and the test
    GEMMs validates its arguments on the host first (EINVAL = 1, no device work)."""
    vp = ctypes.c_void_p
    assert lib.talker_prefill_append(None, 0, None, 1, None, None, None) == 1
    assert lib.talker_prefill_batched(None, 1, None, 1, None, None, None) == 1
    assert lib.talker_prefill_all_rows(None, 0, None, 1, None, None) == 1
    assert lib.talker_set_logit_suppression(None, 0, 0) == 1
    assert lib.talker_set_code_tables(None, None, None, 0, 0) == 1
    assert lib.talker_decode_codes(None, None, None, 1, None, None, None) == 1
    assert lib.talker_frame(None, None, 2, 1, None, None, None, None) == 1
    assert lib.talker_kv_import(None, 0, None, None, 0) == 1
    assert lib.talker_kv_export(None, 0, None, None, 0) == 1
    for mode in (0, 2, 3, 4, 1, 5, -1):
        assert lib.talker_set_prefill_mode(None, mode) == 1
    assert lib.talker_set_decode_mode(None, 0) == 1
    # test GEMMs: null operands, or shapes off the tile grid (N % 128, K % 64)
    buf = vp(1 << 20)   # never dereferenced: the shape check fails first
    assert lib.talker_test_gemm_bf16(None, 1, 64, None, 128, None, 0, 1, None) == 1
    assert lib.talker_test_gemm_bf16(buf, 1, 64, buf, 96, buf, 0, 1, None) == 1
    assert lib.talker_test_gemm_bf16(buf, 1, 48, buf, 128, buf, 0, 1, None) == 1
    assert lib.talker_test_gemm_bf16(buf, 1, 64, buf, 128, buf, 0, 0, None) == 1
    assert lib.talker_test_gemm_swiglu_bf16(None, 1, 64, None, 128, None, None) == 1
    assert lib.talker_test_gemm_swiglu_bf16(buf, 1, 64, buf, 192, buf, None) == 1
    assert lib.talker_head_argmax_noalloc(None, 1, 64, None, 256, 1, None, None, None) == 1
