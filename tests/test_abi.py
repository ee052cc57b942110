"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching CUDA (runs without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

import post_weight_quantization_column_b300 as awq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(awq_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(awq.LIB_PATH):
        from post_weight_quantization_column_b300 import build
        build.build()
    return awq.lib()


def test_header_declares_the_three_calls():
    names = declared_symbols()
    for n in ("awq_act_stats", "awq_search", "awq_quantize_pack"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_symbols():
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in awq.AWQ_STATUS.items():
        assert L.awq_status_string(code).decode().startswith(name)


def _cfg(**kw):
    return awq.make_cfg(**kw)


def test_workspace_queries_are_host_only(L):
    n = ctypes.c_size_t(0)
    cfg = _cfg()
    assert L.awq_search_workspace_size(4096, 4096, 4096, 21, ctypes.byref(cfg), ctypes.byref(n)) == 0
    assert n.value > 21 * 4096 * 4
    assert L.awq_act_stats_workspace_size(16384, 8192, ctypes.byref(n)) == 0 and n.value >= 256
    assert L.awq_pack_workspace_size(256, 256, ctypes.byref(cfg), ctypes.byref(n)) == 0 and n.value >= 4


@pytest.mark.parametrize("kw,code", [
    (dict(N=64, D_in=250, D_out=256), 2),     # D_in not a multiple of the group
    (dict(N=64, D_in=256, D_out=250), 2),     # D_out not a multiple of 8
    (dict(N=0, D_in=256, D_out=256), 2),      # no calibration rows
    (dict(N=64, D_in=256, D_out=256, G=0), 2),
    (dict(N=64, D_in=256, D_out=256, G=65), 2),
])
def test_search_shape_errors(L, kw, code):
    n = ctypes.c_size_t(0)
    cfg = _cfg()
    G = kw.pop("G", 21)
    assert L.awq_search_workspace_size(kw["N"], kw["D_in"], kw["D_out"], G, ctypes.byref(cfg), ctypes.byref(n)) == code


@pytest.mark.parametrize("field,value", [("bits", 3), ("group_size", 100), ("symmetric", 2), ("act_floor", -1.0)])
def test_bad_cfg_is_invalid_arg(L, field, value):
    cfg = _cfg()
    setattr(cfg, field, value)
    n = ctypes.c_size_t(0)
    assert L.awq_search_workspace_size(64, 256, 256, 21, ctypes.byref(cfg), ctypes.byref(n)) == 1


def test_calls_validate_before_cuda(L):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first
    grid = (ctypes.c_double * 21)(*awq.default_grid())
    # null pointers
    assert L.awq_search(None, fake, 64, 256, 256, fake, grid, 21, ctypes.byref(cfg), fake, fake, fake, None,
                        fake, 1 << 20, None) == 1
    # grid value outside [0, 1]
    bad = (ctypes.c_double * 21)(*([2.0] + awq.default_grid()[1:]))
    assert L.awq_search(fake, fake, 64, 256, 256, fake, bad, 21, ctypes.byref(cfg), fake, fake, fake, None,
                        fake, 1 << 40, None) == 1
    # misaligned X
    assert L.awq_search(ctypes.c_void_p(0x1002), fake, 64, 256, 256, fake, grid, 21, ctypes.byref(cfg), fake,
                        fake, fake, None, fake, 1 << 40, None) == 3
    # workspace too small
    assert L.awq_search(fake, fake, 64, 256, 256, fake, grid, 21, ctypes.byref(cfg), fake, fake, fake, None,
                        fake, 16, None) == 4
    # act_stats: no rows, ragged channel count, short leading dimension
    assert L.awq_act_stats(fake, 0, 256, 256, fake, fake, 1 << 20, None) == 2
    assert L.awq_act_stats(fake, 8, 250, 250, fake, fake, 1 << 20, None) == 2
    assert L.awq_act_stats(fake, 8, 256, 128, fake, fake, 1 << 20, None) == 2
    # an empty channel set is a no-op
    assert L.awq_act_stats(fake, 8, 0, 0, fake, fake, 0, None) == 0
    # pack: group does not divide D_in; misaligned qweight
    assert L.awq_quantize_pack(fake, fake, 200, 256, ctypes.byref(cfg), fake, fake, fake, fake, 256, None) == 2
    assert L.awq_quantize_pack(fake, fake, 256, 256, ctypes.byref(cfg), ctypes.c_void_p(0x1001), fake, fake, fake,
                               256, None) == 3
    # s needs 4-byte alignment: at +2 it is refused
    assert L.awq_quantize_pack(fake, ctypes.c_void_p(0x1002), 256, 256, ctypes.byref(cfg), fake, fake, fake, fake,
                               256, None) == 3
    # pack after a search: grid size out of range, group does not divide D_in,
    # misaligned s_star, workspace without the parameter table; empty is a no-op
    ps = L.awq_quantize_pack_searched
    assert ps(fake, 256, 256, 0, ctypes.byref(cfg), fake, 1 << 40, fake, fake, fake, fake, fake, None) == 2
    assert ps(fake, 200, 256, 21, ctypes.byref(cfg), fake, 1 << 40, fake, fake, fake, fake, fake, None) == 2
    assert ps(fake, 256, 252, 21, ctypes.byref(cfg), fake, 1 << 40, fake, fake, fake, fake, fake, None) == 2
    assert ps(fake, 256, 256, 21, ctypes.byref(cfg), fake, 1 << 40, fake, ctypes.c_void_p(0x1004), fake, fake, fake,
              None) == 3
    assert ps(fake, 256, 256, 21, ctypes.byref(cfg), fake, 4096, fake, fake, fake, fake, fake, None) == 4
    assert ps(fake, 0, 256, 21, ctypes.byref(cfg), fake, 0, fake, fake, fake, fake, fake, None) == 0
    # streaming statistic: no running sum; finalize over no rows
    assert L.awq_act_stats_accumulate(fake, 8, 256, 256, None, None, fake, 1 << 20, None) == 1
    assert L.awq_act_stats_accumulate(fake, 8, 256, 256, ctypes.c_void_p(0x1004), None, fake, 1 << 20, None) == 3
    assert L.awq_act_stats_finalize(fake, 0, 256, fake, None) == 2
    # Gram-form search: fewer rows than channels
    n = ctypes.c_size_t(0)
    assert L.awq_search_gram_workspace_size(128, 256, 256, 21, ctypes.byref(cfg), ctypes.byref(n)) == 2
    assert L.awq_search_gram_workspace_size(512, 256, 256, 21, ctypes.byref(cfg), ctypes.byref(n)) == 0 and n.value > 0
    # closed-form scale: alpha outside [0, 1], ragged D_out
    assert L.awq_closed_form_scales(fake, 256, 256, fake, 1.5, ctypes.byref(cfg), fake, None) == 1
    assert L.awq_closed_form_scales(fake, 256, 252, fake, 0.5, ctypes.byref(cfg), fake, None) == 2
    # greedy search: 1 not among the candidates, too many candidates, no passes, ragged D_out
    gs = L.awq_greedy_search
    assert gs(fake, fake, 256, 256, ctypes.byref(cfg), 3, 1, 20, fake, None, None, fake, 1 << 30, None) == 1
    assert gs(fake, fake, 256, 256, ctypes.byref(cfg), 3, -10, 25, fake, None, None, fake, 1 << 30, None) == 1
    assert gs(fake, fake, 256, 256, ctypes.byref(cfg), 0, -10, 20, fake, None, None, fake, 1 << 30, None) == 1
    assert gs(fake, fake, 256, 260, ctypes.byref(cfg), 3, -10, 20, fake, None, None, fake, 1 << 30, None) == 2
    assert gs(fake, fake, 256, 256, ctypes.byref(cfg), 3, -10, 20, fake, None, None, fake, 256, None) == 4
    # W4A16 product: D_in not a multiple of 64, D_out not a multiple of 16,
    # misaligned Y, workspace too small; no rows is a no-op
    mm = L.awq_w4a16_matmul
    assert mm(fake, 8, 96, 256, fake, fake, fake, None, ctypes.byref(cfg), fake, fake, 256, None) == 2
    assert mm(fake, 8, 256, 264, fake, fake, fake, None, ctypes.byref(cfg), fake, fake, 256, None) == 2
    assert mm(fake, 8, 256, 256, fake, fake, fake, None, ctypes.byref(cfg), ctypes.c_void_p(0x1008), fake, 256,
              None) == 3
    assert mm(fake, 8, 256, 256, fake, fake, fake, None, ctypes.byref(cfg), fake, fake, 16, None) == 4
    assert mm(fake, 0, 256, 256, fake, fake, fake, None, ctypes.byref(cfg), fake, fake, 256, None) == 0
    # self-test GEMM: K not a multiple of 64
    assert L.awq_selftest_gemm_bf16(fake, fake, 1, 128, 256, 100, fake, fake, 256, None) == 2


def test_wait_timeout_selftest_validates_on_host(L):
    f = L.awq_selftest_wait_timeout
    f.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    fake = ctypes.c_void_p(0x100000)
    assert f(999, 1, fake, fake, 8192, None) == 1                  # limit below 1 us
    assert f(2_000_000_001, 1, fake, fake, 8192, None) == 1        # limit above the product's 2 s
    assert f(1_000_000, 0, fake, fake, 8192, None) == 2            # no pair
    assert f(1_000_000, 1, fake, ctypes.c_void_p(0x100010), 8192, None) == 3  # ws not 256-byte aligned
    assert f(1_000_000, 1, fake, fake, 4096, None) == 4            # no room for the 4 KB copy source
    assert f(1_000_000, 1, None, fake, 8192, None) == 1
