"""The C ABI library loads and exports every symbol include/*.h declares; host-side argument
checks run without a GPU (no compute call is made)."""
import ctypes
import glob
import os
import re

import pytest

import expert_cached_routed_router_b300 as ftm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(hdr).read(), flags=re.S)
        names |= set(re.findall(r"\b(ft_[a-z_0-9]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = ftm.load_library()
    declared = _declared()
    assert declared, "no declarations found"
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared == set(ftm.EXPORTS)


def test_binding_has_the_c_names():
    for name in ftm.EXPORTS:
        if name != "ft_last_error":
            assert callable(getattr(ftm, name)), name


@pytest.mark.parametrize("args", [
    (0, 16, 2, 256, 128, 16),      # L < 1
    (1, 16, 17, 256, 128, 16),     # k > E
    (1, 2000, 2, 256, 128, 16),    # E > 1024
    (1, 16, 2, 200, 128, 16),      # d not a multiple of 128
    (1, 16, 2, 256, 100, 16),      # d_ff not a multiple of 128
    (1, 16, 2, 256, 128, 0),       # no slots
    (1, 64, 40, 256, 128, 16),     # k > 32
    (1, 16, 2, 8192, 128, 16),     # d > 4096
])
def test_create_rejects_bad_shapes(args):
    with pytest.raises(ftm.FtError) as ei:
        ftm.ft_moe_create(*args)
    assert ei.value.code == ftm.FT_ERR_INVALID


def test_create_rejects_bad_weight_format():
    with pytest.raises(ftm.FtError) as ei:
        ftm.ft_moe_create(1, 16, 2, 256, 128, 16, weight_format=2)
    assert ei.value.code == ftm.FT_ERR_INVALID
    with pytest.raises(ftm.FtError) as ei:
        ftm.ft_moe_create(1, 16, 2, 256, 128, 16, n_shared=1, weight_format=1)
    assert ei.value.code == ftm.FT_ERR_INVALID


def test_null_handle_is_rejected():
    lib = ftm.load_library()
    assert lib.ft_moe_forward(None, 0, None, 1, None, None) == ftm.FT_ERR_INVALID
    assert b"null handle" in lib.ft_last_error()
    assert lib.ft_cache_resize(None, 4) == ftm.FT_ERR_INVALID
    s = ftm.ft_cache_stats_t()
    assert lib.ft_cache_stats(None, ctypes.byref(s)) == ftm.FT_ERR_INVALID
    lib.ft_moe_destroy(None)   # ignored


def test_options_struct_layout_matches_header():
    hdr = open(os.path.join(ROOT, "include", "ft_moe.h")).read()
    body = re.search(r"typedef struct \{(.*?)\} ft_moe_opts;", hdr, re.S).group(1)
    names = re.findall(r"^\s*int (\w+);", body, re.M)
    assert [f for f, _ in ftm.ft_moe_opts._fields_] == names
    assert ctypes.sizeof(ftm.ft_moe_opts) == 4 * len(names)
    body = re.search(r"typedef struct \{(.*?)\} ft_cache_stats_t;", hdr, re.S).group(1)
    fields = re.findall(r"^\s*(uint64_t|int32_t) (\w+);", body, re.M)
    assert [f for f, _ in ftm.ft_cache_stats_t._fields_] == [n for _, n in fields]
    assert ctypes.sizeof(ftm.ft_cache_stats_t) == sum(8 if t == "uint64_t" else 4
                                                     for t, _ in fields)
