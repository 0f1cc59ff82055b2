"""CPU-side checks of the C ABI library: it builds for sm_103a, loads without
a GPU, exports every function include/ice.h declares, and its host-only
entry points behave; the product package and the oracle share no code."""
import ctypes
import os
import re

import pytest

import semantic_paged_kv_gb300 as ice
from semantic_paged_kv_gb300 import build as icebuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    icebuild.build()
    return ice.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ice.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(ice_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(ice.exported_symbols()) == names


def test_host_only_entry_points(lib):
    assert "sm_103a" in ice.ice_version()
    assert ice.ice_status_string(ice.ICE_ERR_CAPACITY) == "capacity exceeded"
    assert ice.ice_page_bound(1000, 1, 16) == 63
    assert ice.ice_page_bound(1000, 100, 16) == (1000 + 15 * 100) // 16
    # sink / window pages: ceil(sink / 16) + ceil(window / 16), the window cut at the sink
    pp = lib.ice_positional_pages
    assert pp(900, 40, 70, 16) == 3 + 5 and pp(900, 0, 0, 16) == 0 and pp(900, 900, 10, 16) == 57
    assert pp(900, 500, 500, 16) == 32 + 25 and pp(10, 3, 4, 16) == 2 and pp(0, 5, 5, 16) == 0
    assert pp(-1, 0, 0, 16) == -1 and pp(100, 0, 0, 8) == -1
    cfg = ice.Config(batch=2, n_q_heads=8, n_kv_heads=2, n_tokens=5000)
    assert ice.ice_build_workspace_bytes(cfg.params()) > 2 * 2 * 5000 * 8
    assert ice.ice_decode_workspace_bytes(cfg.params(), 256, 64) > 0


@pytest.mark.parametrize("fields,status", [({"head_dim": 64}, ice.ICE_ERR_UNSUPPORTED),
                                           ({"page_size": 8}, ice.ICE_ERR_UNSUPPORTED),
                                           ({"n_levels": 4}, ice.ICE_ERR_UNSUPPORTED),
                                           ({"n_levels": 1}, ice.ICE_ERR_UNSUPPORTED),
                                           ({"n_levels": 3, "np_cap": 50001}, ice.ICE_ERR_UNSUPPORTED),
                                           ({"n_q_heads": 48}, ice.ICE_ERR_UNSUPPORTED),
                                           ({"n_kv_heads": 3}, ice.ICE_ERR_INVALID_ARG),
                                           ({"batch": 4096}, ice.ICE_ERR_INVALID_ARG),
                                           ({"batch": 0}, ice.ICE_ERR_INVALID_ARG),
                                           ({"dtype": 7}, ice.ICE_ERR_INVALID_ARG),
                                           ({"promote_thresh": 2 ** 32 + 1}, ice.ICE_ERR_INVALID_ARG),
                                           ({"n_cap": 10}, ice.ICE_ERR_INVALID_ARG),
                                           ({"n_tokens": -1}, ice.ICE_ERR_INVALID_ARG),
                                           ({"np_cap": 0}, ice.ICE_ERR_INVALID_ARG),
                                           ({"page_cap": 0}, ice.ICE_ERR_INVALID_ARG),
                                           ({"n_sink": -1}, ice.ICE_ERR_INVALID_ARG),
                                           ({"n_window": -1}, ice.ICE_ERR_INVALID_ARG)],
                         ids=lambda x: "-".join(f"{k}={v}" for k, v in x.items()) if isinstance(x, dict) else str(x))
def test_invalid_params_rejected_on_host(lib, fields, status):
    p = ice.Config(batch=1, n_q_heads=8, n_kv_heads=2, n_tokens=100).params()
    for field, value in fields.items():
        setattr(p, field, value)
    with pytest.raises(ice.IceError) as ei:
        ice.ice_build_workspace_bytes(p)
    assert ei.value.status == status
    assert lib.ice_last_error().decode()


def test_struct_layouts_match_header():
    assert ctypes.sizeof(ice.IceParams) == 72
    assert ctypes.sizeof(ice.IceIndex) == 25 * 8


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "semantic_paged_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"\bimport\s+oracle\b|\bfrom\s+oracle\b|oracle\.c|liboracle|orc_", txt), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            txt = open(os.path.join(ROOT, "oracle", f), encoding="utf-8").read()
            assert not re.search(r"\bimport\s+semantic_paged_kv_gb300|\bfrom\s+semantic_paged_kv_gb300|"
                                 r"#\s*include\s*[<\"].*(ice\.h|\.cuh)", txt), f


def test_config_capacities_cover_positional_pages_and_descent_lists(lib):
    """Host-side sizing: the default page capacity and the decode output width
    include the sink / window pages; a three-level decode workspace holds the
    per-head page lists of the descent."""
    base = ice.Config(batch=1, n_q_heads=8, n_kv_heads=2, n_tokens=1000)
    pos = ice.Config(batch=1, n_q_heads=8, n_kv_heads=2, n_tokens=1000, n_sink=40, n_window=70)
    assert pos.n_pos == 3 + 5 and base.n_pos == 0
    assert pos.page_cap == base.page_cap + pos.n_pos
    assert ice.max_selected(pos, 64) == min(4 * 4 + 8, pos.page_cap)  # g = 4 heads x 4 pages + 8 positional
    three = ice.Config(batch=2, n_q_heads=8, n_kv_heads=2, n_tokens=1000, n_levels=3)
    assert ice.ice_decode_workspace_bytes(three.params(), 16, ice.max_selected(three, 16)) >= 4 * 4 * 4 * 32
    # descent: at most 32 pages per head; more is refused before anything runs
    assert ice.ice_build_workspace_bytes(three.params()) > ice.ice_build_workspace_bytes(
        ice.Config(batch=2, n_q_heads=8, n_kv_heads=2, n_tokens=1000).params())
