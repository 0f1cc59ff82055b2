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


@pytest.mark.parametrize("n,p,n_sink,n_window", [(16384, 1 / 16, 0, 0), (100000, 1 / 16, 0, 0), (5003, 0.95, 0, 0),
                                                 (700, 1.0, 0, 0), (1000, 0.0, 40, 70), (0, 1 / 16, 0, 0)])
def test_default_capacities(lib, n, p, n_sink, n_window):
    """ice_default_capacities: np_cap = the binomial mean of promoted tokens
    plus 8 standard deviations plus 16 (at most n_cap, at least 1); page_cap
    = ice_page_bound(n_cap, np_cap) + the positional pages."""
    import math
    prm = ice.Config(batch=1, n_q_heads=4, n_kv_heads=1, n_tokens=n, promote_p=p, n_sink=n_sink,
                     n_window=n_window, np_cap=1, page_cap=1).params()
    prm.np_cap = prm.page_cap = 0
    assert lib.ice_default_capacities(ctypes.byref(prm)) == 0
    nc = max(n, 1)
    q = ice.promote_threshold(p) / 2 ** 32
    mu = nc * q
    assert prm.n_cap == nc
    assert prm.np_cap == max(1, min(nc, math.floor(mu + 8 * math.sqrt(mu * (1 - q) + 1) + 16)))
    assert prm.page_cap == max(1, ice.ice_page_bound(nc, prm.np_cap) + lib.ice_positional_pages(n, n_sink, n_window, 16))
    cfg = ice.Config(batch=1, n_q_heads=4, n_kv_heads=1, n_tokens=n, promote_p=p, n_sink=n_sink, n_window=n_window)
    assert (cfg.np_cap, cfg.page_cap) == (prm.np_cap, prm.page_cap)
    bad = ice.Config(batch=1, n_q_heads=4, n_kv_heads=1, n_tokens=100).params()
    bad.page_size = 8
    assert lib.ice_default_capacities(ctypes.byref(bad)) == ice.ICE_ERR_UNSUPPORTED


@pytest.mark.parametrize("levels,with_pool,dtype", [(2, 1, ice.ICE_BF16), (3, 1, ice.ICE_FP32), (2, 0, ice.ICE_BF16)])
def test_index_slab_layout(lib, levels, with_pool, dtype):
    """ice_index_bytes / ice_index_layout: every array of the index at a
    256-byte aligned offset of one slab, in field order, disjoint, each as
    large as its documented shape; the pool and the level-2 arrays only when
    counted.  Nothing is read or written at the (fake) base address."""
    cfg = ice.Config(batch=3, n_q_heads=8, n_kv_heads=2, n_tokens=1000, n_levels=levels, dtype=dtype)
    prm = cfg.params()
    n = ctypes.c_size_t(0)
    assert lib.ice_index_bytes(ctypes.byref(prm), with_pool, ctypes.byref(n)) == 0
    base = 1 << 40
    st = ice.IceIndex()
    assert lib.ice_index_layout(ctypes.byref(prm), with_pool, base, ctypes.byref(st)) == 0
    U, Np, Pc, Nc, S, d = cfg.units, cfg.np_cap, cfg.page_cap, cfg.n_cap, 16, 128
    esz = 2 if dtype == ice.ICE_BF16 else 4
    size = {"n_parents": 4 * U, "n_pages": 4 * U, "n_indexed": 4 * U, "m2": 8 * U, "parent_tok": 4 * U * Np,
            "parent_keys": esz * U * Np * d, "parent_e": 4 * U * Np, "parent_corr": 4 * U * Np,
            "parent_first_page": 4 * U * Np, "parent_last_page": 4 * U * Np, "parent_n_pages": 4 * U * Np,
            "page_parent": 4 * U * Pc, "page_len": 4 * U * Pc, "page_next": 4 * U * Pc,
            "page_tokens": 4 * U * Pc * S, "token_parent": 4 * U * Nc, "token_page": 4 * U * Nc,
            "token_slot": 4 * U * Nc, "pool_k": esz * U * Pc * S * d, "pool_v": esz * U * Pc * S * d,
            "n_nodes2": 4 * U, "node2": 4 * U * Np, "parent2": 4 * U * Np, "child_start": 4 * U * (Np + 1),
            "children": 4 * U * Np}
    end = 0
    for f in ice.INDEX_FIELDS:
        ptr = getattr(st, f)
        counted = (with_pool or f not in ("pool_k", "pool_v")) and (levels == 3 or f not in
                                                                      ("n_nodes2", "node2", "parent2",
                                                                       "child_start", "children"))
        if not counted:
            assert ptr is None, f
            continue
        off = ptr - base
        assert off % 256 == 0 and off >= end, f
        end = off + size[f]
    assert end <= n.value < end + 256
    # refusals: unaligned or missing base
    assert lib.ice_index_layout(ctypes.byref(prm), with_pool, base + 16, ctypes.byref(st)) == ice.ICE_ERR_INVALID_ARG
    assert lib.ice_index_layout(ctypes.byref(prm), with_pool, None, ctypes.byref(st)) == ice.ICE_ERR_INVALID_ARG


def test_decode_plan_host_query(lib):
    """ice_decode_plan answers on the host (where the SM count reads as 1, so
    no cluster plan fits): bf16 with g <= 8 and k <= 32 takes the score table
    and selecting attention CTAs, 16 heads per group the top-k kernel, more
    than 32 pages per head the SIMT selection, three levels the descent."""
    base = dict(batch=1, n_q_heads=8, n_kv_heads=2, n_tokens=3000)
    plan = lambda cfg, budget: ice.ice_decode_plan(cfg.params(), budget, ice.max_selected(cfg, budget))[0]
    assert plan(ice.Config(**base), 256) == ice.ICE_PLAN_SCORE_SELECT
    assert plan(ice.Config(**{**base, "n_q_heads": 32}), 256) == ice.ICE_PLAN_SCORE_TOPK
    assert plan(ice.Config(**base), 1024) == ice.ICE_PLAN_SIMT
    assert plan(ice.Config(**base, n_levels=3), 256) == ice.ICE_PLAN_DESCENT
    with pytest.raises(ice.IceError):
        ice.ice_decode_plan(ice.Config(**base).params(), -1, 8)
