"""GPU parity of every step of the hot path against the CPU oracle, called
through the C ABI (libice.so) on seeded workloads shaped like the pages'
models: small enough for the oracle to finish in seconds, large enough to
span several tiles and a ragged tail, plus the edge cases."""
import numpy as np
import pytest
import torch

import oracle
import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import (DeviceDrawnRun, DeviceRun, check_build_level2, check_build_positional, check_build_unit,
                         check_decode_descent, check_decode_unit, check_level2_unit, check_pack_unit, host_tables,
                         to_dev)

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


def _all_units(run, budgets, fused=True, sample=None):
    for u in range(run.cfg.units):
        check_build_unit(run, u, sample_tokens=sample)
    for bgt in budgets:
        Q, buf, st = run.decode(bgt, fused=fused)
        assert st == ice.ICE_OK
        for u in range(run.cfg.units):
            check_decode_unit(run, u, Q, bgt, buf)


def _all_units_decode(run, budgets, fused=True):
    for bgt in budgets:
        Q, buf, st = run.decode(bgt, fused=fused)
        assert st == ice.ICE_OK
        for u in range(run.cfg.units):
            check_decode_unit(run, u, Q, bgt, buf)


def test_tiny_fp32_full():
    """The tiny fp32 workload (1 KV head, 4 query heads, N = 2048) end to end."""
    run = DeviceRun(W["tiny"])
    assert run.status == ice.ICE_OK
    _all_units(run, [64, 128], fused=True)
    _all_units(run, [64], fused=False)


@pytest.mark.parametrize("assign", ["auto", "simt"])
def test_llama_shaped_bf16_ragged(assign):
    """Llama-3.1-8B head layout (g = 4), bf16, a ragged N spanning several
    2048-token tiles and 128-row tiles, two sequences, needle planted."""
    w = W["llama31_8b_16k"].scaled(n_tokens=5003, batch=2, n_q_heads=8, n_kv_heads=2)
    run = DeviceRun(w, assign=assign)
    assert run.status == ice.ICE_OK
    _all_units(run, [64, 128, 256])


def test_many_parent_tiles_ring_wrap():
    """Np ~ 750 parents: three 256-parent MMA tiles per CTA, so the shared-memory
    ring and the two TMEM accumulators are reused; assignment checked on a
    seeded sample of tokens, everything else on all tokens."""
    w = W["llama31_8b_16k"].scaled(n_tokens=12003, n_q_heads=4, n_kv_heads=1)
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    _all_units(run, [256], sample=3000)


def test_llama_full_size_sampled():
    """The full Llama-3.1-8B-shaped layer (32 query / 8 KV heads, N = 16384,
    needle) in the launch configuration the benchmark times: promotion, pages,
    pool and decode checked in full, the assignment on 1500 sampled tokens per
    unit."""
    run = DeviceRun(W["llama31_8b_16k"])
    assert run.status == ice.ICE_OK
    _all_units(run, [64, 128, 256], sample=1500)


def test_fused_decode_equals_separate_calls():
    w = W["llama31_8b_16k"].scaled(n_tokens=3000, n_q_heads=8, n_kv_heads=2)
    run = DeviceRun(w)
    Q1, a, _ = run.decode(128, fused=True)
    Q2, b, _ = run.decode(128, fused=False)
    for x, y in [(a.sel_pages, b.sel_pages), (a.sel_count, b.sel_count), (a.kbuf, b.kbuf), (a.vbuf, b.vbuf),
                 (a.buf_len, b.buf_len)]:
        assert torch.equal(x, y)
    # the two paths split the pages differently before the log-sum-exp merge
    assert torch.max(torch.abs(a.O - b.O)).item() <= 1e-5


@pytest.mark.parametrize("shape", ["tiny_fp32", "llama_cluster", "qwen_many_units", "longchat_many_units",
                                   "qwen_one_cta_per_unit"])
def test_decode_without_contiguous_buffer(shape):
    """ice_decode_step with kbuf = vbuf = buf_len = NULL gathers the pages on
    chip only: same page lists and bit-identical O as with the buffer, on
    each kernel path (fp32 and bf16 per-unit clusters, the tensor-core score
    table with the selecting MMA attention for many units, and for one CTA per
    unit)."""
    w = {"tiny_fp32": W["tiny"],
         "llama_cluster": W["llama31_8b_16k"].scaled(n_tokens=3000, n_q_heads=8, n_kv_heads=2),
         "qwen_many_units": W["qwen3_32b_100k"].scaled(n_tokens=3000, batch=3, centres=256),
         "longchat_many_units": W["longchat_7b_100k"].scaled(n_tokens=2500, batch=1, n_q_heads=24, n_kv_heads=24,
                                                             centres=256),
         "qwen_one_cta_per_unit": W["qwen3_32b_100k"].scaled(n_tokens=2200, batch=20, centres=128)}[shape]
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    for bgt in (64, 256):
        Q, a, st_a = run.decode(bgt, contiguous=True)
        _, b, st_b = run.decode(bgt, contiguous=False)
        assert st_a == ice.ICE_OK and st_b == ice.ICE_OK
        assert torch.equal(a.sel_count, b.sel_count)
        assert torch.equal(a.sel_pages, b.sel_pages)
        assert torch.all(b.buf_len == 0)  # untouched
        assert torch.equal(a.O, b.O)
        check_decode_unit(run, run.cfg.units - 1, Q, bgt, a)


def test_qwen_shaped_g8_mha_longchat_shaped_g1():
    for w in (W["qwen3_32b_100k"].scaled(n_tokens=4100, batch=2, n_q_heads=16, n_kv_heads=2, centres=512),
              W["longchat_7b_100k"].scaled(n_tokens=4100, batch=1, n_q_heads=3, n_kv_heads=3, centres=512)):
        run = DeviceRun(w)
        assert run.status == ice.ICE_OK
        _all_units(run, [64, 256])


def test_many_units_take_select_and_attention_kernels():
    """More units than one wave of per-unit clusters: ice_decode_step runs the
    tensor-core selection and the split attention (Qwen3-shaped g = 8 and
    LongChat-shaped g = 1 groups), every unit checked."""
    for w in (W["qwen3_32b_100k"].scaled(n_tokens=3000, batch=3, centres=256),
              W["longchat_7b_100k"].scaled(n_tokens=2500, batch=1, n_q_heads=24, n_kv_heads=24, centres=256)):
        run = DeviceRun(w)
        assert run.status == ice.ICE_OK
        assert run.cfg.units * 8 > torch.cuda.get_device_properties(0).multi_processor_count
        for u in (0, run.cfg.units - 1):
            check_build_unit(run, u)
        _all_units_decode(run, [64, 256], fused=True)
        _all_units_decode(run, [128], fused=False)


def test_one_attention_cta_per_unit():
    """More units than SMs with a 128-page selection: the MMA attention runs
    one CTA per unit and writes O directly (fused and separate calls)."""
    w = W["qwen3_32b_100k"].scaled(n_tokens=2200, batch=20, centres=128)
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    assert run.cfg.units >= torch.cuda.get_device_properties(0).multi_processor_count
    for fused in (True, False):
        Q, buf, st = run.decode(256, fused=fused)
        assert st == ice.ICE_OK
        for u in (0, 77, run.cfg.units - 1):
            check_decode_unit(run, u, Q, 256, buf)


def test_longchat_100k_full_size_sampled():
    """The LongChat-7B-shaped layer at its full size (32 KV heads, N = 100000,
    log-normal norms) in the launch configuration the benchmark times: the
    selection runs as several segments per unit.  Build checked on two units
    (assignment on 800 sampled tokens), decode on four."""
    run = DeviceRun(W["longchat_7b_100k"])
    assert run.status == ice.ICE_OK
    for u in (3, 30):
        check_build_unit(run, u, sample_tokens=800)
    for bgt in (64, 256):
        Q, buf, st = run.decode(bgt)
        assert st == ice.ICE_OK
        for u in (0, 3, 17, 30):
            check_decode_unit(run, u, Q, bgt, buf)


def test_qwen_100k_full_size_sampled():
    """The Qwen3-32B-shaped decode batch at its full size (16 sequences x 8
    KV heads, g = 8, N = 100000, budget 256) on the benchmark's own inputs
    (drawn on the device) and in its launch configuration: the score table on
    the tensor cores, the per-unit selection and the MMA attention.  Build
    checked on two units (assignment on 800 sampled tokens), decode on four,
    across both ends of the batch."""
    run = DeviceDrawnRun(W["qwen3_32b_100k"])
    assert run.status == ice.ICE_OK
    assert run.cfg.units == 128
    for u in (9, 118):
        check_build_unit(run, u, sample_tokens=800)
    Q, buf, st = run.decode(256)
    assert st == ice.ICE_OK
    for u in (0, 9, 77, 127):
        check_decode_unit(run, u, Q, 256, buf)


def test_qwen_100k_three_levels_full_size_sampled():
    """The same batch with a third level, as the benchmark's descent decode
    runs it.  On eight units spread over the batch: level 1 as in the
    two-level build (assignment on 600 sampled tokens plus every parent);
    level-2 promotion exact, level-2 parents tie-aware and children exact
    against oracle.build_level2 over the checked level 1; the descent
    selection against oracle.select_descent with near-ties at either level
    enumerated; the attention over the selected pages."""
    w = W["qwen3_32b_100k"]
    run = DeviceDrawnRun(w, n_levels=3)
    assert run.status == ice.ICE_OK
    th = oracle.promote_threshold(w.promote_p)
    H, units = run.h, (0, 9, 31, 50, 64, 77, 118, 127)
    lv2s, idxs = {}, {}
    for u in units:
        check_build_unit(run, u, sample_tokens=600)
        b, h = run.unit(u)
        K = run.K[b, h].astype(np.float64)
        _, M2, e = oracle.lift(K)
        Np, P = int(H["n_parents"][u]), int(H["n_pages"][u])
        pt = H["parent_tok"][u, :Np]
        lv2 = oracle.build_level2(dict(parent_tok=pt, parent_keys=K[pt], parent_e=e[pt]), seed=w.seed, layer=0, seq=b,
                                  head=h, thresh=th)
        lv2s[u] = check_level2_unit(run, u, K, e, M2, lv2)
        pk, pv = run.pool(u)  # checked bit-exact by check_build_unit
        idxs[u] = dict(pool_k=pk, pool_v=pv, page_len=H["page_len"][u, :P])
    Q, buf, st = run.decode(256)
    assert st == ice.ICE_OK
    for u in units:
        check_decode_descent(run, u, Q, 256, buf, lv2s[u], idxs[u])


def test_promote_all_is_exact_topk_mips():
    """p = 1: one-token pages, so selection is exact top-k inner product search."""
    w = W["tiny"].scaled(n_tokens=700, promote_p=1.0)
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    assert int(run.h["n_pages"][0]) == 700
    _all_units(run, [16 * 5, 16 * 40])
    Q, buf, _ = run.decode(16 * 9)
    s = torch.tensor(Q[0], dtype=torch.float64) @ torch.tensor(run.K[0, 0], dtype=torch.float64).T
    top = torch.topk(s, 9, dim=1).indices
    got = set(buf.sel_pages[0, : int(buf.sel_count[0])].cpu().tolist())
    toks = set(run.h["page_tokens"][0, sorted(got), 0].tolist())
    assert toks == set(top.reshape(-1).tolist())


def test_pack_with_many_parents_uses_tile_kernels():
    """p = 0.95 on N = 10000: ~9500 parents, too many for the per-unit
    cluster packer's shared memory, so pages are built by the tile kernels
    (count, scan, rank); checked bit-exactly against the oracle's packing of
    the GPU's assignment, then decoded."""
    w = W["llama31_8b_16k"].scaled(n_tokens=10000, n_q_heads=4, n_kv_heads=1, promote_p=0.95)
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    assert run.cfg.np_cap * 24 > 225 * 1024
    check_pack_unit(run, 0)
    Q, buf, st = run.decode(256)
    assert st == ice.ICE_OK
    check_decode_unit(run, 0, Q, 256, buf)


def test_promote_none_is_sequential_paging():
    """p = 0: one parent (the smallest draw), so pages are sequential 16-token pages."""
    w = W["tiny"].scaled(n_tokens=1000, promote_p=0.0)
    run = DeviceRun(w)
    assert int(run.h["n_parents"][0]) == 1
    assert np.array_equal(run.h["token_page"][0, :1000], np.arange(1000) // 16)
    _all_units(run, [64])


def test_full_budget_is_dense_attention():
    w = W["llama31_8b_16k"].scaled(n_tokens=2500, n_q_heads=8, n_kv_heads=2)
    run = DeviceRun(w)
    P = int(run.h["n_pages"].max())
    Q, buf, _ = run.decode(16 * P)
    for u in range(run.cfg.units):
        assert int(buf.sel_count[u]) == int(run.h["n_pages"][u])
    q = torch.tensor(Q, dtype=torch.float64).reshape(1, 2, 4, 128)
    K = torch.tensor(run.K[0], dtype=torch.float64)[:, None].expand(2, 4, -1, -1)
    V = torch.tensor(run.V[0], dtype=torch.float64)[:, None].expand(2, 4, -1, -1)
    dense = torch.nn.functional.scaled_dot_product_attention(q[0][:, :, None], K, V)[:, :, 0].reshape(8, 128)
    assert torch.max(torch.abs(buf.O[0].double().cpu() - dense)) < 2e-3


@pytest.mark.parametrize("n", [0, 1, 17, 2049])
def test_small_and_empty_units(n):
    w = W["tiny"].scaled(n_tokens=n)
    run = DeviceRun(w, n_cap=max(n, 1))
    assert run.status == ice.ICE_OK
    _all_units(run, [64])


def test_needle_page_selected_at_every_budget():
    """Behavioural check from the passkey claim: the planted needle key's page
    is selected for its query head at budgets 64/128/256."""
    w = W["llama31_8b_16k"].scaled(n_tokens=6000, n_q_heads=8, n_kv_heads=2)
    run = DeviceRun(w)
    for bgt in (64, 128, 256):
        Q, buf, _ = run.decode(bgt)
        for u in range(run.cfg.units):
            pos = workloads.needle_position(w, 0, 0, u, 6000)
            page = int(run.h["token_page"][u, pos])
            got = buf.sel_pages[u, : int(buf.sel_count[u])].cpu().tolist()
            assert page in got


def test_capacity_error_is_reported_not_overrun():
    w = W["tiny"].scaled(n_tokens=3000)
    run = DeviceRun(w, np_cap=20, page_cap=200)
    assert run.status == ice.ICE_ERR_CAPACITY
    assert int(run.h["n_parents"][0]) == 20


def test_invalid_arguments_rejected():
    cfg = ice.Config(batch=1, n_q_heads=4, n_kv_heads=1, n_tokens=64)
    p = cfg.params()
    p.head_dim = 64
    with pytest.raises(ice.IceError) as ei:
        ice.ice_build_workspace_bytes(p)
    assert ei.value.status == ice.ICE_ERR_UNSUPPORTED
    p = cfg.params()
    idx = ice.Index(cfg)
    K = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    small = ice.workspace(256)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ice.IceError) as ei:
        ice.ice_build_index(p, K, K, idx, small, err)
    assert ei.value.status == ice.ICE_ERR_INVALID_ARG
    # the decode step's contiguous buffer: all three pointers or none
    buf = ice.DecodeBuffers(cfg, 64)
    Q = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ice.IceError) as ei:
        ice.ice_decode_step(p, idx, Q, 64, buf.sel_pages, buf.sel_count, None, buf.vbuf, buf.buf_len, 0.1, buf.O,
                            buf.ws, err)
    assert ei.value.status == ice.ICE_ERR_INVALID_ARG


def _reused_run(run0: DeviceRun, layer: int = 1, in_place: bool = False) -> DeviceRun:
    """Layer `layer` built by ice_build_index_reuse on run0's index."""
    r = object.__new__(DeviceRun)
    r.w, r.layer = run0.w, layer
    r.cfg = ice.Config(**{**run0.cfg.__dict__, "layer": layer})
    r.K, r.V = workloads.batch_kv(r.w, layer)
    dt = r.cfg.torch_dtype
    r.Kd, r.Vd = to_dev(r.K, dt), to_dev(r.V, dt)
    r.idx = run0.idx if in_place else ice.Index(r.cfg)
    r.params = r.cfg.params()
    r.ws = ice.workspace(ice.ice_build_workspace_bytes(r.params))
    r.err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ice.ice_build_index_reuse(r.params, r.Kd, r.Vd, run0.idx, r.idx, r.ws, r.err)
    r.status = ice.ice_check(r.err)
    r.h = host_tables(r.idx)
    return r


def _check_reuse_unit(run1, u, ref, N):
    """Every table, the lift values and the pool of reused unit u against the
    oracle's reuse."""
    H, Np, P = run1.h, len(ref["parent_tok"]), int(ref["n_pages"])
    assert int(H["n_parents"][u]) == Np and int(H["n_pages"][u]) == P and int(H["n_indexed"][u]) == N
    assert np.array_equal(H["parent_tok"][u, :Np], ref["parent_tok"])
    assert np.array_equal(H["token_parent"][u, :N], ref["token_parent"])
    for f in ("page_parent", "page_len", "page_tokens"):
        assert np.array_equal(H[f][u, :P], ref[f]), f
    assert np.array_equal(H["token_page"][u, :N], ref["token_page"])
    assert np.array_equal(H["token_slot"][u, :N], ref["token_slot"])
    assert abs(H["m2"][u] - ref["M2"]) <= 1e-12 * max(ref["M2"], 1e-30)
    assert np.allclose(H["parent_e"][u, :Np], ref["parent_e"], rtol=2e-7, atol=2e-7 * np.sqrt(ref["M2"]))
    assert np.array_equal(H["parent_keys"][u, :Np], ref["parent_keys"].astype(np.float32))
    pk, pv = run1.pool(u)
    assert np.array_equal(pk, ref["pool_k"].astype(np.float32)) and np.array_equal(pv, ref["pool_v"].astype(np.float32))
    if "level2" in ref:
        n2 = len(ref["level2"]["node2"])
        assert int(H["n_nodes2"][u]) == n2
        for f, n in (("node2", n2), ("parent2", Np), ("child_start", n2 + 1), ("children", Np)):
            assert np.array_equal(H[f][u, :n], ref["level2"][f]), f


@pytest.mark.parametrize("shape", ["llama_bf16", "tiny_fp32", "in_place"])
def test_reuse_build_matches_oracle(shape):
    """ice_build_index_reuse: the next layer on this layer's parents,
    assignment and pages, against oracle.build_unit_reuse over this layer's
    checked structure (every assignment difference a near-tie), on every
    unit, then the decode step over the reused index."""
    w = W["tiny"] if shape == "tiny_fp32" else W["llama31_8b_16k"].scaled(n_tokens=4003, batch=2, n_q_heads=8,
                                                                          n_kv_heads=2)
    run0 = DeviceRun(w)
    assert run0.status == ice.ICE_OK
    prevs = [check_build_positional(run0, u) for u in range(run0.cfg.units)]  # layer 0, checked
    run1 = _reused_run(run0, in_place=shape == "in_place")
    assert run1.status == ice.ICE_OK
    N = w.n_tokens
    for u in range(run1.cfg.units):
        b, h = run1.unit(u)
        # the oracle's reuse rule over the device's checked layer-0 structure
        ref = oracle.build_unit_reuse(run1.K[b, h], run1.V[b, h], prevs[u])
        _check_reuse_unit(run1, u, ref, N)
    for bgt in (64, 256):
        Q, buf, st = run1.decode(bgt)
        assert st == ice.ICE_OK
        for u in range(run1.cfg.units):
            check_decode_unit(run1, u, Q, bgt, buf)


@pytest.mark.parametrize("shape,n_sink,n_window", [("llama_bf16", 64, 250), ("tiny_fp32", 16, 100),
                                                   ("llama_bf16", 3, 0), ("many_units", 32, 130),
                                                   ("no_middle", 2000, 2000)])
def test_sink_and_window_pages(shape, n_sink, n_window):
    """Sink and recent-window tokens kept as positional pages outside the
    index: on every unit, the middle's index against
    oracle.build_unit_positional (parents and M exact, every assignment
    difference a checked near-tie, pages, spans and pool exact against the
    oracle's packing of the device's assignment), then every decode path
    attends over the selected pages plus all positional pages."""
    w = {"llama_bf16": W["llama31_8b_16k"].scaled(n_tokens=4003, batch=2, n_q_heads=8, n_kv_heads=2),
         "tiny_fp32": W["tiny"],
         "many_units": W["qwen3_32b_100k"].scaled(n_tokens=3000, batch=3, centres=256),
         "no_middle": W["llama31_8b_16k"].scaled(n_tokens=3000, n_q_heads=8, n_kv_heads=2)}[shape]
    run = DeviceRun(w, n_sink=n_sink, n_window=n_window)
    assert run.status == ice.ICE_OK
    for u in range(run.cfg.units):
        check_build_positional(run, u)
    for bgt in (64, 256):
        for fused in (True, False):
            Q, buf, st = run.decode(bgt, fused=fused)
            assert st == ice.ICE_OK
            for u in range(run.cfg.units):
                check_decode_unit(run, u, Q, bgt, buf)


def test_insert_rejected_with_positional_pages():
    w = W["llama31_8b_16k"].scaled(n_tokens=1000, n_q_heads=4, n_kv_heads=1)
    run = DeviceRun(w, n_sink=16, n_window=32)
    ws = ice.workspace(ice.ice_insert_workspace_bytes(run.params))
    kn = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ice.IceError) as ei:
        ice.ice_insert_tokens(run.params, run.idx, kn, kn, ws, run.err)
    assert ei.value.status == ice.ICE_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,n_sink,n_window", [("llama_bf16", 0, 0), ("tiny_fp32", 0, 0), ("many_units", 0, 0),
                                                   ("llama_bf16", 32, 96), ("dense_levels", 0, 0),
                                                   ("sparse_levels", 0, 0), ("wide_group_fp32", 0, 0)])
def test_three_levels_build_and_descent(shape, n_sink, n_window):
    """n_levels = 3, every unit: level 1 as in the two-level build; level-2
    promotion exact, level-2 parents tie-aware and children exact against
    oracle.build_level2 over the checked level 1; the descent selection
    against oracle.select_descent with near-ties at either level enumerated;
    the attention over the selected pages against the oracle; through
    ice_select_pages and ice_decode_step."""
    w = {"llama_bf16": W["llama31_8b_16k"].scaled(n_tokens=6003, batch=2, n_q_heads=8, n_kv_heads=2, centres=512),
         "tiny_fp32": W["tiny"],
         "many_units": W["qwen3_32b_100k"].scaled(n_tokens=4000, batch=3, centres=256),
         # p = 1/2: ~1500 level-2 nodes per unit
         "dense_levels": W["llama31_8b_16k"].scaled(n_tokens=6000, n_q_heads=8, n_kv_heads=2, promote_p=0.5),
         # p = 1/64: ~25 parents per unit, most units promote none again (the smallest-draw fallback)
         "sparse_levels": W["llama31_8b_16k"].scaled(n_tokens=1600, batch=2, n_q_heads=8, n_kv_heads=2,
                                                     promote_p=1.0 / 64),
         # fp32 with 12 query heads a group: the descent's 16-warp CTA, CUDA-core scoring of fp32 rows
         "wide_group_fp32": W["tiny"].scaled(n_tokens=3000, n_q_heads=12, n_kv_heads=1)}[shape]
    run = DeviceRun(w, n_levels=3, n_sink=n_sink, n_window=n_window)
    assert run.status == ice.ICE_OK
    idxs, lv2s = {}, {}
    for u in range(run.cfg.units):
        idxs[u] = check_build_positional(run, u)
        lv2s[u] = check_build_level2(run, u, idxs[u])
    for bgt in (64, 256):
        for fused in (True, False):
            Q, buf, st = run.decode(bgt, fused=fused)
            assert st == ice.ICE_OK
            for u in range(run.cfg.units):
                check_decode_descent(run, u, Q, bgt, buf, lv2s[u], idxs[u])


def test_reuse_with_sink_window_and_three_levels():
    """The inter-layer reuse of an index with sink / window pages and a third
    level: tables, level 2, keys, M over the middle and pool against
    oracle.build_unit_reuse; then the descent decode over the result."""
    w = W["llama31_8b_16k"].scaled(n_tokens=4003, batch=2, n_q_heads=8, n_kv_heads=2, centres=512)
    run0 = DeviceRun(w, n_levels=3, n_sink=48, n_window=160)
    assert run0.status == ice.ICE_OK
    prevs = {}
    for u in range(run0.cfg.units):  # layer 0 with its level 2, checked
        prevs[u] = check_build_positional(run0, u)
        prevs[u]["level2"] = check_build_level2(run0, u, prevs[u])
    run1 = _reused_run(run0)
    assert run1.status == ice.ICE_OK
    N, refs = w.n_tokens, {}
    for u in range(run1.cfg.units):
        b, h = run1.unit(u)
        refs[u] = oracle.build_unit_reuse(run1.K[b, h], run1.V[b, h], prevs[u])
        _check_reuse_unit(run1, u, refs[u], N)
    Q, buf, st = run1.decode(128)
    assert st == ice.ICE_OK
    for u, ref in refs.items():
        check_decode_descent(run1, u, Q, 128, buf, ref["level2"], ref)


@pytest.mark.parametrize("shape,budget,plan,attn", [
    ("cluster_bf16", 256, ice.ICE_PLAN_CLUSTER_BF16, ice.ICE_PLAN_ATTN_MMA),
    ("cluster_bf16_k64", 1024, ice.ICE_PLAN_CLUSTER, ice.ICE_PLAN_ATTN_MMA),
    ("cluster_fp32", 64, ice.ICE_PLAN_CLUSTER, ice.ICE_PLAN_ATTN_SIMT),
    ("score_select_many_units", 256, ice.ICE_PLAN_SCORE_SELECT, ice.ICE_PLAN_ATTN_MMA),
    ("score_topk_g16", 256, ice.ICE_PLAN_SCORE_TOPK, ice.ICE_PLAN_ATTN_MMA),
    ("simt_select_k64_bf16", 1024, ice.ICE_PLAN_SIMT, ice.ICE_PLAN_ATTN_MMA),
    ("simt_fp32_many_units", 64, ice.ICE_PLAN_SIMT, ice.ICE_PLAN_ATTN_SIMT),
    ("simt_attention_bf16", 1024, ice.ICE_PLAN_SIMT, ice.ICE_PLAN_ATTN_SIMT)])
def test_every_decode_plan_against_the_oracle(shape, budget, plan, attn):
    """Each kernel path of ice_decode_step (ice_decode_plan names it) and
    each attention kernel, on a shape that selects it: the bf16 and generic
    cluster decodes, the score table with selecting attention CTAs and with
    the top-k kernel (16 query heads per group), the SIMT selection (more than
    32 pages per head) with the MMA and with the SIMT attention (a warp would
    hold more than 32 pages), and fp32 with many units.  The step (fused call
    and separate calls) checked against the oracle."""
    w = {"cluster_bf16": W["llama31_8b_16k"].scaled(n_tokens=3000, n_q_heads=8, n_kv_heads=2),
         "cluster_bf16_k64": W["llama31_8b_16k"].scaled(n_tokens=3000, n_q_heads=8, n_kv_heads=2),
         "cluster_fp32": W["tiny"],
         "score_select_many_units": W["qwen3_32b_100k"].scaled(n_tokens=2200, batch=20, centres=128),
         "score_topk_g16": W["llama31_8b_16k"].scaled(n_tokens=3000, batch=12, n_q_heads=32, n_kv_heads=2),
         "simt_select_k64_bf16": W["llama31_8b_16k"].scaled(n_tokens=3000, batch=3),
         "simt_fp32_many_units": W["tiny"].scaled(n_tokens=1500, batch=20),
         "simt_attention_bf16": W["qwen3_32b_100k"].scaled(n_tokens=3000, batch=19, centres=128)}[shape]
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    max_sel = ice.max_selected(run.cfg, budget)
    assert ice.ice_decode_plan(run.params, budget, max_sel) == (plan, attn)
    units = list(range(run.cfg.units)) if run.cfg.units <= 24 else [0, 7, 50, run.cfg.units - 1]
    for u in units[:4]:
        check_build_unit(run, u)
    for fused in (True, False):
        Q, buf, st = run.decode(budget, fused=fused)
        assert st == ice.ICE_OK
        for u in units:
            check_decode_unit(run, u, Q, budget, buf)


def test_three_levels_many_level2_nodes():
    """p = 1/2 on one 20,000-token unit: about 10,000 parents and 5,000
    level-2 nodes, more than the descent keeps in shared memory (about 2,700
    per head at g = 4), so the level-2 scores go through the decode
    workspace.  Level 1, level 2 and the descent selection (near-ties
    enumerated) against the oracle, and the attention over the selected
    pages."""
    w = W["llama31_8b_16k"].scaled(n_tokens=20000, n_q_heads=4, n_kv_heads=1, promote_p=0.5)
    run = DeviceRun(w, n_levels=3)
    assert run.status == ice.ICE_OK
    assert int(run.h["n_nodes2"][0]) > 4096
    idx = check_build_positional(run, 0)
    lv2 = check_build_level2(run, 0, idx)
    assert ice.ice_decode_plan(run.params, 256, ice.max_selected(run.cfg, 256))[0] == ice.ICE_PLAN_DESCENT
    for bgt in (64, 256):
        for fused in (True, False):
            Q, buf, st = run.decode(bgt, fused=fused)
            assert st == ice.ICE_OK
            check_decode_descent(run, 0, Q, bgt, buf, lv2, idx)


def test_three_levels_many_candidates_per_head():
    """p = 1/64 on one 65,536-token unit with 16 query heads per KV head:
    about 1,000 parents under some 20 level-2 nodes.  At a budget of 512
    tokens (k = 32) each head takes every level-2 node, so its candidates (all
    parents) outgrow the keys the descent keeps in shared memory per head
    (about 630 at g = 16) and go through the decode workspace; at 64 tokens
    they fit.  Level 1, level 2, the descent selection (near-ties enumerated)
    and the attention against the oracle."""
    w = W["llama31_8b_16k"].scaled(n_tokens=65536, n_q_heads=16, n_kv_heads=1, promote_p=1.0 / 64)
    run = DeviceRun(w, n_levels=3)
    assert run.status == ice.ICE_OK
    idx = check_build_positional(run, 0)
    lv2 = check_build_level2(run, 0, idx)
    starts = np.asarray(lv2["child_start"])
    # at k = 32 pages every head takes all level-2 nodes: all parents are its candidates
    assert len(starts) - 1 <= 32 and int(starts[-1]) > 640
    assert ice.ice_decode_plan(run.params, 512, ice.max_selected(run.cfg, 512))[0] == ice.ICE_PLAN_DESCENT
    for bgt in (64, 512):
        Q, buf, st = run.decode(bgt, fused=True)
        assert st == ice.ICE_OK
        check_decode_descent(run, 0, Q, bgt, buf, lv2, idx)
