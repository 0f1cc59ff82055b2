"""The pinned host page pool (step a12): building into it and decoding
straight from it (direct), and the staged path (host-thread gather into
pinned staging, one bulk cudaMemcpyAsync, attention over the copy), both
checked against the same layer built and decoded with the pool in HBM."""
import os

import numpy as np
import pytest
import torch

import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import cfg_of, to_dev

pytestmark = pytest.mark.gpu


def _build(cfg, K, V, host_pool=None):
    idx = ice.Index(cfg, host_pool=host_pool)
    p = cfg.params()
    ws = ice.workspace(ice.ice_build_workspace_bytes(p))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ice.ice_build_index(p, K, V, idx, ws, err)
    assert ice.ice_check(err) == ice.ICE_OK
    return idx


def _decode(cfg, idx, Q, budget):
    buf = ice.DecodeBuffers(cfg, budget)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ice.ice_decode_step(cfg.params(), idx, Q, budget, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf, buf.buf_len,
                        1.0 / np.sqrt(128), buf.O, buf.ws, err)
    assert ice.ice_check(err) == ice.ICE_OK
    return buf


def test_host_pool_direct_and_staged_match_hbm_pool():
    w = workloads.WORKLOADS["qwen3_32b_100k"].scaled(n_tokens=4100, batch=2, n_q_heads=16, n_kv_heads=2, centres=512)
    cfg = cfg_of(w)
    K, V = workloads.batch_kv(w)
    Q = workloads.batch_queries(w)
    dt = cfg.torch_dtype
    Kd, Vd, Qd = to_dev(K, dt), to_dev(V, dt), to_dev(Q, dt)
    budget = 256
    ref_idx = _build(cfg, Kd, Vd)
    ref = _decode(cfg, ref_idx, Qd, budget)

    max_sel = ice.max_selected(cfg, budget)
    hp = ice.HostPool(cfg, max_sel, n_threads=4)
    try:
        idx = _build(cfg, Kd, Vd, host_pool=hp)
        # the pages written over the CPU-GPU link are the HBM pool's pages
        for u in range(cfg.units):
            P = int(ref_idx.n_pages[u])
            for which, dev in (("k", ref_idx.pool_k), ("v", ref_idx.pool_v)):
                host = hp.host_array(which)[u, :P]
                assert np.array_equal(host, dev[u, :P].view(torch.int16).cpu().numpy().view(np.uint16))
        # direct: the fused decode reads its pages from host memory
        got = _decode(cfg, idx, Qd, budget)
        for a, b in [(got.sel_pages, ref.sel_pages), (got.sel_count, ref.sel_count), (got.kbuf, ref.kbuf),
                     (got.vbuf, ref.vbuf), (got.buf_len, ref.buf_len), (got.O, ref.O)]:
            assert torch.equal(a, b)
        # staged: ids back to the host, host gather, one bulk H2D copy, attention
        sel_h, cnt_h = got.sel_pages.cpu(), got.sel_count.cpu()
        plen_h = idx.page_len.cpu()
        dst = torch.zeros(hp.staging_bytes, dtype=torch.uint8, device="cuda")
        ice.ice_host_pool_gather_h2d(hp, cfg.params(), sel_h, cnt_h, plen_h, max_sel, dst)
        U, S, d = cfg.units, cfg.page_size, cfg.head_dim
        nb = U * max_sel * S * d * 2
        kbuf = dst[:nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
        vbuf = dst[nb:2 * nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
        blen = dst[2 * nb:2 * nb + U * max_sel * 4].view(torch.int32).reshape(U, max_sel)
        assert torch.equal(blen, ref.buf_len)
        for u in range(U):
            n = int(ref.sel_count[u])
            assert torch.equal(kbuf[u, :n], ref.kbuf[u, :n]) and torch.equal(vbuf[u, :n], ref.vbuf[u, :n])
        O = torch.zeros_like(ref.O)
        ws = ice.workspace(ice.ice_decode_workspace_bytes(cfg.params(), budget, max_sel))
        ice.ice_sparse_attn_decode(cfg.params(), Qd, kbuf, vbuf, blen, ref.sel_count, 1.0 / np.sqrt(128), O, ws)
        # a different split of the pages before the log-sum-exp merge than the fused step
        assert torch.max(torch.abs(O - ref.O)).item() <= 1e-5
        # host-side checks: a page id outside the pool or a count outside [0, max_sel] is refused, nothing copied
        bad_sel, bad_cnt = sel_h.clone(), cnt_h.clone()
        bad_sel[0, 0] = cfg.page_cap
        bad_cnt[1] = max_sel + 1
        for s_h, c_h in ((bad_sel, cnt_h), (sel_h, bad_cnt)):
            with pytest.raises(ice.IceError) as ex:
                ice.ice_host_pool_gather_h2d(hp, cfg.params(), s_h, c_h, plen_h, max_sel, dst)
            assert ex.value.status == ice.ICE_ERR_INVALID_ARG
    finally:
        hp.close()


def test_host_pool_qwen_full_size():
    """The Qwen3-32B-shaped batch at its full size (16 x 8 units, N = 100000,
    budget 256) with the page pool in pinned host memory, as the benchmark's
    host-pool part runs it on its device-drawn inputs: the pages written over
    the CPU-GPU link equal the HBM pool's on three units, the direct decode
    equals the HBM-pool decode bit for bit on every unit, and the staged path
    (host gather, one bulk copy, attention) reproduces the contiguous buffer
    and the output."""
    w = workloads.WORKLOADS["qwen3_32b_100k"]
    cfg = cfg_of(w)
    Kd, Vd, C = workloads.batch_kv_device(w)
    Qd = workloads.batch_queries_device(w, C)
    del C
    budget = 256
    ref_idx = _build(cfg, Kd, Vd)
    ref = _decode(cfg, ref_idx, Qd, budget)
    max_sel = ice.max_selected(cfg, budget)
    hp = ice.HostPool(cfg, max_sel, n_threads=min(16, os.cpu_count() or 1))
    try:
        idx = _build(cfg, Kd, Vd, host_pool=hp)
        del Kd, Vd
        for u in (0, 70, 127):
            P = int(ref_idx.n_pages[u])
            for which, dev in (("k", ref_idx.pool_k), ("v", ref_idx.pool_v)):
                host = hp.host_array(which)[u, :P]
                assert np.array_equal(host, dev[u, :P].view(torch.int16).cpu().numpy().view(np.uint16))
        got = _decode(cfg, idx, Qd, budget)
        for a, b in [(got.sel_pages, ref.sel_pages), (got.sel_count, ref.sel_count), (got.kbuf, ref.kbuf),
                     (got.vbuf, ref.vbuf), (got.buf_len, ref.buf_len), (got.O, ref.O)]:
            assert torch.equal(a, b)
        sel_h, cnt_h = got.sel_pages.cpu(), got.sel_count.cpu()
        plen_h = idx.page_len.cpu()
        dst = torch.zeros(hp.staging_bytes, dtype=torch.uint8, device="cuda")
        ice.ice_host_pool_gather_h2d(hp, cfg.params(), sel_h, cnt_h, plen_h, max_sel, dst)
        U, S, d = cfg.units, cfg.page_size, cfg.head_dim
        nb = U * max_sel * S * d * 2
        kbuf = dst[:nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
        vbuf = dst[nb:2 * nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
        blen = dst[2 * nb:2 * nb + U * max_sel * 4].view(torch.int32).reshape(U, max_sel)
        assert torch.equal(blen, ref.buf_len)
        n = ref.sel_count.long()
        live = torch.arange(max_sel, device="cuda")[None, :] < n[:, None]  # [U, max_sel]: selected slots
        assert torch.equal(kbuf[live], ref.kbuf[live]) and torch.equal(vbuf[live], ref.vbuf[live])
        O = torch.zeros_like(ref.O)
        ws = ice.workspace(ice.ice_decode_workspace_bytes(cfg.params(), budget, max_sel))
        ice.ice_sparse_attn_decode(cfg.params(), Qd, kbuf, vbuf, blen, ref.sel_count, 1.0 / np.sqrt(128), O, ws)
        assert torch.max(torch.abs(O.float() - ref.O.float())).item() <= 1e-5
    finally:
        hp.close()
