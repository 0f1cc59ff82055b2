"""The pinned host page pool (step a12): building into it and decoding
straight from it over the CPU-GPU link (direct), and the staged path (ids to
the host, host-thread gather into pinned staging, one bulk cudaMemcpyAsync,
attention over the copy).  Both are checked against the CPU oracle: the
build (promotion, assignment tie-aware, pages and the pool read back from
host memory), the selection (near-ties enumerated), the gathered pages and
the attention; and against the same layer with the pool in HBM, bit for bit
where the two must agree."""
import os
import types

import numpy as np
import pytest
import torch

import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import DeviceDrawnRun, DeviceRun, check_build_unit, check_decode_unit

pytestmark = pytest.mark.gpu

BUDGET = 256
SCALE = 1.0 / np.sqrt(128)


def _pool_factory(budget, threads):
    return lambda cfg: ice.HostPool(cfg, ice.max_selected(cfg, budget), n_threads=threads)


def _staged(run, Qd, buf):
    """The staged path over the direct decode's selection: host gather, one
    bulk copy, ice_sparse_attn_decode; returns decode buffers as the checks
    read them (kbuf, vbuf, buf_len, sel_pages, sel_count, O)."""
    cfg, hp = run.cfg, run.hp
    max_sel = buf.sel_pages.shape[-1]
    sel_h, cnt_h = buf.sel_pages.cpu(), buf.sel_count.cpu()
    plen_h = run.idx.page_len.cpu()
    dst = torch.zeros(hp.staging_bytes, dtype=torch.uint8, device="cuda")
    ice.ice_host_pool_gather_h2d(hp, cfg.params(), sel_h, cnt_h, plen_h, max_sel, dst)
    U, S, d = cfg.units, cfg.page_size, cfg.head_dim
    nb = U * max_sel * S * d * 2
    kbuf = dst[:nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
    vbuf = dst[nb:2 * nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
    blen = dst[2 * nb:2 * nb + U * max_sel * 4].view(torch.int32).reshape(U, max_sel)
    O = torch.full_like(buf.O, float("nan"))
    ws = ice.workspace(ice.ice_decode_workspace_bytes(cfg.params(), BUDGET, max_sel))
    ice.ice_sparse_attn_decode(cfg.params(), Qd, kbuf, vbuf, blen, buf.sel_count, SCALE, O, ws)
    torch.cuda.synchronize()
    return types.SimpleNamespace(kbuf=kbuf, vbuf=vbuf, buf_len=blen, sel_pages=buf.sel_pages,
                                 sel_count=buf.sel_count, O=O), (sel_h, cnt_h, plen_h, dst)


def test_host_pool_direct_and_staged_against_the_oracle():
    w = workloads.WORKLOADS["qwen3_32b_100k"].scaled(n_tokens=4100, batch=2, n_q_heads=16, n_kv_heads=2, centres=512)
    run = DeviceRun(w, host_pool=_pool_factory(BUDGET, 4))
    try:
        assert run.status == ice.ICE_OK
        for u in range(run.cfg.units):
            check_build_unit(run, u)  # the pool as read back from pinned host memory
        Q, buf, st = run.decode(BUDGET)  # direct: pages read over the CPU-GPU link
        assert st == ice.ICE_OK
        for u in range(run.cfg.units):
            check_decode_unit(run, u, Q, BUDGET, buf)
        staged, (sel_h, cnt_h, plen_h, dst) = _staged(run, run.queries()[1], buf)
        for u in range(run.cfg.units):
            check_decode_unit(run, u, Q, BUDGET, staged)
        # the same layer with the pool in HBM: identical selection, buffer and output
        ref = DeviceRun(w)
        _, rbuf, _ = ref.decode(BUDGET)
        for a, b in [(buf.sel_pages, rbuf.sel_pages), (buf.sel_count, rbuf.sel_count), (buf.kbuf, rbuf.kbuf),
                     (buf.vbuf, rbuf.vbuf), (buf.buf_len, rbuf.buf_len), (buf.O, rbuf.O)]:
            assert torch.equal(a, b)
        # host-side checks: a page id outside the pool or a count outside [0, max_sel] is refused
        max_sel = buf.sel_pages.shape[-1]
        bad_sel, bad_cnt = sel_h.clone(), cnt_h.clone()
        bad_sel[0, 0] = run.cfg.page_cap
        bad_cnt[1] = max_sel + 1
        for s_h, c_h in ((bad_sel, cnt_h), (sel_h, bad_cnt)):
            with pytest.raises(ice.IceError) as ex:
                ice.ice_host_pool_gather_h2d(run.hp, run.cfg.params(), s_h, c_h, plen_h, max_sel, dst)
            assert ex.value.status == ice.ICE_ERR_INVALID_ARG
    finally:
        run.hp.close()


def test_host_pool_qwen_full_size():
    """The Qwen3-32B-shaped batch at its full size (16 x 8 units, N = 100000,
    budget 256) with the page pool in pinned host memory, as the benchmark's
    host-pool part runs it on its device-drawn inputs: the build on three
    units against the oracle (assignment on 600 sampled tokens, pages and the
    host-resident pool in full), the direct decode and the staged path on
    four units against the oracle, and the direct decode bit for bit against
    the same batch with the pool in HBM on every unit."""
    w = workloads.WORKLOADS["qwen3_32b_100k"]
    run = DeviceDrawnRun(w, host_pool=_pool_factory(BUDGET, min(16, os.cpu_count() or 1)))
    try:
        assert run.status == ice.ICE_OK
        for u in (0, 70, 127):
            check_build_unit(run, u, sample_tokens=600)
        Q, buf, st = run.decode(BUDGET)
        assert st == ice.ICE_OK
        units = (0, 9, 70, 127)
        for u in units:
            check_decode_unit(run, u, Q, BUDGET, buf)
        staged, _ = _staged(run, run.queries()[1], buf)
        for u in units:
            check_decode_unit(run, u, Q, BUDGET, staged)
        # the HBM-pool decode of the same batch (same device draws): identical on every unit
        idx = ice.Index(run.cfg)
        p = run.cfg.params()
        ws = ice.workspace(ice.ice_build_workspace_bytes(p))
        ice.ice_build_index(p, run.Kd, run.Vd, idx, ws, run.err)
        del ws
        rbuf = ice.DecodeBuffers(run.cfg, BUDGET)
        ice.ice_decode_step(p, idx, run.queries()[1], BUDGET, rbuf.sel_pages, rbuf.sel_count, rbuf.kbuf, rbuf.vbuf,
                            rbuf.buf_len, SCALE, rbuf.O, rbuf.ws, run.err)
        assert ice.ice_check(run.err) == ice.ICE_OK
        for a, b in [(buf.sel_pages, rbuf.sel_pages), (buf.sel_count, rbuf.sel_count), (buf.kbuf, rbuf.kbuf),
                     (buf.vbuf, rbuf.vbuf), (buf.buf_len, rbuf.buf_len), (buf.O, rbuf.O)]:
            assert torch.equal(a, b)
    finally:
        run.hp.close()
