"""Failure handling, with every failure made on the host or by a bounded
wait that nothing completes; no test faults, traps or hangs the GPU.

ICE_FAULT (read by the library at every call) injects:
  alloc     the host pool's first pinned allocation fails -> ICE_ERR_OOM
  hostpool  the host pool fails after its allocations     -> ICE_ERR_CUDA
  copy      the staged gather's bulk copy fails           -> ICE_ERR_CUDA
  timeout   the decode kernels' TMA producers issue no copy and their
            bounded waits give up after 20 ms             -> ICE_ERR_TIMEOUT
Each test checks the status, that nothing leaked or stayed broken, and that
the next call without the fault gives the oracle's result."""
import numpy as np
import pytest
import torch

import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import DeviceRun, check_decode_unit

pytestmark = pytest.mark.gpu


def _rss() -> int:
    with open("/proc/self/statm") as f:
        return int(f.read().split()[1]) * 4096


def _cfg(units=2):
    return ice.Config(batch=1, n_q_heads=4 * units, n_kv_heads=units, n_tokens=300000)  # two 0.6 GB pools


@pytest.mark.parametrize("fault,status", [("alloc", ice.ICE_ERR_OOM), ("hostpool", ice.ICE_ERR_CUDA)])
def test_host_pool_create_faults_leave_nothing_behind(monkeypatch, fault, status):
    cfg = _cfg()
    ok = ice.HostPool(cfg, 64, n_threads=2)  # warm the pinned allocator once
    ok.close()
    before = _rss()
    monkeypatch.setenv("ICE_FAULT", fault)
    for _ in range(3):
        with pytest.raises(ice.IceError) as ei:
            ice.HostPool(cfg, 64, n_threads=2)
        assert ei.value.status == status
    # pinned pages are resident: three leaked pool pairs would show as 3.6 GB
    assert _rss() - before < 512 << 20
    monkeypatch.delenv("ICE_FAULT")
    hp = ice.HostPool(cfg, 64, n_threads=2)
    hp.close()


def test_staged_copy_fault_then_recovery(monkeypatch):
    w = workloads.WORKLOADS["qwen3_32b_100k"].scaled(n_tokens=3000, batch=1, n_q_heads=16, n_kv_heads=2,
                                                     centres=256)
    run = DeviceRun(w, host_pool=lambda cfg: ice.HostPool(cfg, ice.max_selected(cfg, 128), n_threads=2))
    try:
        Q, buf, st = run.decode(128)
        assert st == ice.ICE_OK
        cfg, hp = run.cfg, run.hp
        max_sel = buf.sel_pages.shape[-1]
        sel_h, cnt_h, plen_h = buf.sel_pages.cpu(), buf.sel_count.cpu(), run.idx.page_len.cpu()
        dst = torch.zeros(hp.staging_bytes, dtype=torch.uint8, device="cuda")
        monkeypatch.setenv("ICE_FAULT", "copy")
        with pytest.raises(ice.IceError) as ei:
            ice.ice_host_pool_gather_h2d(hp, cfg.params(), sel_h, cnt_h, plen_h, max_sel, dst)
        assert ei.value.status == ice.ICE_ERR_CUDA
        torch.cuda.synchronize()
        assert int(dst.count_nonzero()) == 0  # nothing was copied
        monkeypatch.delenv("ICE_FAULT")
        ice.ice_host_pool_gather_h2d(hp, cfg.params(), sel_h, cnt_h, plen_h, max_sel, dst)
        U, S, d = cfg.units, cfg.page_size, cfg.head_dim
        nb = U * max_sel * S * d * 2
        kbuf = dst[:nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
        vbuf = dst[nb:2 * nb].view(torch.bfloat16).reshape(U, max_sel, S, d)
        blen = dst[2 * nb:2 * nb + U * max_sel * 4].view(torch.int32).reshape(U, max_sel)
        torch.cuda.synchronize()
        assert torch.equal(kbuf, buf.kbuf) and torch.equal(vbuf, buf.vbuf) and torch.equal(blen, buf.buf_len)
    finally:
        run.hp.close()


def test_attention_wait_timeout_is_reported_and_the_context_stays_usable(monkeypatch):
    """With the TMA producers silenced, every warp's bounded wait gives up:
    ice_sparse_attn_decode (no error word) leaves NaN in O, and the decode
    step (the one-kernel decode: parent-table scan and page stream both
    silenced) reports ICE_ERR_TIMEOUT through ice_check.  The kernels
    return; the same calls without the fault then match the oracle."""
    w = workloads.WORKLOADS["qwen3_32b_100k"].scaled(n_tokens=3000, batch=3, centres=256)
    run = DeviceRun(w)
    assert run.status == ice.ICE_OK
    Q, ref, st = run.decode(256, fused=False)
    assert st == ice.ICE_OK
    Qd = run.queries()[1]
    scale = 1.0 / np.sqrt(128)
    monkeypatch.setenv("ICE_FAULT", "timeout")
    O = torch.zeros_like(ref.O)
    ice.ice_sparse_attn_decode(run.params, Qd, ref.kbuf, ref.vbuf, ref.buf_len, ref.sel_count, scale, O, ref.ws)
    torch.cuda.synchronize()
    assert torch.isnan(O).all()
    buf = ice.DecodeBuffers(run.cfg, 256)
    ice.ice_decode_step(run.params, run.idx, Qd, 256, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf, buf.buf_len,
                        scale, buf.O, buf.ws, run.err)
    assert ice.ice_check(run.err) == ice.ICE_ERR_TIMEOUT
    monkeypatch.delenv("ICE_FAULT")
    ice.ice_sparse_attn_decode(run.params, Qd, ref.kbuf, ref.vbuf, ref.buf_len, ref.sel_count, scale, O, ref.ws)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(O - ref.O)).item() <= 1e-5
    Q, buf, st = run.decode(256)
    assert st == ice.ICE_OK
    for u in range(run.cfg.units):
        check_decode_unit(run, u, Q, 256, buf)
