"""The copy / build / decode overlap across layers (the on-device form of
the pages' three-stage pipeline: while layer i is indexed and decoded on the
compute stream, layer i + 1's K, V and Q move from pinned host memory on a
second stream).  Every layer's index and decode step are checked against the
oracle, so the overlap changes no result.  The pattern is the one the
benchmark's e2e leg times; the library needs nothing for it beyond the
stream argument of every entry point."""
import numpy as np
import pytest
import torch

import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import cfg_of, check_build_unit, check_decode_unit, host_tables

pytestmark = pytest.mark.gpu


class _Layer:
    """What the parity helpers read from one layer of the overlapped run."""

    def __init__(self, w, layer, cfg, idx, K, V):
        self.w, self.layer, self.cfg, self.idx, self.K, self.V = w, layer, cfg, idx, K, V

    def unit(self, u):
        return u // self.cfg.n_kv_heads, u % self.cfg.n_kv_heads

    def pool(self, u):
        P = int(self.h["n_pages"][u])
        return self.idx.pool_k[u, :P].float().cpu().numpy(), self.idx.pool_v[u, :P].float().cpu().numpy()


def test_layers_with_next_copy_on_a_second_stream_match_the_oracle():
    w = workloads.WORKLOADS["llama31_8b_16k"].scaled(n_tokens=3000, batch=2, n_q_heads=8, n_kv_heads=2)
    n_layers, budget = 4, 128
    dt = torch.bfloat16
    host = []
    for layer in range(n_layers):
        K, V = workloads.batch_kv(w, layer)
        Q = workloads.batch_queries(w, layer)
        host.append(dict(K=K, V=V, Q=Q, Kh=torch.from_numpy(K).to(dt).pin_memory(),
                         Vh=torch.from_numpy(V).to(dt).pin_memory(), Qh=torch.from_numpy(Q).to(dt).pin_memory()))
    # two device slots for K, V, Q: layer i computes from slot i % 2 while layer i + 1 fills the other
    slots = [{k: torch.empty_like(host[0][k + "h"], device="cuda") for k in ("K", "V", "Q")} for _ in range(2)]
    cfgs = [cfg_of(w, layer=i) for i in range(n_layers)]
    idxs = [ice.Index(c) for c in cfgs]
    bufs = [ice.DecodeBuffers(c, budget) for c in cfgs]
    ws = ice.workspace(ice.ice_build_workspace_bytes(cfgs[0].params()))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(n_layers)]
    done = [torch.cuda.Event() for _ in range(n_layers)]

    def h2d(i):
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(done[i - 2])  # the slot's previous layer has finished with it
            for k in ("K", "V", "Q"):
                slots[i % 2][k].copy_(host[i][k + "h"], non_blocking=True)
            copied[i].record(copy_s)

    scale = 1.0 / np.sqrt(128)
    h2d(0)
    for i in range(n_layers):
        if i + 1 < n_layers:
            h2d(i + 1)  # overlaps layer i's build and decode
        sl, p, b = slots[i % 2], cfgs[i].params(), bufs[i]
        comp_s.wait_event(copied[i])
        ice.ice_build_index(p, sl["K"], sl["V"], idxs[i], ws, err, stream=comp_s)
        ice.ice_decode_step(p, idxs[i], sl["Q"], budget, b.sel_pages, b.sel_count, b.kbuf, b.vbuf, b.buf_len, scale,
                            b.O, b.ws, err, stream=comp_s)
        done[i].record(comp_s)
    torch.cuda.synchronize()
    assert ice.ice_check(err) == ice.ICE_OK
    for i in range(n_layers):
        run = _Layer(w, i, cfgs[i], idxs[i], host[i]["K"], host[i]["V"])
        run.h = host_tables(idxs[i])
        for u in range(cfgs[i].units):
            check_build_unit(run, u)
            check_decode_unit(run, u, host[i]["Q"], budget, bufs[i])
