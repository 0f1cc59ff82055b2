"""The allocation-free attention entry point (ice_sparse_attn_decode_noalloc).

Some callers cannot call cudaMalloc: a plugin inside a serving runtime that
owns all device memory through its own pool, or a decode loop that cannot take
an allocation's implicit synchronisation.  For them the attention step has a
variant that takes no workspace and keeps its scratch in a static device array
of the library.  This test calls it through the C ABI twice in a row and
checks each result against the workspace entry point, within the attention
tolerance the parity tests use; it builds its own inputs, so it passes alone
in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import ATTN_TOL, to_dev

pytestmark = pytest.mark.gpu


def _selected_pages(w, cfg, budget):
    K, V = workloads.batch_kv(w)
    dt = cfg.torch_dtype
    p = cfg.params()
    idx = ice.Index(cfg)
    ws = ice.workspace(ice.ice_build_workspace_bytes(p))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ice.ice_build_index(p, to_dev(K, dt), to_dev(V, dt), idx, ws, err)
    buf = ice.DecodeBuffers(cfg, budget)
    Q = to_dev(workloads.batch_queries(w), dt)
    ice.ice_select_pages(p, idx, Q, budget, buf.sel_pages, buf.sel_count, buf.ws, err)
    ice.ice_gather_pages(p, idx, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf, buf.buf_len)
    assert ice.ice_check(err) == ice.ICE_OK
    return p, buf


def test_noalloc_attention_matches_workspace_entry_point_twice():
    ice.load()
    scale = 1.0 / np.sqrt(128)
    runs = []
    for seed, budget in ((11, 256), (12, 128)):
        w = workloads.WORKLOADS["llama31_8b_16k"].scaled(n_tokens=4000, n_q_heads=16, n_kv_heads=4, seed=seed)
        cfg = ice.Config(batch=1, n_q_heads=16, n_kv_heads=4, n_tokens=4000, seed=seed)
        p, buf = _selected_pages(w, cfg, budget)
        Q = to_dev(workloads.batch_queries(w), cfg.torch_dtype)
        ref = torch.zeros_like(buf.O)
        ice.ice_sparse_attn_decode(p, Q, buf.kbuf, buf.vbuf, buf.buf_len, buf.sel_count, scale, ref, buf.ws)
        runs.append((p, buf, Q, ref))
    # two calls in a row on the shared static scratch, different shapes and inputs
    outs = []
    for p, buf, Q, _ in runs:
        O = torch.full_like(buf.O, float("nan"))
        ice.ice_sparse_attn_decode_noalloc(p, Q, buf.kbuf, buf.vbuf, buf.buf_len, buf.sel_count, scale, O)
        outs.append(O)
    torch.cuda.synchronize()
    for (_, _, _, ref), O in zip(runs, outs):
        assert torch.isfinite(O).all()
        assert torch.max(torch.abs(O - ref)).item() <= ATTN_TOL["bf16"]


def test_noalloc_rejects_shapes_beyond_its_scratch():
    ice.load()
    cfg = ice.Config(batch=64, n_q_heads=1024, n_kv_heads=64, n_tokens=16)
    p = cfg.params()
    t = torch.zeros(16, device="cuda")
    lens = torch.zeros((64 * 64, 4096), dtype=torch.int32, device="cuda")
    with pytest.raises(ice.IceError) as ei:
        ice.ice_sparse_attn_decode_noalloc(p, t, t, t, lens, t, 1.0, t)
    assert ei.value.status == ice.ICE_ERR_CAPACITY
