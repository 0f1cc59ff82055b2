"""GPU parity of the incremental insert (ice_insert_tokens) against the
oracle's insert, step by step, starting both from the same built index.
After every step the device's parent of each new token is compared with the
oracle's nearest parent; a difference must be an fp32 near-tie of the lifted
distance (and rare), and the oracle then continues from the device's choice,
so every unit is checked to the end."""
import numpy as np
import pytest
import torch

import oracle
import semantic_paged_kv_gb300 as ice
import workloads
from parity_util import DeviceRun, TIE_REL, check_build_unit, check_decode_unit, host_tables, to_dev

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS


def _oracle_state(run, u):
    """An oracle UnitIndex holding exactly the GPU's built index of unit u."""
    b, h = run.unit(u)
    H = run.h
    K = run.K[b, h].astype(np.float64)
    _, M2, e = oracle.lift(K)
    Np, P = int(H["n_parents"][u]), int(H["n_pages"][u])
    pk, pv = run.pool(u)
    idx = {"S": run.cfg.page_size, "M2": M2, "parent_tok": H["parent_tok"][u, :Np],
           "parent_keys": K[H["parent_tok"][u, :Np]], "parent_e": e[H["parent_tok"][u, :Np]], "n_pages": P,
           "page_parent": H["page_parent"][u, :P], "page_len": H["page_len"][u, :P],
           "page_tokens": H["page_tokens"][u, :P], "pool_k": pk, "pool_v": pv,
           "token_parent": H["token_parent"][u, :run.cfg.n_tokens], "token_page": H["token_page"][u, :run.cfg.n_tokens],
           "token_slot": H["token_slot"][u, :run.cfg.n_tokens]}
    return oracle.UnitIndex(idx, run.cfg.head_dim, np_cap=run.cfg.np_cap, page_cap=run.cfg.page_cap,
                            n_cap=run.cfg.n_cap)


def _run_inserts(w, steps, sample_tokens=None, **cfg_kw):
    """Build, check the build (assignment on sample_tokens tokens when set),
    then insert `steps` tokens per unit, checking every step."""
    N = w.n_tokens
    run = DeviceRun(w, n_cap=N + steps, **cfg_kw)
    assert run.status == ice.ICE_OK
    cfg, U = run.cfg, run.cfg.units
    for u in range(U):
        check_build_unit(run, u, sample_tokens=sample_tokens)
    new = [workloads.unit_new_tokens(w, 0, *run.unit(u), steps) for u in range(U)]
    ora = [_oracle_state(run, u) for u in range(U)]
    ws = ice.workspace(ice.ice_insert_workspace_bytes(run.params))
    th = oracle.promote_threshold(w.promote_p)
    dt = cfg.torch_dtype
    ties = 0
    for s in range(steps):
        kn = np.stack([new[u][0][s] for u in range(U)]).reshape(cfg.batch, cfg.n_kv_heads, 128)
        vn = np.stack([new[u][1][s] for u in range(U)]).reshape(cfg.batch, cfg.n_kv_heads, 128)
        ice.ice_insert_tokens(run.params, run.idx, to_dev(kn, dt), to_dev(vn, dt), ws, run.err)
        tp_dev = run.idx.token_parent[:, N + s].cpu().numpy()
        for u in range(U):
            b, h = run.unit(u)
            o, k = ora[u], new[u][0][s].astype(np.float64)
            Np = o.n_parents.value
            promoted = oracle.promote_draw(w.seed, 0, b, h, N + s) < th or Np == 0
            parent = -1
            if not promoted:
                # the oracle's nearest parent (its assignment step over the current parents, the
                # build-time M^2), and the device's choice checked against it
                e = np.sqrt(max(o.M2 - k @ k, 0.0))
                best = int(oracle.assign(np.vstack([o.parent_keys[:Np], k]), np.append(o.parent_e[:Np], e),
                                         np.arange(Np))[-1])
                parent = int(tp_dev[u])
                if parent != best:
                    assert 0 <= parent < Np, (u, s, parent)
                    d = lambda m: float(((k - o.parent_keys[m]) ** 2).sum() + (e - o.parent_e[m]) ** 2)
                    assert d(parent) - d(best) <= 2 * TIE_REL * o.M2, (u, s, parent, best)
                    ties += 1
            o.insert(new[u][0][s], new[u][1][s], N + s, seed=w.seed, layer=0, seq=b, head=h, thresh=th, parent=parent)
            assert int(tp_dev[u]) == int(o.token_parent[N + s]), (u, s, "promotion")
    assert ties <= max(2, U * steps // 2000), ties
    assert ice.ice_check(run.err) == ice.ICE_OK
    for u in range(U):
        o = ora[u]
        Np, P = o.n_parents.value, o.n_pages.value
        get = lambda f: getattr(run.idx, f)[u].cpu().numpy()
        assert np.array_equal(get("token_parent")[:N + steps], o.token_parent[:N + steps])
        assert int(run.idx.n_parents[u]) == Np and int(run.idx.n_pages[u]) == P
        assert int(run.idx.n_indexed[u]) == N + steps
        assert np.array_equal(get("parent_tok")[:Np], o.parent_tok[:Np])
        assert np.array_equal(get("page_parent")[:P], o.page_parent[:P])
        assert np.array_equal(get("page_len")[:P], o.page_len[:P])
        assert np.array_equal(get("page_tokens")[:P], o.page_tokens[:P])
        assert np.array_equal(get("token_page")[:N + steps], o.token_page[:N + steps])
        assert np.array_equal(get("token_slot")[:N + steps], o.token_slot[:N + steps])
        assert np.array_equal(run.idx.pool_k[u, :P].float().cpu().numpy(), o.pool_k[:P])
        assert np.array_equal(run.idx.pool_v[u, :P].float().cpu().numpy(), o.pool_v[:P])
        assert np.array_equal(run.idx.parent_keys[u, :Np].float().cpu().numpy(), o.parent_keys[:Np])
        # page chains: every parent's pages in ascending id, linked first -> last
        pp = o.page_parent[:P]
        nxt = get("page_next")
        for m in range(Np):
            pages = np.nonzero(pp == m)[0]
            assert get("parent_first_page")[m] == pages[0] and get("parent_last_page")[m] == pages[-1]
            assert get("parent_n_pages")[m] == len(pages)
            assert [nxt[a] for a in pages] == list(pages[1:]) + [-1]
    # the keys and values of every indexed position, for checks after the inserts
    kn = np.stack([new[u][0] for u in range(U)]).reshape(cfg.batch, cfg.n_kv_heads, steps, 128)
    vn = np.stack([new[u][1] for u in range(U)]).reshape(cfg.batch, cfg.n_kv_heads, steps, 128)
    run.K = np.concatenate([run.K, kn], axis=2)
    run.V = np.concatenate([run.V, vn], axis=2)
    return run


def test_insert_stream_mistral_shaped():
    """Mistral-7B head layout (g = 4), bf16, 48 inserted tokens per unit."""
    w = W["mistral_7b_36k"].scaled(n_tokens=5000, n_q_heads=8, n_kv_heads=2, centres=256)
    run = _run_inserts(w, 48)
    # decode after the inserts sees the updated index
    run.h = host_tables(run.idx)
    Q, buf, st = run.decode(256)
    assert st == ice.ICE_OK
    for u in range(run.cfg.units):
        check_decode_unit(run, u, Q, 256, buf)


def test_insert_stream_mistral_full_size():
    """The Mistral-7B-shaped layer at its full size (32/8 heads, N = 36864)
    with the 128 decode-step inserts the benchmark times, one
    ice_insert_tokens call per step for all 8 units: every unit's tables,
    pool and page chains against the oracle's insert started from the same
    built index, then the decode over the grown index on every unit."""
    w = W["mistral_7b_36k"]
    run = _run_inserts(w, 128, sample_tokens=1500)
    assert int(run.idx.n_indexed.sum()) == run.cfg.units * (w.n_tokens + 128)
    run.h = host_tables(run.idx)
    Q, buf, st = run.decode(256)
    assert st == ice.ICE_OK
    for u in range(run.cfg.units):
        check_decode_unit(run, u, Q, 256, buf)


def test_insert_single_parent_splits_full_page_at_17():
    """p = 0: one parent, sequential pages; the last page (8 tokens) fills,
    and the 17th token of that page opens a new page linked after it."""
    w = W["tiny"].scaled(n_tokens=1000, promote_p=0.0)
    run = _run_inserts(w, 20)
    assert int(run.idx.n_pages[0]) == 64
    assert run.idx.page_len[0, 62].item() == 16 and run.idx.page_len[0, 63].item() == 12
    assert run.idx.page_next[0, 62].item() == 63


def test_insert_every_token_promoted():
    """p = 1: every inserted token becomes a parent with a one-token page."""
    w = W["tiny"].scaled(n_tokens=300, promote_p=1.0)
    run = _run_inserts(w, 10)
    assert int(run.idx.n_parents[0]) == 310 and int(run.idx.n_pages[0]) == 310


def test_insert_capacity_error():
    w = W["tiny"].scaled(n_tokens=100)
    run = DeviceRun(w, n_cap=100)
    ws = ice.workspace(ice.ice_insert_workspace_bytes(run.params))
    kn = torch.zeros((1, 1, 128), device="cuda")
    ice.ice_insert_tokens(run.params, run.idx, kn, kn, ws, run.err)
    assert ice.ice_check(run.err) == ice.ICE_ERR_CAPACITY
    assert int(run.idx.n_indexed[0]) == 100
