"""Pins for the CPU oracle against facts fixed outside it.

Each test checks the oracle against something it cannot agree with by
construction: the published splitmix64 outputs, hand-derived worked examples
(tests/golden), closed forms of the key lift, textbook special cases (one
parent gives sequential paging, p = 1 gives exact top-k inner-product search,
full budget gives dense softmax attention, computed by torch's SDPA), brute
force over subsets on tiny inputs, and statistical properties of the random
promotion.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ promotion draw
def test_splitmix64_published_vectors():
    g = _load("splitmix64_vectors.json")
    s0 = g["streams"][0]
    for n, h in enumerate(s0["outputs_hex"], start=1):
        assert oracle.splitmix64_nth(s0["seed"], n) == int(h, 16)
    s1 = g["streams"][1]
    for n, v in enumerate(s1["outputs_dec"], start=1):
        assert oracle.splitmix64_nth(s1["seed"], n) == int(v)


def test_promote_draw_is_the_stated_stream_composition():
    for seed, layer, seq, head, tok, lvl in [(0, 0, 0, 0, 0, 1), (7, 3, 2, 5, 12345, 1), (2**40 + 3, 31, 15, 63, 99999, 2)]:
        key = oracle.splitmix64_nth(seed, layer + 1)
        ctr = tok | (lvl << 32) | (head << 40) | (seq << 52)
        assert oracle.promote_draw(seed, layer, seq, head, tok, lvl) == oracle.splitmix64_nth(key, ctr + 1) >> 32


@pytest.mark.parametrize("p", [1 / 16, 1 / 4, 1 / 2])
def test_promotion_count_is_binomial(p):
    N = 20000
    th = oracle.promote_threshold(p)
    for head in range(3):
        n = len(oracle.promote(11, 2, 0, head, N, th))
        mu, sd = N * p, math.sqrt(N * p * (1 - p))
        assert abs(n - mu) < 5 * sd


def test_promotion_depends_on_every_key_field_and_is_deterministic():
    th = oracle.promote_threshold(1 / 16)
    base = oracle.promote(5, 1, 2, 3, 4096, th)
    assert np.array_equal(base, oracle.promote(5, 1, 2, 3, 4096, th))
    for args in [(6, 1, 2, 3), (5, 2, 2, 3), (5, 1, 3, 3), (5, 1, 2, 4)]:
        other = oracle.promote(*args, 4096, th)
        assert not np.array_equal(base, other)
    assert np.all(np.diff(base) > 0)  # ascending token order


def test_promotion_extremes():
    assert np.array_equal(oracle.promote(0, 0, 0, 0, 100, oracle.promote_threshold(1.0)), np.arange(100))
    only = oracle.promote(0, 0, 0, 0, 100, 0)
    draws = [oracle.promote_draw(0, 0, 0, 0, j, 1) for j in range(100)]
    assert list(only) == [int(np.argmin(draws))]
    assert len(oracle.promote(0, 0, 0, 0, 0, 0)) == 0


# ---------------------------------------------------------------- the lift
def test_handworked_lift_assign_pack_select():
    g = _load("handworked_d2.json")
    K = np.array(g["keys"], float)
    n, M2, e = oracle.lift(K)
    assert np.allclose(n, g["lift"]["norm2"], rtol=0, atol=0)
    assert M2 == g["lift"]["M2"]
    assert np.allclose(e, g["lift"]["e"], rtol=1e-15, atol=0)
    tp = oracle.assign(K, e, g["parent_tok"])
    assert tp.tolist() == g["token_parent"]
    pk = oracle.pack(tp, len(g["parent_tok"]), g["page_size"])
    for key in ("page_parent", "page_len", "page_tokens", "token_page", "token_slot"):
        assert np.asarray(pk[key]).tolist() == g["pages"][key], key
    pkeys = K[g["parent_tok"]]
    for case in g["select"]:
        head, union = oracle.select(np.array(case["q"], float), pkeys, pk["page_parent"], case["k_pages"])
        assert head.tolist() == case["head_pages"]
        assert union.tolist() == case["union"]


def test_lift_closed_form_all_lifted_norms_equal_M():
    w = workloads.WORKLOADS["tiny"]
    K, _ = workloads.unit_kv(w, 0, 0, 0, 512)
    n, M2, e = oracle.lift(K)
    Kd = K.astype(np.float64)
    lifted = np.concatenate([Kd, e[:, None]], axis=1)
    assert np.allclose(np.linalg.norm(lifted, axis=1), math.sqrt(M2), rtol=1e-14)
    assert e.min() == 0.0 and np.isclose(M2, (Kd * Kd).sum(1).max(), rtol=1e-15)


def _mixture_unit(seed, N, d, centres=8, spread=0.3, lognormal=0.0):
    r = np.random.default_rng(seed)
    C = r.standard_normal((centres, d))
    K = C[r.integers(0, centres, N)] + spread * r.standard_normal((N, d))
    if lognormal:
        K *= np.exp(lognormal * r.standard_normal((N, 1)))
    return workloads.round_bf16(K.astype(np.float32)).astype(np.float64)


@pytest.mark.parametrize("d,p,lognormal", [(4, 1 / 4, 0.0), (8, 1 / 16, 0.5), (128, 1 / 16, 0.0), (128, 1 / 4, 0.5)])
def test_assign_equals_max_lifted_inner_product(d, p, lognormal):
    """argmin of the lifted distance (oracle) == argmax of the lifted inner
    product computed by a matrix product (|k'| = |p'| = M makes them equal)."""
    K = _mixture_unit(int(d * 1000 + p * 64), 384, d, lognormal=lognormal)
    n, M2, e = oracle.lift(K)
    pt = oracle.promote(3, 0, 0, d, len(K), oracle.promote_threshold(p))
    tp = oracle.assign(K, e, pt)
    lifted = np.concatenate([K, e[:, None]], 1)
    ip = lifted @ lifted[pt].T
    expect = np.argmax(ip, axis=1)
    expect[pt] = np.arange(len(pt))
    # accept only exact agreement or a near-tie of the inner product
    best = ip[np.arange(len(K)), expect]
    got = ip[np.arange(len(K)), tp]
    assert np.all((tp == expect) | (best - got <= 1e-9 * M2))
    assert (tp == expect).mean() > 0.99


def test_assign_nearest_promoted_point_brute_force():
    K = _mixture_unit(77, 64, 4)
    n, M2, e = oracle.lift(K)
    pt = oracle.promote(1, 0, 0, 0, len(K), oracle.promote_threshold(1 / 4))
    tp = oracle.assign(K, e, pt)
    for j in range(len(K)):
        if j in set(pt.tolist()):
            assert pt[tp[j]] == j
            continue
        dists = [np.linalg.norm(np.append(K[j], e[j]) - np.append(K[t], e[t])) for t in pt]
        assert tp[j] == int(np.argmin(dists))


# -------------------------------------------------------------- packing
def _check_pack_invariants(tp, Np, S, pk):
    N = len(tp)
    P = pk["n_pages"]
    seen = np.zeros(N, int)
    counts = np.bincount(tp, minlength=Np)
    for p in range(P):
        L = pk["page_len"][p]
        assert 1 <= L <= S
        toks = pk["page_tokens"][p]
        assert np.all(toks[L:] == -1) and np.all(toks[:L] >= 0)
        assert np.all(tp[toks[:L]] == pk["page_parent"][p])  # one parent per page
        assert np.all(np.diff(toks[:L]) > 0)
        seen[toks[:L]] += 1
        for s, j in enumerate(toks[:L]):
            assert pk["token_page"][j] == p and pk["token_slot"][j] == s
    assert np.all(seen == 1)  # every token in exactly one page
    pages_per_parent = np.bincount(pk["page_parent"], minlength=Np)
    assert np.array_equal(pages_per_parent, -(-counts // S))
    assert P <= Np + -(-N // S)
    assert np.all(np.diff(pk["page_parent"]) >= 0)


@pytest.mark.parametrize("seed", range(4))
def test_pack_invariants_random(seed):
    r = np.random.default_rng(seed)
    N, Np, S = int(r.integers(1, 3000)), int(r.integers(1, 200)), 16
    tp = r.integers(0, Np, N).astype(np.int32)
    tp[:Np] = np.arange(Np)  # every parent owns its own token at least
    pk = oracle.pack(tp, Np, S)
    _check_pack_invariants(tp, Np, S, pk)


def test_pack_single_parent_is_sequential_paging():
    """With exactly one parent the pages are the classic sequential paging:
    page i holds tokens 16i .. 16i+15 (papernotes 关键设计 1 / article section 二)."""
    N, S = 1000, 16
    pk = oracle.pack(np.zeros(N, np.int32), 1, S)
    assert pk["n_pages"] == -(-N // S)
    for p in range(pk["n_pages"]):
        toks = pk["page_tokens"][p]
        want = np.arange(p * S, min((p + 1) * S, N))
        assert np.array_equal(toks[: len(want)], want)
    assert np.array_equal(pk["token_page"], np.arange(N) // S)


def test_pack_capacity_error():
    with pytest.raises(RuntimeError):
        oracle.pack(np.zeros(40, np.int32), 1, 16, page_cap=2)


# ------------------------------------------------------------- selection
def test_select_p1_is_exact_topk_mips():
    """p = 1: every token is its own parent with a one-token page, so page
    selection is exact top-k maximum inner product search (torch.topk)."""
    w = workloads.WORKLOADS["tiny"]
    K, V = workloads.unit_kv(w, 0, 0, 0, 300)
    q = workloads.unit_queries(w, 0, 0, 0)
    idx = oracle.build_unit(K, V, seed=0, layer=0, seq=0, head=0, thresh=oracle.promote_threshold(1.0))
    assert idx["n_pages"] == len(K) and np.all(idx["page_len"] == 1)
    assert np.array_equal(idx["page_tokens"][:, 0], np.arange(len(K)))
    k = 10
    head, union = oracle.select(q, idx["parent_keys"], idx["page_parent"], k)
    scores = torch.tensor(q, dtype=torch.float64) @ torch.tensor(K, dtype=torch.float64).T
    top = torch.topk(scores, k, dim=1).indices.numpy()
    for h in range(q.shape[0]):
        assert set(head[h].tolist()) == set(top[h].tolist())
    assert union.tolist() == sorted(set(top.reshape(-1).tolist()))


def test_select_brute_force_subsets():
    """On tiny inputs, the chosen set is the unique k-subset whose every
    member precedes every non-member in the (-score, page id) order."""
    r = np.random.default_rng(5)
    for trial in range(20):
        Np, d = int(r.integers(1, 6)), 3
        tp = r.integers(0, Np, 30).astype(np.int32)
        tp[:Np] = np.arange(Np)
        pk = oracle.pack(tp, Np, 4)
        keys = np.round(r.standard_normal((Np, d)), 1)  # coarse values: ties happen
        q = np.round(r.standard_normal((1, d)), 1)
        P = pk["n_pages"]
        s = keys @ q[0]
        k = int(r.integers(1, P + 1))
        head, union = oracle.select(q, keys, pk["page_parent"], k)
        ok = []
        for T in itertools.combinations(range(P), k):
            Tset = set(T)
            good = all((-s[pk["page_parent"][a]], a) < (-s[pk["page_parent"][b]], b)
                       for a in Tset for b in range(P) if b not in Tset)
            if good:
                ok.append(Tset)
        assert len(ok) == 1
        assert set(head[0].tolist()) == ok[0] and union.tolist() == sorted(ok[0])


def test_select_union_g1_identity_and_k_ge_P():
    w = workloads.WORKLOADS["tiny"]
    K, V = workloads.unit_kv(w, 0, 0, 0, 500)
    idx = oracle.build_unit(K, V, seed=0, layer=0, seq=0, head=0, thresh=oracle.promote_threshold(1 / 16))
    q = workloads.unit_queries(w, 0, 0, 0)
    head, union = oracle.select(q[:1], idx["parent_keys"], idx["page_parent"], 4)
    assert union.tolist() == sorted(head[0].tolist())
    head, union = oracle.select(q, idx["parent_keys"], idx["page_parent"], idx["n_pages"] + 5)
    assert union.tolist() == list(range(idx["n_pages"]))


# ------------------------------------------------------------- attention
def test_attention_handworked():
    g = _load("attention_d2.json")
    a = math.sqrt(2.0) * math.log(2.0)
    kb = np.array([[[0, 0], [a, 0]], [[-a, 0], [50, 0]]], float)
    vb = np.array(g["values"], float)
    out = oracle.attention(np.array(g["q"], float), kb, vb, g["buf_len"])
    assert np.allclose(out, g["out"], rtol=0, atol=1e-13)


def test_full_budget_equals_dense_sdpa():
    """Full budget selects every page, and the masked sparse attention over
    the gathered pages equals dense softmax attention over all N tokens
    (torch.nn.functional.scaled_dot_product_attention, float64)."""
    w = workloads.WORKLOADS["tiny"].scaled(n_tokens=700)
    K, V = workloads.unit_kv(w, 0, 0, 0)
    q = workloads.unit_queries(w, 0, 0, 0)
    idx = oracle.build_unit(K, V, seed=0, layer=0, seq=0, head=0, thresh=oracle.promote_threshold(1 / 16))
    res = oracle.decode_unit(idx, q, budget_tokens=16 * idx["n_pages"])
    assert res["sel_pages"].tolist() == list(range(idx["n_pages"]))
    t = lambda x: torch.tensor(x, dtype=torch.float64)
    dense = torch.nn.functional.scaled_dot_product_attention(t(q)[None, :, None, :], t(K)[None, None].expand(1, q.shape[0], -1, -1),
                                                             t(V)[None, None].expand(1, q.shape[0], -1, -1))
    assert np.allclose(res["out"], dense[0, :, 0].numpy(), rtol=0, atol=1e-12)


def test_attention_subset_equals_sdpa_on_selected_tokens():
    w = workloads.WORKLOADS["tiny"].scaled(n_tokens=900)
    K, V = workloads.unit_kv(w, 0, 0, 0)
    q = workloads.unit_queries(w, 0, 0, 0)
    idx = oracle.build_unit(K, V, seed=0, layer=0, seq=0, head=0, thresh=oracle.promote_threshold(1 / 16))
    res = oracle.decode_unit(idx, q, budget_tokens=64)
    toks = idx["page_tokens"][res["sel_pages"]].reshape(-1)
    toks = toks[toks >= 0]
    t = lambda x: torch.tensor(x, dtype=torch.float64)
    Ks, Vs = t(K[toks]), t(V[toks])
    dense = torch.nn.functional.scaled_dot_product_attention(t(q)[None, :, None, :], Ks[None, None].expand(1, q.shape[0], -1, -1),
                                                             Vs[None, None].expand(1, q.shape[0], -1, -1))
    assert np.allclose(res["out"], dense[0, :, 0].numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- insert
def _unit_invariants(ui):
    d = ui.as_dict()
    P, S = d["n_pages"], d["S"]
    N = int((ui.token_parent >= 0).sum())
    for p in range(P):
        L = d["page_len"][p]
        assert 1 <= L <= S
        toks = d["page_tokens"][p][:L]
        assert np.all(ui.token_parent[toks] == d["page_parent"][p])
        assert np.all(ui.token_page[toks] == p) and np.array_equal(ui.token_slot[toks], np.arange(L))
    assert d["page_len"].sum() == N


def test_insert_p1_creates_one_token_pages():
    w = workloads.WORKLOADS["tiny"]
    K, V = workloads.unit_kv(w, 0, 0, 0, 64)
    th = oracle.promote_threshold(1.0)
    idx = oracle.build_unit(K, V, seed=0, layer=0, seq=0, head=0, thresh=th)
    ui = oracle.UnitIndex(idx, 128, np_cap=80, page_cap=80, n_cap=80)
    Kn, Vn = workloads.unit_new_tokens(w, 0, 0, 0, 8)
    for s in range(8):
        ui.insert(Kn[s], Vn[s], 64 + s, seed=0, layer=0, seq=0, head=0, thresh=th)
        assert ui.n_parents.value == 65 + s and ui.n_pages.value == 65 + s
        assert ui.page_len[64 + s] == 1 and ui.page_tokens[64 + s, 0] == 64 + s
    _unit_invariants(ui)


def test_exact_ties_take_the_lowest_parent():
    """Exact ties of the lifted distance go to the lowest parent index m, in
    the build's assignment and in the insert; a promoted token is its own
    parent even when an earlier parent has the same key (distance 0 too).
    Integer coordinates keep every distance exact in double."""
    # parents: tokens 0 (0, 5) and 1 (5, 0); M^2 = 25, e = 0 for both
    K = np.array([[0, 5], [5, 0], [3, 3], [0, 5], [5, 0]], float)
    n, M2, e = oracle.lift(K)
    assert M2 == 25 and e[0] == 0 and e[1] == 0
    # token 2: |(3,3) - (0,5)|^2 = 9 + 4 = 13 = |(3,3) - (5,0)|^2, same e gap -> m = 0
    assert oracle.assign(K, e, [0, 1]).tolist() == [0, 1, 0, 0, 1]
    # parents with equal keys (tokens 1 and 4): each its own parent; token 2 ties three ways -> m = 0
    assert oracle.assign(K, e, [1, 3, 4]).tolist() == [1, 0, 0, 1, 2]
    # insert: k = (0.5, 0.5, 0, 0) is at lifted distance 1 from both unit parents -> m = 0
    d, S = 4, 16
    P2 = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    idx = {"S": S, "M2": 1.0, "parent_tok": np.array([0, 1]), "parent_keys": P2, "parent_e": np.zeros(2),
           "n_pages": 2, "page_parent": np.array([0, 1]), "page_len": np.array([1, 1]),
           "page_tokens": np.array([[0] + [-1] * 15, [1] + [-1] * 15]), "pool_k": np.zeros((2, S, d)),
           "pool_v": np.zeros((2, S, d)), "token_parent": np.array([0, 1]), "token_page": np.array([0, 1]),
           "token_slot": np.array([0, 0])}
    ui = oracle.UnitIndex(idx, d, np_cap=4, page_cap=8, n_cap=8)
    ui.insert(np.array([0.5, 0.5, 0, 0]), np.ones(d), 2, seed=0, layer=0, seq=0, head=0, thresh=0)
    assert ui.token_parent[2] == 0 and ui.page_len[:2].tolist() == [2, 1]


def test_insert_attaches_to_nearest_parent_and_splits_at_17():
    """Keys equal to parent 0's key attach to parent 0 (distance 0); once its
    last page holds 16 tokens the 17th opens a new page."""
    d, S = 4, 16
    K = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    V = np.zeros_like(K)
    idx = {"S": S, "M2": 1.0, "parent_tok": np.array([0, 1]), "parent_keys": K, "parent_e": np.zeros(2),
           "n_pages": 2, "page_parent": np.array([0, 1]), "page_len": np.array([1, 1]),
           "page_tokens": np.array([[0] + [-1] * 15, [1] + [-1] * 15]), "pool_k": np.zeros((2, S, d)),
           "pool_v": np.zeros((2, S, d)), "token_parent": np.array([0, 1]), "token_page": np.array([0, 1]),
           "token_slot": np.array([0, 0])}
    ui = oracle.UnitIndex(idx, d, np_cap=4, page_cap=8, n_cap=64)
    pos = 2
    for _ in range(40):
        ui.insert(K[0], np.ones(d), pos, seed=0, layer=0, seq=0, head=0, thresh=0)  # thresh 0: never promoted
        pos += 1
    assert ui.n_pages.value == 4  # page 0 filled to 16, then pages 2 and 3
    assert ui.page_len[:4].tolist() == [16, 1, 16, 9]
    assert ui.page_parent[:4].tolist() == [0, 1, 0, 0]
    _unit_invariants(ui)


def test_insert_stream_keeps_invariants_and_matches_rebuild_when_nothing_promotes():
    """With promotion switched off for the new tokens, inserting tokens one by
    one attaches each to its nearest parent exactly as a build over all the
    tokens with the same parents and the same M would (the page layout then
    differs only in page numbering, so compare the parent of every token)."""
    w = workloads.WORKLOADS["tiny"]
    K, V = workloads.unit_kv(w, 0, 0, 0, 400)
    th = oracle.promote_threshold(1 / 16)
    idx = oracle.build_unit(K, V, seed=0, layer=0, seq=0, head=0, thresh=th)
    Kn, Vn = workloads.unit_new_tokens(w, 0, 0, 0, 50)
    Kn = Kn * 0.5  # keep |k| < M so that the extra coordinate never clamps
    ui = oracle.UnitIndex(idx, 128, np_cap=100, page_cap=200, n_cap=450)
    for s in range(50):
        ui.insert(Kn[s], Vn[s], 400 + s, seed=0, layer=0, seq=0, head=0, thresh=0)
    _unit_invariants(ui)
    Kall = np.concatenate([K, Kn]).astype(np.float64)
    n = (Kall ** 2).sum(1)
    e = np.sqrt(np.maximum(idx["M2"] - n, 0))
    tp = oracle.assign(Kall, e, idx["parent_tok"])
    assert np.array_equal(ui.token_parent[:450], tp)


# ------------------------------------------------------- inter-layer reuse
def _reuse_pair(n_tokens=1500, centres=24):
    w = workloads.WORKLOADS["llama31_8b_16k"].scaled(n_tokens=n_tokens, centres=centres, dtype="fp32")
    th = oracle.promote_threshold(w.promote_p)
    K0, V0 = workloads.unit_kv(w, 0, 0, 1)
    K1, V1 = workloads.unit_kv(w, 1, 0, 1)
    prev = oracle.build_unit(K0, V0, seed=w.seed, layer=0, seq=0, head=1, thresh=th)
    return w, th, (K0, V0), (K1, V1), prev


def test_reuse_of_own_index_is_the_full_build():
    """Reusing a unit's own node structure on its own keys reproduces the full
    build (lift, promotion, nearest-parent assignment, pack, scatter)."""
    w, th, (K0, V0), _, prev = _reuse_pair()
    r = oracle.build_unit_reuse(K0, V0, prev)
    for f in ("parent_tok", "token_parent", "page_parent", "page_len", "page_tokens", "token_page", "token_slot",
              "parent_keys", "parent_e", "pool_k", "pool_v", "e"):
        assert np.array_equal(np.asarray(r[f]), np.asarray(prev[f])), f
    assert r["M2"] == prev["M2"] and r["n_pages"] == prev["n_pages"]


def test_reuse_on_another_layer_keeps_pages_and_takes_this_layers_keys():
    w, th, _, (K1, V1), prev = _reuse_pair()
    r = oracle.build_unit_reuse(K1, V1, prev)
    for f in ("parent_tok", "token_parent", "page_parent", "page_len", "page_tokens", "token_page", "token_slot"):
        assert np.array_equal(np.asarray(r[f]), np.asarray(prev[f])), f
    K = K1.astype(np.float64)
    n2 = np.einsum("ij,ij->i", K, K)
    assert abs(r["M2"] - n2.max()) <= 1e-14 * n2.max()  # summation order only
    assert np.array_equal(r["parent_keys"], K[prev["parent_tok"]])
    # closed form of the lift: every lifted parent has norm M
    pe = np.asarray(r["parent_e"])
    assert np.allclose(n2[prev["parent_tok"]] + pe ** 2, r["M2"], rtol=1e-12, atol=1e-9)
    # the pool holds this layer's rows in the kept pages, zero pads
    for p in range(r["n_pages"]):
        for s in range(16):
            t = r["page_tokens"][p][s]
            want = K1[t] if t >= 0 else np.zeros(K1.shape[1])
            assert np.array_equal(r["pool_k"][p][s], want)
    _check_pack_invariants(r["token_parent"], len(r["parent_tok"]), 16, r)


def test_reuse_full_budget_is_dense_attention_of_this_layer():
    """With every page selected, decode over the reused index is dense softmax
    attention over all N tokens of the new layer (torch SDPA, float64)."""
    w, th, _, (K1, V1), prev = _reuse_pair(n_tokens=700)
    r = oracle.build_unit_reuse(K1, V1, prev)
    q = workloads.unit_queries(w, 1, 0, 1)
    dec = oracle.decode_unit(r, q, budget_tokens=16 * r["n_pages"])
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    kt = torch.from_numpy(K1.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(V1.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    assert np.max(np.abs(dec["out"] - ref)) < 1e-12


# ------------------------------------------------- sink and window pages
def _pos_unit(N=900, n_sink=40, n_window=70, seed_layer=0, **kw):
    w = workloads.WORKLOADS["llama31_8b_16k"].scaled(n_tokens=N, centres=24, dtype="fp32", **kw)
    th = oracle.promote_threshold(w.promote_p)
    K, V = workloads.unit_kv(w, seed_layer, 0, 0)
    idx = oracle.build_unit_positional(K, V, seed=w.seed, layer=seed_layer, seq=0, head=0, thresh=th,
                                       n_sink=n_sink, n_window=n_window)
    return w, th, K, V, idx


def test_positional_build_without_sink_or_window_is_the_plain_build():
    w, th, K, V, idx = _pos_unit(n_sink=0, n_window=0)
    ref = oracle.build_unit(K, V, seed=w.seed, layer=0, seq=0, head=0, thresh=th)
    for f in ("parent_tok", "token_parent", "page_parent", "page_len", "page_tokens", "token_page", "token_slot",
              "parent_keys", "pool_k", "pool_v"):
        assert np.array_equal(np.asarray(idx[f]), np.asarray(ref[f])), f
    assert idx["n_pages"] == ref["n_pages"] and idx["n_pos"] == 0 and idx["M2"] == ref["M2"]


@pytest.mark.parametrize("n_sink,n_window", [(40, 70), (16, 0), (0, 33), (5, 1)])
def test_positional_pages_are_sequential_and_the_middle_is_indexed(n_sink, n_window):
    N, S = 900, 16
    w, th, K, V, idx = _pos_unit(N=N, n_sink=n_sink, n_window=n_window)
    se, ws = n_sink, N - n_window
    P, n_pos = idx["n_pages"], idx["n_pos"]
    assert n_pos == -(-n_sink // S) + -(-n_window // S)
    P_sem = P - n_pos
    # positional pages: textbook sequential paging of the sink, then of the window
    want = [np.arange(a, min(a + S, se)) for a in range(0, se, S)] + [np.arange(a, min(a + S, N)) for a in range(ws, N, S)]
    for i, toks in enumerate(want):
        p = P_sem + i
        assert idx["page_parent"][p] == -1 and idx["page_len"][p] == len(toks)
        assert np.array_equal(idx["page_tokens"][p][: len(toks)], toks) and np.all(idx["page_tokens"][p][len(toks):] == -1)
    # promotion: exactly the middle tokens the plain promotion over all N picks
    full = oracle.promote(w.seed, 0, 0, 0, N, th)
    mid = full[(full >= se) & (full < ws)]
    if len(mid):
        assert np.array_equal(idx["parent_tok"], mid)
    # M is the middle's largest norm; every middle token's parent is its nearest promoted point
    Km = K[se:ws].astype(np.float64)
    assert abs(idx["M2"] - np.einsum("ij,ij->i", Km, Km).max()) <= 1e-14 * idx["M2"]
    assert np.all(idx["token_parent"][:se] == -2) and np.all(idx["token_parent"][ws:] == -2)
    tp = idx["token_parent"][se:ws]
    pk = K[idx["parent_tok"]].astype(np.float64)
    M2 = idx["M2"]
    e_m = np.sqrt(np.maximum(0.0, M2 - np.einsum("ij,ij->i", Km, Km)))
    e_p = np.sqrt(np.maximum(0.0, M2 - np.einsum("ij,ij->i", pk, pk)))
    d2 = ((Km[:, None, :] - pk[None, :, :]) ** 2).sum(-1) + (e_m[:, None] - e_p[None, :]) ** 2
    best = d2.min(1)
    assert np.all(d2[np.arange(len(tp)), tp] <= best + 1e-9 * M2)
    # every token in exactly one page
    seen = np.zeros(N, int)
    for p in range(P):
        for sl, t in enumerate(idx["page_tokens"][p]):
            if t >= 0:
                seen[t] += 1
                assert idx["token_page"][t] == p and idx["token_slot"][t] == sl
    assert np.all(seen == 1)
    assert np.all(idx["page_parent"][:P_sem] >= 0)


@pytest.mark.parametrize("n_sink,n_window", [(40, 70), (900, 0), (500, 500)])
def test_positional_full_budget_is_dense_attention(n_sink, n_window):
    """Every page selected (or no middle at all): dense softmax attention over
    all N tokens (torch SDPA, float64)."""
    w, th, K, V, idx = _pos_unit(N=900, n_sink=n_sink, n_window=n_window)
    q = workloads.unit_queries(w, 0, 0, 0)
    dec = oracle.decode_unit(idx, q, budget_tokens=16 * max(1, idx["n_pages"]))
    assert len(dec["sel_pages"]) == idx["n_pages"]
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    kt = torch.from_numpy(K.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(V.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    assert np.max(np.abs(dec["out"] - ref)) < 1e-12


def test_positional_small_budget_attends_sink_window_and_selected_pages():
    """A small budget: the union is the selected middle pages plus every
    sink and window page, and attention equals SDPA over exactly those tokens."""
    w, th, K, V, idx = _pos_unit(N=900, n_sink=20, n_window=50)
    q = workloads.unit_queries(w, 0, 0, 0)
    dec = oracle.decode_unit(idx, q, budget_tokens=32)
    P, n_pos = idx["n_pages"], idx["n_pos"]
    sel = dec["sel_pages"]
    assert np.all(np.diff(sel) > 0) and set(range(P - n_pos, P)) <= set(sel.tolist())
    toks = np.concatenate([idx["page_tokens"][p][idx["page_tokens"][p] >= 0] for p in sel])
    assert set(range(20)) <= set(toks.tolist()) and set(range(850, 900)) <= set(toks.tolist())
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    kt = torch.from_numpy(K[toks].astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(V[toks].astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    assert np.max(np.abs(dec["out"] - ref)) < 1e-12


# ------------------------------------------------------------ three levels
def _l3_unit(N=3000, centres=48, promote_p=1.0 / 16, seed_head=0):
    w = workloads.WORKLOADS["llama31_8b_16k"].scaled(n_tokens=N, centres=centres, dtype="fp32",
                                                      promote_p=promote_p)
    th = oracle.promote_threshold(w.promote_p)
    K, V = workloads.unit_kv(w, 0, 0, seed_head)
    idx = oracle.build_unit(K, V, seed=w.seed, layer=0, seq=0, head=seed_head, thresh=th)
    lv2 = oracle.build_level2(idx, seed=w.seed, layer=0, seq=0, head=seed_head, thresh=th)
    return w, th, K, V, idx, lv2


def test_level2_nodes_assignment_and_children():
    w, th, K, V, idx, lv2 = _l3_unit()
    Np, node2, p2 = len(idx["parent_tok"]), lv2["node2"], lv2["parent2"]
    # promotion: exactly the parents whose level-2 draw is below the threshold
    want = [m for m, t in enumerate(idx["parent_tok"]) if oracle.promote_draw(w.seed, 0, 0, 0, int(t), 2) < th]
    assert list(node2) == want and len(want) > 0
    mu, sd = Np * w.promote_p, math.sqrt(Np * w.promote_p * (1 - w.promote_p))
    assert abs(len(node2) - mu) <= 5 * sd
    # every parent's level-2 parent is its nearest level-2 node (brute force in the lifted space)
    P = np.hstack([idx["parent_keys"], np.asarray(idx["parent_e"])[:, None]])
    D = ((P[:, None, :] - P[node2][None, :, :]) ** 2).sum(-1)
    assert np.all(D[np.arange(Np), p2] <= D.min(1) + 1e-12 * idx["M2"])
    assert np.all(p2[node2] == np.arange(len(node2)))  # level-2 nodes are their own parents
    # children: every parent in exactly one group, ascending inside it
    cs, ch = lv2["child_start"], lv2["children"]
    assert cs[0] == 0 and cs[-1] == Np and np.array_equal(np.sort(ch), np.arange(Np))
    for i in range(len(node2)):
        grp = ch[cs[i]:cs[i + 1]]
        assert np.all(np.diff(grp) > 0) and np.all(p2[grp] == i) and node2[i] in grp


def test_descent_expanding_every_level2_node_is_the_flat_selection():
    """With k at least the number of level-2 nodes every parent is a
    candidate, so the descent picks what the exact parent scan picks."""
    w, th, K, V, idx, lv2 = _l3_unit(N=1200, centres=16)
    q = workloads.unit_queries(w, 0, 0, 0)
    k = len(lv2["node2"])
    assert k <= 16 * 4
    heads, union = oracle.select_descent(q, idx, lv2, k)
    head_flat, union_flat = oracle.select(q, idx["parent_keys"], idx["page_parent"], k)
    assert np.array_equal(union, union_flat)
    for hh in range(len(q)):
        flat = [p for p in head_flat[hh] if p >= 0]
        assert heads[hh] == flat


def test_descent_with_every_token_promoted_is_exact_topk_mips():
    """p = 1: every token is a parent and a level-2 node with a one-token page;
    the descent is the exact top-k of q.k (torch.topk)."""
    w, th, K, V, idx, lv2 = _l3_unit(N=500, promote_p=1.0)
    q = workloads.unit_queries(w, 0, 0, 0)
    for k in (1, 5, 17):
        heads, union = oracle.select_descent(q, idx, lv2, k)
        for hh in range(len(q)):
            s = torch.from_numpy(K.astype(np.float64) @ q[hh].astype(np.float64))
            top = torch.topk(s, k).indices.numpy()
            assert sorted(heads[hh]) == sorted(idx["token_page"][top].tolist())


def test_decode_unit_three_levels_attends_over_the_descent_pages():
    w, th, K, V, idx, lv2 = _l3_unit()
    q = workloads.unit_queries(w, 0, 0, 0)
    idx3 = dict(idx, level2=lv2)
    dec = oracle.decode_unit(idx3, q, budget_tokens=128)
    _, union = oracle.select_descent(q, idx, lv2, 8)
    assert np.array_equal(dec["sel_pages"], union)
    toks = np.concatenate([idx["page_tokens"][p][idx["page_tokens"][p] >= 0] for p in union])
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    kt = torch.from_numpy(K[toks].astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(V[toks].astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    assert np.max(np.abs(dec["out"] - ref)) < 1e-12


def test_reuse_of_own_positional_three_level_index_is_itself():
    """Reusing a unit's own index with sink / window pages and a third level
    on its own keys gives back that index (M over the middle, pages and level
    2 kept)."""
    w, th, K, V, idx = _pos_unit(N=1200, n_sink=40, n_window=70)
    idx = dict(idx, level2=oracle.build_level2(idx, seed=w.seed, layer=0, seq=0, head=0, thresh=th))
    r = oracle.build_unit_reuse(K, V, idx)
    for f in ("parent_tok", "token_parent", "page_parent", "page_len", "page_tokens", "token_page", "token_slot",
              "parent_keys", "parent_e", "pool_k", "pool_v"):
        assert np.array_equal(np.asarray(r[f]), np.asarray(idx[f])), f
    assert r["M2"] == idx["M2"] and r["n_pos"] == idx["n_pos"] and r["level2"] is idx["level2"]


def test_level2_with_no_parent_promoted_takes_the_smallest_draw():
    """p small enough that no parent passes the level-2 draw: the parent of
    smallest level-2 draw (lowest m on ties) becomes the single level-2 node,
    and every parent is its child."""
    for seed_head in range(6):
        w, th, K, V, idx, lv2 = _l3_unit(N=400, promote_p=1.0 / 64, seed_head=seed_head)
        pt = idx["parent_tok"]
        draws = [oracle.promote_draw(w.seed, 0, 0, seed_head, int(t), 2) for t in pt]
        if any(d < th for d in draws):
            continue
        assert list(lv2["node2"]) == [int(np.argmin(draws))]
        assert np.all(lv2["parent2"] == 0)
        assert list(lv2["child_start"]) == [0, len(pt)] and np.array_equal(lv2["children"], np.arange(len(pt)))
        return
    pytest.skip("every seed promoted some parent to level 2")


def test_handworked_three_levels_and_descent():
    g = _load("handworked_descent_d2.json")
    K = np.array(g["keys"], float)
    n, M2, e = oracle.lift(K)
    assert M2 == 25 and np.all(e == 0)
    tp = oracle.assign(K, e, g["parent_tok"])
    assert tp.tolist() == g["token_parent"]
    pk = oracle.pack(tp, len(g["parent_tok"]), g["page_size"])
    for key in ("page_parent", "page_len", "page_tokens"):
        assert np.asarray(pk[key]).tolist() == g["pages"][key], key
    idx = dict(pk, S=g["page_size"], parent_tok=np.array(g["parent_tok"]), parent_keys=K[g["parent_tok"]],
               parent_e=e[g["parent_tok"]], token_parent=tp)
    # level 2 with the nodes of the example (the promotion draws are pinned separately)
    p2 = oracle.assign(idx["parent_keys"], idx["parent_e"], g["node2"])
    assert p2.tolist() == g["parent2"]
    order = np.argsort(p2, kind="stable")
    assert order.tolist() == g["children"]
    lv2 = dict(node2=np.array(g["node2"]), parent2=p2, child_start=np.array(g["child_start"]),
               children=np.array(g["children"]))
    for case in g["descent"]:
        heads, union = oracle.select_descent(np.array(case["q"], float), idx, lv2, case["k_pages"])
        assert heads == case["head_pages"], case["why"]
        assert union.tolist() == case["union"], case["why"]


def test_handworked_sink_and_window():
    g = _load("handworked_sink_window_d2.json")
    K, V = np.array(g["keys"], float), np.array(g["values"], float)
    assert oracle.positional_split(len(K), g["n_sink"], g["n_window"]) == tuple(g["split"])
    assert oracle.positional_pages(len(K), g["n_sink"], g["n_window"], g["page_size"]) == g["n_pos"]
    idx = oracle.build_unit_positional(K, V, seed=0, layer=0, seq=0, head=0, thresh=oracle.promote_threshold(1.0),
                                       S=g["page_size"], n_sink=g["n_sink"], n_window=g["n_window"])
    assert idx["M2"] == g["M2"] and np.asarray(idx["parent_e"]).tolist() == g["parent_e"]
    for key in ("parent_tok", "token_parent", "page_parent", "page_len", "page_tokens", "token_page", "token_slot"):
        assert np.asarray(idx[key]).tolist() == g[key], key
    assert idx["n_pages"] == g["n_pages"] and idx["n_pos"] == g["n_pos"]
    for case in g["decode"]:
        dec = oracle.decode_unit(idx, np.array(case["q"], float), case["budget_tokens"])
        assert dec["sel_pages"].tolist() == case["sel_pages"], case["why"]
        if "out" in case:
            assert np.allclose(dec["out"], case["out"], rtol=0, atol=1e-15), case["why"]
