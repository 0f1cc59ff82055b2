"""The GPU parity checks themselves, on the CPU: do they notice a difference?

The comparison helpers of the GPU tests (parity_util.check_build_unit,
check_decode_unit) are fed the oracle's own index and decode outputs dressed
as device outputs (CPU tensors in the layout the library writes): they must
pass.  Then one output at a time is changed the way a kernel bug would
change it (a token under a farther parent, two tokens swapped between pages,
a pool value, a promoted token, M^2, a selected page, a gathered row, a page
length, the attention output, the wrong page of a parent that straddles the
budget, a tied page dropped, a parent under a far level-2 node) and the same
helper must fail, while a reorder of parents that tie within the tolerance
passes.  Nothing here runs the CUDA library."""
import types

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import (check_build_positional, check_build_unit, check_decode_unit, check_descent_selection,
                         check_level2_unit, check_union, cfg_of, legal_selections, pages_by_parent)

W = workloads.WORKLOADS["tiny"].scaled(n_tokens=700)
BUDGET = 64


class _Run:
    """What the helpers read from a device run, filled from the oracle (one unit)."""

    def __init__(self, n_sink: int = 0, n_window: int = 0, K=None):
        w = self.w = W
        self.cfg = cfg_of(w, layer=0, n_sink=n_sink, n_window=n_window)
        self.layer = 0
        self.K, self.V = workloads.batch_kv(w, 0)
        if K is not None:
            self.K = K
        th = oracle.promote_threshold(w.promote_p)
        if n_sink or n_window:
            ref = oracle.build_unit_positional(self.K[0, 0], self.V[0, 0], seed=w.seed, layer=0, seq=0, head=0,
                                               thresh=th, n_sink=n_sink, n_window=n_window)
        else:
            ref = oracle.build_unit(self.K[0, 0], self.V[0, 0], seed=w.seed, layer=0, seq=0, head=0, thresh=th)
        self.ref = ref
        cfg, N, S, d = self.cfg, w.n_tokens, self.cfg.page_size, self.cfg.head_dim
        Np, P = len(ref["parent_tok"]), int(ref["n_pages"])
        npc, pc = cfg.np_cap, cfg.page_cap

        def row(a, cap, fill, dtype=np.int32):
            out = np.full((1, cap) + np.shape(a)[1:], fill, dtype)
            out[0, :len(a)] = a
            return out

        pp = np.asarray(ref["page_parent"])
        cnt = np.bincount(pp[pp >= 0], minlength=Np)
        first = np.concatenate([[0], np.cumsum(cnt)[:-1]])
        nxt = np.arange(1, P + 1)
        nxt[np.cumsum(cnt) - 1] = -1
        nxt[len(pp[pp >= 0]):] = -1
        self.h = {"n_parents": np.array([Np]), "n_pages": np.array([P]), "n_indexed": np.array([N]),
                  "m2": np.array([ref["M2"]]), "parent_tok": row(ref["parent_tok"], npc, -1),
                  "parent_e": row(np.asarray(ref["parent_e"], np.float32), npc, 0, np.float32),
                  "token_parent": row(ref["token_parent"], N, -1), "token_page": row(ref["token_page"], N, -1),
                  "token_slot": row(ref["token_slot"], N, -1), "page_parent": row(pp, pc, -1),
                  "page_len": row(ref["page_len"], pc, 0), "page_tokens": row(ref["page_tokens"], pc, -1),
                  "parent_n_pages": row(cnt, npc, 0), "parent_first_page": row(first, npc, 0),
                  "parent_last_page": row(first + cnt - 1, npc, 0), "page_next": row(nxt, pc, -1)}
        pool_k = torch.zeros((1, pc, S, d))
        pool_v = torch.zeros((1, pc, S, d))
        pool_k[0, :P] = torch.from_numpy(ref["pool_k"])
        pool_v[0, :P] = torch.from_numpy(ref["pool_v"])
        keys = torch.zeros((1, npc, d))
        keys[0, :Np] = torch.from_numpy(np.asarray(ref["parent_keys"]))
        self.idx = types.SimpleNamespace(pool_k=pool_k, pool_v=pool_v, parent_keys=keys)

    def unit(self, u):
        return u // self.cfg.n_kv_heads, u % self.cfg.n_kv_heads

    def pool(self, u):
        P = int(self.h["n_pages"][u])
        return self.idx.pool_k[u, :P].numpy(), self.idx.pool_v[u, :P].numpy()

    def decode(self, budget: int = BUDGET):
        """(Q, buffers) as ice_decode_step leaves them, from the oracle's decode."""
        g = self.cfg.group
        Q = workloads.batch_queries(self.w, 0, 0)
        dec = oracle.decode_unit(self.ref, Q[0, :g], budget)
        return Q, self.buffers(Q, dec["sel_pages"], budget)

    def buffers(self, Q, sel_pages, budget: int = BUDGET):
        """Decode buffers that are consistent with the union sel_pages: the
        pages gathered from the pool and the oracle's attention over them."""
        cfg, g = self.cfg, self.cfg.group
        max_sel, S, d = g * (budget // cfg.page_size) + cfg.n_pos, cfg.page_size, cfg.head_dim
        sel_pages = np.asarray(sel_pages, np.int32)
        kb, vb, bl = oracle.gather(self.ref["pool_k"], self.ref["pool_v"], self.ref["page_len"], sel_pages)
        out = oracle.attention(Q[0, :g], kb, vb, bl)
        n = len(sel_pages)
        sel = torch.full((1, max_sel), -1, dtype=torch.int32)
        sel[0, :n] = torch.from_numpy(sel_pages)
        kbuf, vbuf = torch.zeros((1, max_sel, S, d)), torch.zeros((1, max_sel, S, d))
        kbuf[0, :n], vbuf[0, :n] = torch.from_numpy(kb), torch.from_numpy(vb)
        blen = torch.zeros((1, max_sel), dtype=torch.int32)
        blen[0, :n] = torch.from_numpy(np.asarray(bl))
        O = torch.from_numpy(out).float().reshape(1, g, d)
        return types.SimpleNamespace(sel_pages=sel, sel_count=torch.tensor([n], dtype=torch.int32), kbuf=kbuf,
                                     vbuf=vbuf, buf_len=blen, O=O)


def test_checks_accept_the_oracles_own_outputs():
    run = _Run()
    check_build_unit(run, 0)
    Q, buf = run.decode()
    check_decode_unit(run, 0, Q, BUDGET, buf)


def _far_parent(run):
    """A non-promoted token moved to the parent farthest from it."""
    ref, H = run.ref, run.h
    K = run.K[0, 0].astype(np.float64)
    e = oracle.lift(K)[2]
    pt = ref["parent_tok"]
    j = next(t for t in range(len(K)) if t not in set(pt.tolist()))
    d2 = ((K[pt] - K[j]) ** 2).sum(1) + (e[pt] - e[j]) ** 2
    H["token_parent"][0, j] = int(np.argmax(d2))


def _swap_tokens(run):
    """Two tokens of different pages exchanged in page_tokens."""
    pt = run.h["page_tokens"][0]
    a, b = pt[0, 0], pt[1, 0]
    pt[0, 0], pt[1, 0] = b, a


def _pool_value(run):
    run.idx.pool_k[0, 0, 0, 0] += 0.5


def _promoted_token(run):
    run.h["parent_tok"][0, 0] += 1


def _m2(run):
    run.h["m2"][0] *= 1 + 1e-9


BUILD_PLANTS = {"token_under_a_far_parent": _far_parent, "tokens_swapped_between_pages": _swap_tokens,
                "pool_value": _pool_value, "promoted_token": _promoted_token, "m2_off_by_1e-9": _m2}


@pytest.mark.parametrize("plant", list(BUILD_PLANTS))
def test_build_check_rejects_a_planted_difference(plant):
    run = _Run()
    BUILD_PLANTS[plant](run)
    with pytest.raises(AssertionError):
        check_build_unit(run, 0)


def _other_page(run, buf):
    """One selected page replaced by the best page that was not selected."""
    n = int(buf.sel_count[0])
    sel = set(buf.sel_pages[0, :n].tolist())
    P = int(run.h["n_pages"][0])
    g = run.cfg.group
    q = workloads.batch_queries(run.w, 0, 0)[0, :g].astype(np.float64)
    pk = np.asarray(run.ref["parent_keys"])
    s = (pk @ q.T).max(1)[np.asarray(run.ref["page_parent"])]
    out = max((p for p in range(P) if p not in sel), key=lambda p: s[p])
    new = sorted((sel - {buf.sel_pages[0, n - 1].item()}) | {out})
    buf.sel_pages[0, :n] = torch.tensor(new, dtype=torch.int32)


def _gathered_row(run, buf):
    buf.vbuf[0, 0, 0, 0] += 0.25


def _page_length(run, buf):
    buf.buf_len[0, 0] -= 1


def _output(run, buf):
    buf.O[0, 0, 0] += 1e-4  # the fp32 tolerance is 1e-5


DECODE_PLANTS = {"another_page_selected": _other_page, "gathered_row": _gathered_row, "page_length": _page_length,
                 "attention_output": _output}


@pytest.mark.parametrize("plant", list(DECODE_PLANTS))
def test_decode_check_rejects_a_planted_difference(plant):
    run = _Run()
    Q, buf = run.decode()
    DECODE_PLANTS[plant](run, buf)
    with pytest.raises(AssertionError):
        check_decode_unit(run, 0, Q, BUDGET, buf)


def test_decode_check_with_sink_and_window_pages():
    """The positional branch of check_decode_unit: the oracle's own decode
    passes; a union without its last positional page fails."""
    run = _Run(n_sink=16, n_window=40)
    assert run.cfg.n_pos == 4
    Q, buf = run.decode()
    check_decode_unit(run, 0, Q, BUDGET, buf)
    n = int(buf.sel_count[0])
    buf.sel_pages[0, n - 1] = -1
    buf.sel_count[0] = n - 1
    buf.buf_len[0, n - 1] = 0
    with pytest.raises(AssertionError):
        check_decode_unit(run, 0, Q, BUDGET, buf)


# ------------------------------------------------ selection near-tie rules --
def test_legal_selections_enumerates_only_reorders_of_tied_parents():
    """Groups 1 and 2 tie within the tolerance at the boundary (k = 3):
    either may come first, and a group's pages go in id order."""
    s = [5.0, 3.0, 3.0 + 1e-9, 1.0]
    items = [[0], [1, 2], [3], [4, 5]]
    got = legal_selections(s, items, 3, 1e-6)
    assert got == {frozenset({0, 1, 2}), frozenset({0, 1, 3}), frozenset({0, 3, 1})}
    assert frozenset({0, 2, 3}) not in got  # the tied parent's second page without its first
    got = legal_selections(s, items, 2, 1e-6)
    assert got == {frozenset({0, 1}), frozenset({0, 3})}
    # outside the tolerance the order is fixed
    assert legal_selections([5.0, 3.0, 2.9, 1.0], items, 2, 1e-6) == {frozenset({0, 1})}
    # equal fp32 scores interleave pages by id in the flat order, not in the descent's
    both = {frozenset({0, 5}), frozenset({3, 8})}
    assert legal_selections([1.0, 1.0], [[0, 5], [3, 8]], 2, 0.0) == both | {frozenset({0, 3})}
    assert legal_selections([1.0, 1.0], [[0, 5], [3, 8]], 2, 0.0, interleave=False) == both
    # fewer items than k: all of them
    assert legal_selections([1.0, 2.0], [[0], [1]], 5, 1e-6) == {frozenset({0, 1})}


def test_check_union_needs_one_legal_selection_per_head():
    h0 = {frozenset({1, 2}), frozenset({1, 3})}
    h1 = {frozenset({7, 8})}
    check_union([1, 2, 7, 8], [h0, h1])
    check_union([1, 3, 7, 8], [h0, h1])
    for bad in ([1, 7, 8], [1, 2, 3, 7, 8], [1, 2, 7], [1, 2, 7, 8, 9]):
        with pytest.raises(AssertionError):
            check_union(bad, [h0, h1])


def _straddle(run, budget):
    """(head list, union, k-th page a, next page b of the same parent) for a
    head whose k-th page's parent has a page beyond the budget, or None."""
    g = run.cfg.group
    Q = workloads.batch_queries(run.w, 0, 0)
    q = Q[0, :g].astype(np.float64)
    head, union = oracle.select(q, run.ref["parent_keys"], run.ref["page_parent"], budget // 16)
    pages_of = pages_by_parent(run.ref["page_parent"], len(run.ref["parent_tok"]))
    for hh in range(g):
        a = int(head[hh][-1])
        own = pages_of[int(run.ref["page_parent"][a])]
        later = [p for p in own if p > a and p not in set(union.tolist())]
        others = set(head[np.arange(g) != hh].reshape(-1).tolist())
        if later and a not in others:
            return Q, head[hh], union, a, later[0]
    return None


def _straddle_case():
    run = _Run()
    for budget in range(32, 257, 16):
        c = _straddle(run, budget)
        if c:
            return run, budget, c
    raise AssertionError("no straddling parent in the tiny workload")


def test_decode_check_rejects_the_wrong_page_of_a_straddling_parent():
    """A head's k-th page is the first page of a parent whose next page is
    not selected; the union with that next page instead (same parent, same
    score, buffers and attention consistent with it) must fail."""
    run, budget, (Q, _, union, a, b) = _straddle_case()
    check_decode_unit(run, 0, Q, budget, run.buffers(Q, union, budget))
    bad = sorted((set(union.tolist()) - {a}) | {b})
    with pytest.raises(AssertionError):
        check_decode_unit(run, 0, Q, budget, run.buffers(Q, bad, budget))


def test_decode_check_rejects_one_tied_page_dropped():
    """The same head's k-th page dropped from the union (its parent's score
    is the boundary itself): the head would hold k - 1 pages."""
    run, budget, (Q, _, union, a, _) = _straddle_case()
    bad = sorted(set(union.tolist()) - {a})
    with pytest.raises(AssertionError):
        check_decode_unit(run, 0, Q, budget, run.buffers(Q, bad, budget))


def test_decode_check_accepts_a_reorder_of_near_tied_parents():
    """Parent tokens given equal keys: the k-th page's parent and the next
    parent in the head's order tie exactly, so a device may take the other
    parent's first page at the boundary; the helper accepts that union and
    still rejects a page from an untied parent."""
    base = _Run()
    g = base.cfg.group
    Q = workloads.batch_queries(base.w, 0, 0)
    q = Q[0, :g].astype(np.float64)
    for hh in range(g):
        s = base.ref["parent_keys"] @ q[hh]
        order = np.argsort(-s, kind="stable")
        m1, m2 = int(order[0]), int(order[1])
        K = base.K.copy()
        K[0, 0, base.ref["parent_tok"][m2]] = K[0, 0, base.ref["parent_tok"][m1]]
        run = _Run(K=K)
        head, union = oracle.select(q, run.ref["parent_keys"], run.ref["page_parent"], 1)
        pages_of = pages_by_parent(run.ref["page_parent"], len(run.ref["parent_tok"]))
        lo, hi = min(m1, m2), max(m1, m2)
        if int(head[hh][0]) != pages_of[lo][0] or pages_of[hi][0] in set(union.tolist()):
            continue
        others = set(np.delete(head, hh, axis=0).reshape(-1).tolist())
        if pages_of[lo][0] in others:
            continue
        alt = sorted((set(union.tolist()) - {pages_of[lo][0]}) | {pages_of[hi][0]})
        check_decode_unit(run, 0, Q, 16, run.buffers(Q, alt, 16))
        far = max(range(int(run.ref["n_pages"])), key=lambda p: -s[run.ref["page_parent"][p]])
        bad = sorted((set(union.tolist()) - {pages_of[lo][0]}) | {far})
        with pytest.raises(AssertionError):
            check_decode_unit(run, 0, Q, 16, run.buffers(Q, bad, 16))
        return
    raise AssertionError("no head with a usable tie")


# ------------------------------------------------- three levels (descent) --
def _run3():
    run = _Run()
    th = oracle.promote_threshold(run.w.promote_p)
    lv2 = oracle.build_level2(run.ref, seed=run.w.seed, layer=0, seq=0, head=0, thresh=th)
    run.ref["level2"] = lv2
    Np, n2 = len(run.ref["parent_tok"]), len(lv2["node2"])
    npc = run.cfg.np_cap

    def row(a, cap):
        out = np.full((1, cap), -1, np.int32)
        out[0, :len(a)] = a
        return out

    run.h.update({"n_nodes2": np.array([n2]), "node2": row(lv2["node2"], npc), "parent2": row(lv2["parent2"], npc),
                  "child_start": row(lv2["child_start"], npc + 1), "children": row(lv2["children"], npc)})
    return run, lv2


def test_descent_checks_accept_the_oracle_and_reject_planted_differences():
    run, lv2_ref = _run3()
    K = run.K[0, 0].astype(np.float64)
    _, M2, e = oracle.lift(K)
    lv2 = check_level2_unit(run, 0, K, e, M2, lv2_ref)
    g = run.cfg.group
    Q = workloads.batch_queries(run.w, 0, 0)
    dec = oracle.decode_unit(run.ref, Q[0, :g], BUDGET)
    check_descent_selection(run, 0, Q[0, :g], BUDGET // 16, dec["sel_pages"], lv2)
    # another page in the union
    sel = set(dec["sel_pages"].tolist())
    out = next(p for p in range(int(run.ref["n_pages"])) if p not in sel)
    with pytest.raises(AssertionError):
        check_descent_selection(run, 0, Q[0, :g], BUDGET // 16, sorted(sel | {out}), lv2)
    # a page dropped
    with pytest.raises(AssertionError):
        check_descent_selection(run, 0, Q[0, :g], BUDGET // 16, sorted(sel - {min(sel)}), lv2)
    # a parent moved to the level-2 node farthest from it
    Np = len(run.ref["parent_tok"])
    m = next(m for m in range(Np) if m not in set(lv2_ref["node2"].tolist()))
    pt = run.ref["parent_tok"]
    d2 = [((K[pt[m]] - K[pt[i]]) ** 2).sum() + (e[pt[m]] - e[pt[i]]) ** 2 for i in lv2_ref["node2"]]
    run.h["parent2"][0, m] = int(np.argmax(d2))
    with pytest.raises(AssertionError):
        check_level2_unit(run, 0, K, e, M2, lv2_ref)


def test_positional_build_check_accepts_the_oracle_and_rejects_planted_differences():
    """check_build_positional (sink and window pages): the oracle's own build
    passes; a middle token under a far parent, a positional token given a
    parent, and two tokens swapped between pages each fail."""
    check_build_positional(_Run(n_sink=16, n_window=40), 0)
    run = _Run(n_sink=16, n_window=40)
    K = run.K[0, 0].astype(np.float64)
    e = run.ref["e"]
    pt = run.ref["parent_tok"]
    j = next(t for t in range(16, 700 - 40) if t not in set(pt.tolist()))
    d2 = ((K[pt] - K[j]) ** 2).sum(1) + (e[pt] - e[j]) ** 2
    run.h["token_parent"][0, j] = int(np.argmax(d2))
    with pytest.raises(AssertionError):
        check_build_positional(run, 0)
    run = _Run(n_sink=16, n_window=40)
    run.h["token_parent"][0, 3] = 0
    with pytest.raises(AssertionError):
        check_build_positional(run, 0)
    run = _Run(n_sink=16, n_window=40)
    _swap_tokens(run)
    with pytest.raises(AssertionError):
        check_build_positional(run, 0)
