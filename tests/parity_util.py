"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
on seeded workloads and compare every output with the CPU oracle.

Comparison rules (the reading of the pages' tolerance statement):
  * integer outputs (promotion, page tables, selections, copies) are compared
    bit-exactly;
  * a parent assignment may differ from the oracle's only at a near-tie: the
    oracle's lifted squared distance to the GPU's parent exceeds the best one
    by at most 2e-6 * M^2 (a 1e-6 relative tie in the lifted inner product
    k'.p', whose scale is |k'|^2 = M^2);
  * a selected page set may differ only through the order of DIFFERENT
    parents whose scores lie within 1e-6 * |q| * M of the k-th page's score
    (parents above that band are required in full; pages of one parent are
    always taken in page-id order; each query head selects exactly
    min(k, pages) pages): every head's legal selections are enumerated and
    the union must be the union of one legal selection per head;
  * attention outputs within 2e-3 max-abs (bf16 inputs) or 1e-5 (fp32).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import semantic_paged_kv_gb300 as ice
import workloads

TIE_REL = 1e-6
ATTN_TOL = {"bf16": 2e-3, "fp32": 1e-5}


def cfg_of(w: workloads.Workload, **kw) -> ice.Config:
    return ice.Config(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_tokens=w.n_tokens,
                      dtype=ice.ICE_BF16 if w.dtype == "bf16" else ice.ICE_FP32, promote_p=w.promote_p,
                      seed=w.seed, layer=kw.pop("layer", 0), **kw)


def to_dev(x: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda").to(dtype)


def host_tables(idx) -> dict:
    """Host copies of every index array but the pool (parent keys as fp32);
    arrays the index does not have (level 2 with two levels) are left out."""
    return {f: getattr(idx, f).float().cpu().numpy() if f == "parent_keys" else getattr(idx, f).cpu().numpy()
            for f in ice.INDEX_FIELDS if f not in ("pool_k", "pool_v") and getattr(idx, f) is not None}


class DeviceRun:
    """One layer built and decoded on the GPU, with host copies of everything."""

    def __init__(self, w: workloads.Workload, layer: int = 0, assign: str = "auto", host_pool=None, **cfg_kw):
        """host_pool: a callable cfg -> ice.HostPool; the pool then lives in
        pinned host memory (step a12) and the kernels reach it over the
        CPU-GPU link."""
        self.w = w
        self.cfg = cfg_of(w, layer=layer, **cfg_kw)
        self.layer = layer
        self.K, self.V = workloads.batch_kv(w, layer)
        dt = self.cfg.torch_dtype
        self.Kd, self.Vd = to_dev(self.K, dt), to_dev(self.V, dt)
        self.hp = host_pool(self.cfg) if host_pool else None
        self.idx = ice.Index(self.cfg, host_pool=self.hp)
        self.params = self.cfg.params()
        self.ws = ice.workspace(ice.ice_build_workspace_bytes(self.params))
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if assign == "auto":
            ice.ice_build_index(self.params, self.Kd, self.Vd, self.idx, self.ws, self.err)
        else:
            ice.ice_build_lift_promote(self.params, self.Kd, self.idx, self.ws, self.err)
            (ice.ice_build_assign_simt if assign == "simt" else ice.ice_build_assign)(
                self.params, self.Kd, self.idx, self.ws, self.err)
            ice.ice_build_pack(self.params, self.Kd, self.Vd, self.idx, self.ws, self.err)
        self.status = ice.ice_check(self.err)
        self.h = host_tables(self.idx)

    def pool(self, u):
        """Host copies (fp32) of unit u's pages, from HBM or the host pool."""
        P = int(self.h["n_pages"][u])
        hp = getattr(self, "hp", None)
        if hp is not None:
            def bits(which):
                x = hp.host_array(which)[u, :P]
                return (x.astype(np.uint32) << 16).view(np.float32) if self.cfg.dtype == ice.ICE_BF16 else \
                    x.view(np.float32).copy()
            return bits("k"), bits("v")
        return (self.idx.pool_k[u, :P].float().cpu().numpy(), self.idx.pool_v[u, :P].float().cpu().numpy())

    def unit(self, u):
        return u // self.cfg.n_kv_heads, u % self.cfg.n_kv_heads

    def queries(self, step: int = 0):
        """(host Q, device Q) of a decode step."""
        Q = workloads.batch_queries(self.w, self.layer, step)
        return Q, to_dev(Q, self.cfg.torch_dtype)

    def decode(self, budget: int, fused: bool = True, step: int = 0, contiguous: bool = True):
        """contiguous=False: ice_decode_step without kbuf/vbuf/buf_len (pages
        gathered on chip only)."""
        Q, Qd = self.queries(step)
        buf = ice.DecodeBuffers(self.cfg, budget)
        scale = 1.0 / np.sqrt(self.cfg.head_dim)
        if fused:
            kb, vb, bl = (buf.kbuf, buf.vbuf, buf.buf_len) if contiguous else (None, None, None)
            ice.ice_decode_step(self.params, self.idx, Qd, budget, buf.sel_pages, buf.sel_count, kb, vb, bl, scale,
                                buf.O, buf.ws, self.err)
        else:
            ice.ice_select_pages(self.params, self.idx, Qd, budget, buf.sel_pages, buf.sel_count, buf.ws, self.err)
            ice.ice_gather_pages(self.params, self.idx, buf.sel_pages, buf.sel_count, buf.kbuf, buf.vbuf, buf.buf_len)
            ice.ice_sparse_attn_decode(self.params, Qd, buf.kbuf, buf.vbuf, buf.buf_len, buf.sel_count, scale, buf.O,
                                       buf.ws)
        st = ice.ice_check(self.err)
        return Q, buf, st


class _UnitArrays:
    """K or V [B, H, N, d] on the device; [b, h] gives the host copy of one
    unit (fp32), made on first use."""

    def __init__(self, t: torch.Tensor):
        self.t, self.cache = t, {}

    def __getitem__(self, bh):
        if bh not in self.cache:
            self.cache[bh] = self.t[bh].float().cpu().numpy()
        return self.cache[bh]


class _UnitRows:
    """An index array [U, ...] on the device; [u, ...] indexes the host copy
    of row u, made on first use."""

    def __init__(self, t: torch.Tensor):
        self.t, self.cache = t, {}

    def __getitem__(self, key):
        u, rest = (key[0], key[1:]) if isinstance(key, tuple) else (key, ())
        u = int(u)
        if u not in self.cache:
            r = self.t[u]
            self.cache[u] = (r.float() if r.dtype == torch.bfloat16 else r).cpu().numpy()
        return self.cache[u][rest] if rest else self.cache[u]


class DeviceDrawnRun(DeviceRun):
    """A full-size layer on inputs drawn on the device
    (workloads.batch_kv_device / batch_queries_device, the benchmark's own
    inputs), built with ice_build_index.  Only the units a test looks at are
    copied to the host: their K, V rows and index rows, on first use; units
    are independent problems, so the oracle needs nothing else."""

    def __init__(self, w: workloads.Workload, layer: int = 0, host_pool=None, **cfg_kw):
        self.w = w
        self.cfg = cfg_of(w, layer=layer, **cfg_kw)
        self.layer = layer
        self.Kd, self.Vd, self.C = workloads.batch_kv_device(w, layer)
        self.K, self.V = _UnitArrays(self.Kd), _UnitArrays(self.Vd)
        self.hp = host_pool(self.cfg) if host_pool else None
        self.idx = ice.Index(self.cfg, host_pool=self.hp)
        self.params = self.cfg.params()
        self.ws = ice.workspace(ice.ice_build_workspace_bytes(self.params))
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ice.ice_build_index(self.params, self.Kd, self.Vd, self.idx, self.ws, self.err)
        self.status = ice.ice_check(self.err)
        self.h = {f: _UnitRows(getattr(self.idx, f)) for f in ice.INDEX_FIELDS
                  if f not in ("pool_k", "pool_v") and getattr(self.idx, f) is not None}

    def queries(self, step: int = 0):
        assert step == 0
        Qd = workloads.batch_queries_device(self.w, self.C, self.layer)
        return Qd.float().cpu().numpy(), Qd


# ------------------------------------------------------------ comparisons --
def lifted_d2(K, e, j, t):
    """Oracle-precision lifted squared distance between tokens j and t."""
    dk = K[j].astype(np.float64) - K[t].astype(np.float64)
    return float(dk @ dk + (e[j] - e[t]) ** 2)


def check_assignment_ties(dist, js, tp_gpu, tp_ora, M2: float, what="") -> np.ndarray:
    """Every token j in js whose device parent differs from the oracle's must
    be an fp32 near-tie: dist(j, m) is the oracle's lifted squared distance
    from token j to parent m, and the device's parent may be farther than the
    oracle's by at most 2 * TIE_REL * M^2.  The number of such tokens is
    capped (at most 2, or one in 2000).  Returns the mismatched tokens."""
    js = np.asarray(js)
    mism = js[np.asarray(tp_gpu)[js] != np.asarray(tp_ora)[js]]
    for j in mism:
        a, o = dist(j, int(tp_gpu[j])), dist(j, int(tp_ora[j]))
        assert a - o <= 2 * TIE_REL * M2, (what, int(j), int(tp_gpu[j]), int(tp_ora[j]), a, o)
    assert len(mism) <= max(2, len(js) // 2000), (what, len(mism))
    return mism


# At most this many different parents (or level-2 nodes) may lie in one
# near-tie band; their weak orders are enumerated (4683 for six).
MAX_TIED = 6


def _weak_orders(items):
    """Every ordered partition of items into non-empty blocks: the orders a
    device may give to scores that agree within the tolerance (a block is a
    set of exactly equal fp32 scores)."""
    items = list(items)
    if not items:
        yield []
        return
    n = len(items)
    for mask in range(1, 1 << n):
        block = [items[i] for i in range(n) if mask >> i & 1]
        rest = [items[i] for i in range(n) if not mask >> i & 1]
        for tail in _weak_orders(rest):
            yield [block] + tail


def legal_selections(s, items, k: int, tol: float, interleave: bool = True, what="") -> set:
    """Every set of min(k, #items) items that a device may select.

    Group i (a parent, or a level-2 node) has score s[i] (the oracle's, in
    double) and owns items[i] (its page ids, ascending; or [i]).  The
    reference takes items in the order (-s, item id) when interleave (pages
    of exactly tied parents mix by page id: the flat selection), else
    (-s, group index) with a group's items in id order (the descent), and
    keeps the first k.  A device that computes s in fp32 may order groups
    whose scores lie within tol of the k-th item's score in any weak order;
    groups above that band are selected in full, groups below it not at all,
    and a group's items are always taken in id order."""
    s = np.asarray(s, np.float64)
    sizes = np.array([len(x) for x in items], np.int64)
    total = int(sizes.sum())
    k_eff = min(k, total)
    if k_eff == 0:
        return {frozenset()}
    grp = np.repeat(np.arange(len(items)), sizes)
    ids = np.concatenate([np.asarray(x, np.int64) for x in items if len(x)])
    order = np.lexsort((ids, -s[grp])) if interleave else np.lexsort((ids, grp, -s[grp]))
    T = s[grp[order[k_eff - 1]]]
    R = frozenset(ids[s[grp] > T + tol].tolist())
    tied = [int(i) for i in np.nonzero((np.abs(s - T) <= tol) & (sizes > 0))[0]]
    need = k_eff - len(R)
    assert 1 <= need <= k_eff, (what, need)
    assert len(tied) <= MAX_TIED, (what, "too many near-tied groups", len(tied))
    out = set()
    for blocks in _weak_orders(tied):
        picked = []
        for blk in blocks:
            if interleave:
                picked += sorted(int(x) for i in blk for x in items[i])
            else:
                for i in sorted(blk):
                    picked += [int(x) for x in items[i]]
            if len(picked) >= need:
                break
        out.add(R | frozenset(picked[:need]))
    return out


def legal_descent_selections(qh, pkeys, pages_of, node2, child_start, children, k: int, tol: float, what="") -> set:
    """Every page set one query head may select by descent through level 2:
    the legal sets of k level-2 nodes (order (-q.p, i)), then for each, the
    legal page sets of their children (order (-q.p, m), a parent's pages in
    id order), k pages."""
    s2 = pkeys[node2] @ qh if len(node2) else np.zeros(0)
    out = set()
    for nodes in legal_selections(s2, [[i] for i in range(len(node2))], k, tol, interleave=False, what=what):
        cand = sorted(int(m) for i in nodes for m in children[child_start[i]:child_start[i + 1]])
        s1 = pkeys[cand] @ qh if cand else np.zeros(0)
        out |= legal_selections(s1, [pages_of[m] for m in cand], k, tol, interleave=False, what=what)
    return out


def check_union(got, per_head: list, what=""):
    """got (the device's ascending union) must be the union of one legal
    selection of every query head."""
    gs = frozenset(int(x) for x in got)
    states = {frozenset()}
    for hh, cands in enumerate(per_head):
        inside = [c for c in cands if c <= gs]
        assert inside, (what, "head", hh, "has no legal selection inside the union",
                        sorted(gs ^ set().union(*cands)) if cands else None)
        states = {st | c for st in states for c in inside}
        assert len(states) <= 200000, (what, "too many combinations")
    assert gs in states, (what, "the union is not made of one legal selection per head")


def pages_by_parent(page_parent, Np: int) -> list:
    """Page ids of every parent m < Np, ascending (pages of parent -1, the
    positional ones, belong to none)."""
    pp = np.asarray(page_parent)
    sem = np.nonzero(pp >= 0)[0]
    order = sem[np.argsort(pp[sem], kind="stable")]
    cnt = np.bincount(pp[sem], minlength=Np)[:Np]
    return [x.tolist() for x in np.split(order, np.cumsum(cnt)[:-1])] if Np else []


def check_level2_unit(run: DeviceRun, u: int, K, e, M2: float, lv2_ref: dict) -> dict:
    """Level 2 of unit u against the oracle's level 2 over the same parents:
    node2 exact; parent2 tie-aware (a parent may sit under another level-2
    node only at an fp32 near-tie of the lifted distance, and rarely);
    child_start / children exact against the oracle's grouping of the
    device's parent2.  K, e: the unit's keys and lifted coordinates (oracle
    precision).  Returns the device's level 2, checked."""
    H = run.h
    Np = int(H["n_parents"][u])
    pt = H["parent_tok"][u, :Np]
    n2 = len(lv2_ref["node2"])
    assert int(H["n_nodes2"][u]) == n2 and np.array_equal(H["node2"][u, :n2], lv2_ref["node2"]), (u, "node2")
    p2 = H["parent2"][u, :Np]
    node_tok = pt[lv2_ref["node2"]]
    check_assignment_ties(lambda m, i: lifted_d2(K, e, pt[m], node_tok[i]), np.arange(Np), p2, lv2_ref["parent2"],
                          M2, what=("unit", u, "level 2"))
    grp = oracle.level2_groups(p2, n2)
    assert np.array_equal(H["child_start"][u, :n2 + 1], grp["child_start"]), (u, "child_start")
    assert np.array_equal(H["children"][u, :Np], grp["children"]), (u, "children")
    return dict(node2=lv2_ref["node2"], parent2=p2.astype(np.int32), **grp)


def check_descent_selection(run: DeviceRun, u: int, q, k_pages: int, got, lv2: dict):
    """The device's union got (positional pages included) of unit u against
    the oracle's descent over the device's checked tables and level 2
    (near-ties at either level enumerated)."""
    H = run.h
    b, h = run.unit(u)
    Np, P = int(H["n_parents"][u]), int(H["n_pages"][u])
    Ps = P - run.cfg.n_pos
    got = np.asarray(got)
    assert np.all(np.diff(got) > 0)
    assert np.array_equal(got[got >= Ps], np.arange(Ps, P)), (u, "positional pages")
    got_sem = got[got < Ps]
    pkeys = run.K[b, h][H["parent_tok"][u, :Np]].astype(np.float64)
    q = np.asarray(q, np.float64)
    tables = dict(parent_keys=pkeys, n_pages=Ps, page_parent=H["page_parent"][u, :Ps])
    _, union = oracle.select_descent(q, tables, lv2, k_pages)
    if np.array_equal(got_sem, union):
        return
    M = np.sqrt(float(H["m2"][u]))
    pages_of = pages_by_parent(H["page_parent"][u, :Ps], Np)
    per_head = [legal_descent_selections(q[hh], pkeys, pages_of, lv2["node2"], lv2["child_start"], lv2["children"],
                                         k_pages, TIE_REL * np.linalg.norm(q[hh]) * M, what=("unit", u, "head", hh))
                for hh in range(len(q))]
    check_union(got_sem, per_head, what=("unit", u, "descent"))


def check_build_unit(run: DeviceRun, u: int, sample_tokens: int | None = None):
    """Promotion, lift, parent assignment (tie-aware), pages and pool of unit u.

    With sample_tokens set, the assignment is checked on that many seeded
    tokens (plus every parent); everything else on all tokens."""
    b, h = run.unit(u)
    w, cfg, H = run.w, run.cfg, run.h
    K = run.K[b, h].astype(np.float64)
    V = run.V[b, h].astype(np.float64)
    N = cfg.n_tokens
    th = oracle.promote_threshold(w.promote_p)
    # promotion: exact
    pt = oracle.promote(w.seed, run.layer, b, h, N, th)
    Np = int(H["n_parents"][u])
    assert Np == len(pt), (u, Np, len(pt))
    assert np.array_equal(H["parent_tok"][u, :Np], pt)
    assert int(H["n_indexed"][u]) == N
    if N == 0:
        assert int(H["n_pages"][u]) == 0
        return
    # lift
    n, M2, e = oracle.lift(K)
    assert abs(H["m2"][u] - M2) <= 1e-12 * M2
    assert np.allclose(H["parent_e"][u, :Np], e[pt].astype(np.float32), rtol=2e-7, atol=2e-7 * np.sqrt(M2))
    assert np.array_equal(run.idx.parent_keys[u, :Np].float().cpu().numpy(), run.K[b, h][pt])
    # assignment
    tp_gpu = H["token_parent"][u, :N]
    if sample_tokens is None:
        tp_ora = oracle.assign(K, e, pt)
        js = np.arange(N)
    else:
        rng = np.random.default_rng(1234 + u)
        js = np.unique(np.concatenate([rng.integers(0, N, sample_tokens), pt]))
        # oracle on the sample: the parents first, then the sampled tokens
        sub = np.concatenate([pt, js])
        sub_tp = oracle.assign(K[sub], e[sub], np.arange(len(pt)))
        tp_ora = np.full(N, -1)
        tp_ora[js] = sub_tp[len(pt):]
    check_assignment_ties(lambda j, m: lifted_d2(K, e, j, pt[m]), js, tp_gpu, tp_ora, M2, what=("unit", u))
    check_pack_unit(run, u)


def check_pack_unit(run: DeviceRun, u: int):
    """Pages, page tables and pool of unit u: the oracle packs the GPU's own
    assignment, and every table must match bit-exactly."""
    b, h = run.unit(u)
    cfg, H = run.cfg, run.h
    K = run.K[b, h].astype(np.float64)
    V = run.V[b, h].astype(np.float64)
    N = cfg.n_tokens
    Np = int(H["n_parents"][u])
    tp_gpu = H["token_parent"][u, :N]
    pk = oracle.pack(tp_gpu, Np, cfg.page_size)
    P = pk["n_pages"]
    assert int(H["n_pages"][u]) == P
    for key in ("page_parent", "page_len", "page_tokens"):
        assert np.array_equal(H[key][u, :P], pk[key]), key
    assert np.array_equal(H["token_page"][u, :N], pk["token_page"])
    assert np.array_equal(H["token_slot"][u, :N], pk["token_slot"])
    cnt = np.bincount(pk["page_parent"], minlength=Np)
    first = np.concatenate([[0], np.cumsum(cnt)[:-1]])
    assert np.array_equal(H["parent_n_pages"][u, :Np], cnt)
    assert np.array_equal(H["parent_first_page"][u, :Np], first)
    assert np.array_equal(H["parent_last_page"][u, :Np], first + cnt - 1)
    nxt = np.arange(1, P + 1)
    nxt[np.cumsum(cnt) - 1] = -1
    assert np.array_equal(H["page_next"][u, :P], nxt)
    # pool: exact copies, pad slots zero
    ok, ov = oracle.scatter(K, V, pk["page_tokens"], cfg.page_size)
    gk, gv = run.pool(u)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def check_build_positional(run: DeviceRun, u: int) -> dict:
    """The build of unit u when it may hold sink / window pages (none when
    n_sink = n_window = 0): parents and M^2 exact, the middle tokens'
    assignment tie-aware (check_assignment_ties), then the pages, token
    tables, parent spans and pool bit-exact against the oracle's packing of
    the device's (checked) assignment.  Returns the device's structure as an
    oracle index dict, for the reuse, level-2 and decode checks."""
    b, h = run.unit(u)
    w, cfg, H = run.w, run.cfg, run.h
    N, S = cfg.n_tokens, cfg.page_size
    th = oracle.promote_threshold(w.promote_p)
    K = run.K[b, h].astype(np.float64)
    V = run.V[b, h].astype(np.float64)
    ref = oracle.build_unit_positional(K, V, seed=w.seed, layer=run.layer, seq=b, head=h, thresh=th,
                                       n_sink=cfg.n_sink, n_window=cfg.n_window)
    pt, M2 = ref["parent_tok"], ref["M2"]
    Np = len(pt)
    assert int(H["n_parents"][u]) == Np and np.array_equal(H["parent_tok"][u, :Np], pt), (u, "parents")
    assert int(H["n_indexed"][u]) == N
    assert abs(H["m2"][u] - M2) <= 1e-12 * max(M2, 1e-30), (u, "M^2")
    assert np.allclose(H["parent_e"][u, :Np], np.asarray(ref["parent_e"], np.float32), rtol=2e-7,
                       atol=2e-7 * np.sqrt(M2)), (u, "parent_e")
    assert np.array_equal(run.idx.parent_keys[u, :Np].float().cpu().numpy(), run.K[b, h][pt]), (u, "parent keys")
    se, ws = ref["split"]
    tp = H["token_parent"][u, :N]
    assert np.all(tp[:se] == -2) and np.all(tp[ws:] == -2), (u, "positional tokens")
    e = ref["e"]
    check_assignment_ties(lambda j, m: lifted_d2(K, e, j, pt[m]), np.arange(se, ws), tp, ref["token_parent"], M2,
                          what=("unit", u))
    pk = oracle.pack_positional(tp[se:ws], Np, N, se, ws, S)
    P, n_pos = pk["n_pages"], pk["n_pos"]
    assert int(H["n_pages"][u]) == P, (u, "n_pages")
    for f in ("page_parent", "page_len", "page_tokens"):
        assert np.array_equal(H[f][u, :P], pk[f]), (u, f)
    assert np.array_equal(H["token_page"][u, :N], pk["token_page"]), (u, "token_page")
    assert np.array_equal(H["token_slot"][u, :N], pk["token_slot"]), (u, "token_slot")
    Ps = P - n_pos
    cnt = np.bincount(pk["page_parent"][:Ps], minlength=Np)[:Np]
    first = np.concatenate([[0], np.cumsum(cnt)[:-1]])[:Np]
    assert np.array_equal(H["parent_n_pages"][u, :Np], cnt)
    assert np.array_equal(H["parent_first_page"][u, :Np], first)
    assert np.array_equal(H["parent_last_page"][u, :Np], first + cnt - 1)
    nxt = np.arange(1, Ps + 1)
    if Np:
        nxt[np.cumsum(cnt) - 1] = -1
    assert np.array_equal(H["page_next"][u, :Ps], nxt), (u, "page_next")
    ok, ov = oracle.scatter(K, V, pk["page_tokens"], S)
    gk, gv = run.pool(u)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov), (u, "pool")
    return dict(ref, **pk, pool_k=ok, pool_v=ov)


def check_build_level2(run: DeviceRun, u: int, idx: dict) -> dict:
    """Level 2 of unit u over its checked level 1 (idx from
    check_build_positional): the oracle's level-2 build over the same
    parents, then check_level2_unit.  Returns the checked level 2."""
    b, h = run.unit(u)
    w = run.w
    th = oracle.promote_threshold(w.promote_p)
    K = run.K[b, h].astype(np.float64)
    e = np.where(np.isnan(idx["e"]), 0.0, idx["e"])
    lv2 = oracle.build_level2(idx, seed=w.seed, layer=run.layer, seq=b, head=h, thresh=th)
    return check_level2_unit(run, u, K, e, idx["M2"], lv2)


def check_decode_descent(run: DeviceRun, u: int, Q: np.ndarray, budget: int, buf, lv2: dict, idx: dict):
    """A three-level decode of unit u: the descent selection tie-aware
    (check_descent_selection), the attention over the device's selection
    against the oracle's (pages from idx, the checked structure)."""
    b, h = run.unit(u)
    g = run.cfg.group
    q = Q[b, h * g:(h + 1) * g].astype(np.float64)
    cnt = int(buf.sel_count[u])
    sel = buf.sel_pages[u].cpu().numpy()
    got = sel[:cnt]
    assert np.all(sel[cnt:] == -1)
    check_descent_selection(run, u, q, -(-budget // run.cfg.page_size), got, lv2)
    kb, vb, bl = oracle.gather(idx["pool_k"], idx["pool_v"], idx["page_len"], got)
    out = oracle.attention(q, kb, vb, bl, 1.0 / np.sqrt(run.cfg.head_dim))
    gpu = buf.O[b, h * g:(h + 1) * g].cpu().numpy()
    assert np.max(np.abs(gpu - out)) <= ATTN_TOL[run.w.dtype], (u, np.max(np.abs(gpu - out)))


def check_decode_unit(run: DeviceRun, u: int, Q: np.ndarray, budget: int, buf):
    """Selection (tie-aware), gather (exact) and attention (tolerance) of unit u."""
    b, h = run.unit(u)
    cfg, H = run.cfg, run.h
    g = cfg.group
    q = Q[b, h * g:(h + 1) * g].astype(np.float64)
    Np = int(H["n_parents"][u])
    P = int(H["n_pages"][u])
    pkeys = run.K[b, h][H["parent_tok"][u, :Np]].astype(np.float64)
    k_pages = -(-budget // cfg.page_size)
    cnt = int(buf.sel_count[u])
    sel = buf.sel_pages[u].cpu().numpy()
    got = sel[:cnt]
    assert np.all(sel[cnt:] == -1)
    if P == 0:
        assert cnt == 0
        assert np.all(buf.O[b, h * g:(h + 1) * g].cpu().numpy() == 0)
        return
    n_pos = run.cfg.n_pos  # positional (sink / window) pages: the last n_pos, always in the union
    Ps = P - n_pos
    assert np.all(np.diff(got) > 0)
    assert np.array_equal(got[got >= Ps], np.arange(Ps, P)), (u, "positional pages")
    got_sem = got[got < Ps]
    head, union = oracle.select(q, pkeys, H["page_parent"][u, :Ps], k_pages)
    if not np.array_equal(got_sem, union):
        # near-tie protocol: every head's legal selections under fp32 reordering of tied parents
        M = np.sqrt(float(H["m2"][u]))
        pages_of = pages_by_parent(H["page_parent"][u, :Ps], Np)
        per_head = [legal_selections(pkeys @ q[hh], pages_of, k_pages, TIE_REL * np.linalg.norm(q[hh]) * M,
                                     what=("unit", u, "head", hh)) for hh in range(g)]
        check_union(got_sem, per_head, what=("unit", u))
    # gather: exact copies of the selected pages
    pk_all, pv_all = run.pool(u)
    pk_sel, pv_sel = pk_all[got], pv_all[got]
    kb = buf.kbuf[u, :cnt].float().cpu().numpy()
    vb = buf.vbuf[u, :cnt].float().cpu().numpy()
    bl = buf.buf_len[u].cpu().numpy()
    assert np.array_equal(kb, pk_sel) and np.array_equal(vb, pv_sel)
    assert np.array_equal(bl[:cnt], H["page_len"][u, got]) and np.all(bl[cnt:] == 0)
    # attention over the GPU's selection
    out = oracle.attention(q, kb, vb, bl[:cnt], 1.0 / np.sqrt(cfg.head_dim))
    gpu = buf.O[b, h * g:(h + 1) * g].cpu().numpy()
    tol = ATTN_TOL[run.w.dtype]
    assert np.max(np.abs(gpu - out)) <= tol, (u, np.max(np.abs(gpu - out)))
