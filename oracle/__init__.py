"""IceCache CPU oracle (test infrastructure only).

The plain C restatement of the method lives in ``oracle.c``; this module
compiles it with gcc into ``liboracle.so`` next to it and wraps each step for
numpy arrays.  Every floating-point step runs in IEEE double on inputs that
are exact in double (bf16 or fp32 values widened).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import this package.  The product library
(``semantic_paged_kv_gb300``) never imports it and shares no code with it.

Steps and their sources (page title, section):
  lift, promote, assign, pack, insert -- IceCache popular-science article
      (aitangshan.cn/news/751385) section 三; papernotes.org "IceCache:
      Memory-Efficient KV-cache Management for Long-Sequence LLMs",
      关键设计 2.
  select + GQA union -- papernotes 关键设计 3; article section 六.
  gather -- papernotes 关键设计 4; article section 四.
  attention -- papernotes 关键设计 1 (the a_ij formula).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_NOMEM, ERR_CAPACITY = 0, 1, 3, 4


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, u64, u32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double
        lib.orc_splitmix64_mix.argtypes = [u64]
        lib.orc_splitmix64_mix.restype = u64
        lib.orc_splitmix64_nth.argtypes = [u64, u64]
        lib.orc_splitmix64_nth.restype = u64
        lib.orc_promote_draw.argtypes = [u64, i32, i32, i32, i64, i32]
        lib.orc_promote_draw.restype = u32
        lib.orc_lift.argtypes = [P, i64, i32, P, P, P]
        lib.orc_promote.argtypes = [u64, i32, i32, i32, i64, u64, P, P]
        lib.orc_assign.argtypes = [P, P, i64, i32, P, i32, P]
        lib.orc_pack.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P]
        lib.orc_scatter.argtypes = [P, P, i64, i32, i32, i32, P, P, P]
        lib.orc_select.argtypes = [P, i32, i32, P, i32, P, i32, i32, P, P, P]
        lib.orc_gather.argtypes = [P, P, P, i32, i32, i32, P, i32, P, P, P]
        lib.orc_attention.argtypes = [P, i32, i32, P, P, P, i32, i32, f64, P]
        lib.orc_insert.argtypes = [u64, i32, i32, i32, u64, i32, i32, f64, P, P, i64, i32,
                                   i32, P, P, P, P,
                                   i32, P, P, P, P, P, P,
                                   i64, P, P, P]
        for name in ("orc_lift", "orc_promote", "orc_assign", "orc_pack", "orc_scatter",
                     "orc_select", "orc_gather", "orc_attention", "orc_insert"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc: int, what: str):
    if rc != OK:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- hash ----
def splitmix64_mix(z: int) -> int:
    return int(_load().orc_splitmix64_mix(z & 0xFFFFFFFFFFFFFFFF))


def splitmix64_nth(s0: int, n: int) -> int:
    return int(_load().orc_splitmix64_nth(s0 & 0xFFFFFFFFFFFFFFFF, n & 0xFFFFFFFFFFFFFFFF))


def promote_draw(seed: int, layer: int, seq: int, head: int, token: int, level: int = 1) -> int:
    return int(_load().orc_promote_draw(seed, layer, seq, head, token, level))


def promote_threshold(p: float) -> int:
    """floor(p * 2^32) for p in [0, 1] (2^32 means always promoted)."""
    return int(np.floor(p * 4294967296.0))


# ---------------------------------------------------------- build steps ----
def lift(K) -> tuple[np.ndarray, float, np.ndarray]:
    K = _f64(K)
    N, d = K.shape
    n = np.empty(N, np.float64)
    e = np.empty(N, np.float64)
    M2 = ctypes.c_double(0.0)
    _check(_load().orc_lift(_p(K), N, d, _p(n), ctypes.byref(M2), _p(e)), "lift")
    return n, float(M2.value), e


def promote(seed: int, layer: int, seq: int, head: int, N: int, thresh: int) -> np.ndarray:
    out = np.empty(max(N, 1), np.int32)
    np_ = ctypes.c_int32(0)
    _check(_load().orc_promote(seed, layer, seq, head, N, thresh, _p(out), ctypes.byref(np_)), "promote")
    return out[: np_.value].copy()


def assign(K, e, parent_tok) -> np.ndarray:
    K = _f64(K)
    e = _f64(e)
    pt = _i32(parent_tok)
    N, d = K.shape
    out = np.empty(max(N, 1), np.int32)
    _check(_load().orc_assign(_p(K), _p(e), N, d, _p(pt), len(pt), _p(out)), "assign")
    return out[:N].copy()


def page_capacity(N: int, Np: int, S: int) -> int:
    """Upper bound on pages: sum_m ceil(c_m / S) <= (N + (S-1) Np) / S."""
    return (N + (S - 1) * Np) // S


def pack(token_parent, Np: int, S: int, page_cap: int | None = None) -> dict:
    tp = _i32(token_parent)
    N = len(tp)
    cap = page_capacity(N, Np, S) if page_cap is None else page_cap
    c1 = max(cap, 1)
    page_parent = np.full(c1, -1, np.int32)
    page_len = np.zeros(c1, np.int32)
    page_tokens = np.full(c1 * S, -1, np.int32)
    token_page = np.full(max(N, 1), -1, np.int32)
    token_slot = np.full(max(N, 1), -1, np.int32)
    P = ctypes.c_int32(0)
    _check(_load().orc_pack(_p(tp), N, Np, S, cap, ctypes.byref(P), _p(page_parent), _p(page_len),
                            _p(page_tokens), _p(token_page), _p(token_slot)), "pack")
    P = P.value
    return dict(n_pages=P, page_parent=page_parent[:P].copy(), page_len=page_len[:P].copy(),
                page_tokens=page_tokens[: P * S].reshape(P, S).copy(),
                token_page=token_page[:N].copy(), token_slot=token_slot[:N].copy())


def scatter(K, V, page_tokens: np.ndarray, S: int) -> tuple[np.ndarray, np.ndarray]:
    K = _f64(K)
    V = _f64(V)
    N, d = K.shape
    pt = _i32(page_tokens).reshape(-1)
    P = pt.size // S
    pk = np.zeros((max(P, 1), S, d), np.float64)
    pv = np.zeros((max(P, 1), S, d), np.float64)
    _check(_load().orc_scatter(_p(K), _p(V), N, d, S, P, _p(pt), _p(pk), _p(pv)), "scatter")
    return pk[:P].copy(), pv[:P].copy()


# ---------------------------------------------------------- decode steps ----
def select(q, parent_keys, page_parent, k_pages: int) -> tuple[np.ndarray, np.ndarray]:
    """Returns (head_pages [g, k_pages] with -1 pad, union [count] ascending)."""
    q = _f64(q)
    pk = _f64(parent_keys)
    pp = _i32(page_parent)
    g, d = q.shape
    Np = pk.shape[0] if pk.size else 0
    P = len(pp)
    head = np.full(max(g * k_pages, 1), -1, np.int32)
    sel = np.full(max(g * k_pages, 1), -1, np.int32)
    cnt = ctypes.c_int32(0)
    _check(_load().orc_select(_p(q), g, d, _p(pk if pk.size else np.zeros(1)), Np, _p(pp if P else np.zeros(1, np.int32)),
                              P, k_pages, _p(head), _p(sel), ctypes.byref(cnt)), "select")
    return head[: g * k_pages].reshape(g, k_pages).copy(), sel[: cnt.value].copy()


def gather(pool_k, pool_v, page_len, sel_pages) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    pk = _f64(pool_k)
    pv = _f64(pool_v)
    P, S, d = pk.shape
    sel = _i32(sel_pages)
    U = len(sel)
    kb = np.zeros((max(U, 1), S, d), np.float64)
    vb = np.zeros((max(U, 1), S, d), np.float64)
    bl = np.zeros(max(U, 1), np.int32)
    _check(_load().orc_gather(_p(pk), _p(pv), _p(_i32(page_len)), P, S, d, _p(sel), U, _p(kb), _p(vb), _p(bl)),
           "gather")
    return kb[:U].copy(), vb[:U].copy(), bl[:U].copy()


def attention(q, kbuf, vbuf, buf_len, scale: float | None = None) -> np.ndarray:
    q = _f64(q)
    g, d = q.shape
    kb = _f64(kbuf)
    vb = _f64(vbuf)
    U = kb.shape[0]
    S = kb.shape[1] if kb.ndim == 3 else 1
    bl = _i32(buf_len)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((g, d), np.float64)
    _check(_load().orc_attention(_p(q), g, d, _p(kb if U else np.zeros(1)), _p(vb if U else np.zeros(1)),
                                 _p(bl if U else np.zeros(1, np.int32)), U, S, float(scale), _p(out)), "attention")
    return out


# ------------------------------------------------------- whole-unit drivers ----
def build_unit(K, V, *, seed: int, layer: int, seq: int, head: int, thresh: int, S: int = 16) -> dict:
    """All build steps (a1-a5) for one (seq, layer, KV head) unit."""
    K = _f64(K)
    V = _f64(V)
    N = K.shape[0]
    n, M2, e = lift(K)
    parent_tok = promote(seed, layer, seq, head, N, thresh)
    token_parent = assign(K, e, parent_tok)
    pk = pack(token_parent, len(parent_tok), S)
    pool_k, pool_v = scatter(K, V, pk["page_tokens"], S)
    return dict(n=n, M2=M2, e=e, parent_tok=parent_tok, parent_keys=K[parent_tok] if N else K[:0],
                parent_e=e[parent_tok] if N else e[:0], token_parent=token_parent,
                pool_k=pool_k, pool_v=pool_v, S=S, **pk)


# ------------------------------------------- sink and recent-window pages ----
def positional_split(N: int, n_sink: int, n_window: int) -> tuple[int, int]:
    """(sink_end, window_start) of a build over N tokens.  The article's
    section 六 splits the tokens into the first few anchor (sink) tokens, the
    window of the newest tokens, and everything in between; the sink and
    window stay resident and only the middle goes into the index.  Sink =
    [0, sink_end), window = [window_start, N), middle = [sink_end,
    window_start); a window reaching into the sink is cut at the sink."""
    se = min(max(n_sink, 0), N)
    return se, max(se, N - max(n_window, 0))


def positional_pages(N: int, n_sink: int, n_window: int, S: int = 16) -> int:
    se, ws = positional_split(N, n_sink, n_window)
    return -(-se // S) + -(-(N - ws) // S)


def promote_range(seed: int, layer: int, seq: int, head: int, lo: int, hi: int, thresh: int) -> np.ndarray:
    """Promotion restricted to the tokens [lo, hi) (article section 三's random
    promotion, over the indexed tokens only): token j is promoted iff its
    draw is below thresh; if none is, the token of smallest draw (lowest j
    on ties) is.  Token ids stay absolute."""
    d = np.array([promote_draw(seed, layer, seq, head, j) for j in range(lo, hi)], np.int64)
    if hi <= lo:
        return np.zeros(0, np.int32)
    out = np.nonzero(d < thresh)[0]
    if len(out) == 0:
        out = np.array([int(np.argmin(d))])
    return (out + lo).astype(np.int32)


def build_unit_positional(K, V, *, seed: int, layer: int, seq: int, head: int, thresh: int, S: int = 16,
                          n_sink: int = 0, n_window: int = 0) -> dict:
    """Build of one unit whose first n_sink and last n_window tokens are kept
    as positional pages (article section 六: the anchor and window pages stay
    on the GPU, only the middle tokens are managed by the index).  The middle
    tokens go through the steps of build_unit (lift with M over the middle,
    promotion among the middle, nearest parent, pack); the sink tokens then
    fill pages P_sem .. in chunks of S in token order, and the window tokens
    the pages after them.  Positional pages have no parent (-1) and their
    tokens token_parent -2."""
    K = _f64(K)
    V = _f64(V)
    N = K.shape[0]
    se, ws = positional_split(N, n_sink, n_window)
    Km = K[se:ws]
    n_m, M2, e_m = lift(Km) if ws > se else (np.zeros(0), 0.0, np.zeros(0))
    parent_tok = promote_range(seed, layer, seq, head, se, ws, thresh)
    Np = len(parent_tok)
    tp_mid = assign(Km, e_m, parent_tok - se) if Np else np.zeros(0, np.int32)
    pk = pack_positional(tp_mid, Np, N, se, ws, S)
    pool_k, pool_v = scatter(K, V, pk["page_tokens"], S)
    e = np.full(N, np.nan)
    e[se:ws] = e_m
    return dict(n=n_m, M2=M2, e=e, parent_tok=parent_tok, parent_keys=K[parent_tok] if Np else K[:0],
                parent_e=e[parent_tok] if Np else e[:0], pool_k=pool_k, pool_v=pool_v, S=S, **pk)


def pack_positional(tp_mid, Np: int, N: int, se: int, ws: int, S: int = 16) -> dict:
    """The pages of a unit with sink / window tokens (article section 六):
    the middle tokens [se, ws) with parents tp_mid (middle-relative token
    order) packed as in pack(), then the sink tokens [0, se) in positional
    pages of S in token order, then the window tokens [ws, N).  Returns the
    page and token tables over all N tokens (token_parent -2 outside the
    middle, page_parent -1 for positional pages)."""
    tp_mid = np.asarray(tp_mid, np.int32)
    pk = pack(tp_mid, Np, S) if ws > se else dict(n_pages=0, page_parent=np.zeros(0, np.int32),
                                                   page_len=np.zeros(0, np.int32),
                                                   page_tokens=np.zeros((0, S), np.int32),
                                                   token_page=np.zeros(0, np.int32), token_slot=np.zeros(0, np.int32))
    P_sem = pk["n_pages"]
    sem_tokens = np.where(pk["page_tokens"] >= 0, pk["page_tokens"] + se, -1)
    ranges = [(a, min(a + S, se)) for a in range(0, se, S)] + [(a, min(a + S, N)) for a in range(ws, N, S)]
    pos_tokens = np.full((len(ranges), S), -1, np.int32)
    for i, (a, b) in enumerate(ranges):
        pos_tokens[i, : b - a] = np.arange(a, b)
    page_tokens = np.concatenate([sem_tokens.astype(np.int32), pos_tokens]).astype(np.int32)
    P = P_sem + len(ranges)
    page_parent = np.concatenate([pk["page_parent"], np.full(len(ranges), -1, np.int32)]).astype(np.int32)
    page_len = np.concatenate([pk["page_len"], np.array([b - a for a, b in ranges], np.int32)]).astype(np.int32)
    token_parent = np.full(N, -2, np.int32)
    token_parent[se:ws] = tp_mid
    token_page = np.full(N, -1, np.int32)
    token_slot = np.full(N, -1, np.int32)
    for p in range(P):
        for sl in range(S):
            t = page_tokens[p, sl]
            if t >= 0:
                token_page[t], token_slot[t] = p, sl
    return dict(token_parent=token_parent, n_pages=P, n_pos=len(ranges), split=(se, ws), page_parent=page_parent,
                page_len=page_len, page_tokens=page_tokens, token_page=token_page, token_slot=token_slot)


# ------------------------------------------------------------ level 2 ----
def build_level2(idx: dict, *, seed: int, layer: int, seq: int, head: int, thresh: int) -> dict:
    """The level above the parents (papernotes 关键设计 2: points are promoted
    at random level by level and every point of a level takes its nearest
    point one level up as parent; article section 三).  A parent (level-1
    node) m is promoted to level 2 iff the draw of its token at level 2 is
    below thresh; if none is, the one of smallest draw (lowest m on ties).
    Level-2 nodes i = 0.. are those parents in ascending m (node2[i] = m).
    parent2[m]: the level-2 node nearest to parent m in lifted space (the
    parents' keys with their lifted coordinate; ties to the lowest i), a
    level-2 node being its own.  children: the parents grouped by parent2,
    ascending m inside a group, group i at [child_start[i], child_start[i+1])."""
    pt = np.asarray(idx["parent_tok"], np.int64)
    Np = len(pt)
    if Np == 0:
        return dict(node2=np.zeros(0, np.int32), parent2=np.zeros(0, np.int32),
                    child_start=np.zeros(1, np.int32), children=np.zeros(0, np.int32))
    d2 = np.array([promote_draw(seed, layer, seq, head, int(t), 2) for t in pt], np.int64)
    node2 = np.nonzero(d2 < thresh)[0]
    if len(node2) == 0:
        node2 = np.array([int(np.argmin(d2))])
    node2 = node2.astype(np.int32)
    parent2 = assign(idx["parent_keys"], idx["parent_e"], node2)
    return dict(node2=node2, parent2=parent2.astype(np.int32), **level2_groups(parent2, len(node2)))


def level2_groups(parent2, n2: int) -> dict:
    """The children of every level-2 node: the parents grouped by their
    level-2 parent (ascending m inside a group), group i at
    children[child_start[i] : child_start[i + 1])."""
    parent2 = np.asarray(parent2, np.int64)
    order = np.argsort(parent2, kind="stable").astype(np.int32)
    counts = np.bincount(parent2, minlength=n2)
    child_start = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return dict(child_start=child_start, children=order)


def select_descent(q, idx: dict, lv2: dict, k_pages: int) -> tuple[list, np.ndarray]:
    """Page selection by descent through level 2 (papernotes 关键设计 2: the
    query finds the k nearest points of the top level, then continues among
    their children; 关键设计 3: per head, union over the GQA group).  With
    the lifted query q' = [q, 0], nearest means largest q.p.  Per head: the
    first k = k_pages level-2 nodes in (-q.p, i) order, then their children
    in (-q.p, m) order, whose pages (page-id order inside a parent) are taken
    until k pages.  Returns (per-head page lists, ascending union) over the
    semantic pages."""
    q = _f64(q)
    pk = _f64(idx["parent_keys"])
    node2, ch, cs = lv2["node2"], lv2["children"], lv2["child_start"]
    n_pos = int(idx.get("n_pos", 0))
    P_sem = int(idx["n_pages"]) - n_pos
    page_parent = np.asarray(idx["page_parent"][:P_sem])
    pages_of = [[] for _ in range(len(pk))]
    for pg, m in enumerate(page_parent):
        pages_of[m].append(pg)
    heads, union = [], set()
    for qh in q:
        s2 = pk[node2] @ qh if len(node2) else np.zeros(0)
        top2 = sorted(range(len(node2)), key=lambda i: (-s2[i], i))[:k_pages]
        cand = [int(m) for i in top2 for m in ch[cs[i]:cs[i + 1]]]
        s1 = {m: float(pk[m] @ qh) for m in cand}
        pages = []
        for m in sorted(cand, key=lambda m: (-s1[m], m)):
            for pg in pages_of[m]:
                if len(pages) < k_pages:
                    pages.append(pg)
        heads.append(pages)
        union |= set(pages)
    return heads, np.array(sorted(union), np.int32)


def build_unit_reuse(K, V, prev: dict, S: int = 16) -> dict:
    """Build of one unit on another layer's node structure (the inter-layer
    index reuse of the article's section 五, "IceCache (reuse)"; its mechanism
    is not described, so this is the stated rule): the promoted tokens and
    the token -> parent assignment are prev's; the lift (M^2, e) comes from
    this layer's keys (step a1), the pages from packing prev's assignment
    (step a4), the pool from this layer's K and V (step a5).  With sink /
    window pages in prev, M is taken over the indexed middle tokens and every
    page is kept as it is; a third level in prev is kept too.  prev must index
    the same N tokens."""
    K = _f64(K)
    V = _f64(V)
    N = K.shape[0]
    parent_tok = np.asarray(prev["parent_tok"], np.int32)
    token_parent = np.asarray(prev["token_parent"][:N], np.int32)
    if len(token_parent) != N or (len(parent_tok) and (parent_tok.min() < 0 or parent_tok.max() >= N)):
        raise ValueError("prev does not index the same N tokens")
    extra = {k: prev[k] for k in ("level2",) if k in prev}  # a third level is node structure too: kept
    if int(prev.get("n_pos", 0)) or "split" in prev:
        # sink / window pages: M over the indexed (middle) tokens, every page kept as it is
        se, ws = prev["split"]
        n, M2, e_m = lift(K[se:ws]) if ws > se else (np.zeros(0), 0.0, np.zeros(0))
        e = np.full(N, np.nan)
        e[se:ws] = e_m
        pk = {f: prev[f] for f in ("n_pages", "n_pos", "split", "page_parent", "page_len", "page_tokens",
                                   "token_page", "token_slot")}
    else:
        n, M2, e = lift(K)
        pk = pack(token_parent, len(parent_tok), S)
    pool_k, pool_v = scatter(K, V, pk["page_tokens"], S)
    return dict(n=n, M2=M2, e=e, parent_tok=parent_tok, parent_keys=K[parent_tok] if N else K[:0],
                parent_e=e[parent_tok] if N else e[:0], token_parent=token_parent,
                pool_k=pool_k, pool_v=pool_v, S=S, **pk, **extra)


def decode_unit(idx: dict, q, budget_tokens: int, scale: float | None = None) -> dict:
    """Decode steps a6-a10 for one unit and its g query heads."""
    S = idx["S"]
    k_pages = -(-budget_tokens // S)
    n_pos = int(idx.get("n_pos", 0))  # positional (sink / window) pages: the last n_pos, always attended
    P_sem = int(idx["n_pages"]) - n_pos
    if "level2" in idx:  # three levels: descent through level 2
        head_pages, sel = select_descent(q, idx, idx["level2"], k_pages)
    else:
        head_pages, sel = select(q, idx["parent_keys"], idx["page_parent"][:P_sem], k_pages)
    if n_pos:
        sel = np.concatenate([sel, np.arange(P_sem, P_sem + n_pos, dtype=np.int32)]).astype(np.int32)
    kb, vb, bl = gather(idx["pool_k"], idx["pool_v"], idx["page_len"], sel)
    out = attention(q, kb, vb, bl, scale)
    return dict(head_pages=head_pages, sel_pages=sel, kbuf=kb, vbuf=vb, buf_len=bl, out=out)


class UnitIndex:
    """Mutable per-unit index for the incremental insert (capacities fixed)."""

    def __init__(self, idx: dict, d: int, np_cap: int, page_cap: int, n_cap: int):
        S = idx["S"]
        self.S, self.d, self.M2 = S, d, float(idx["M2"])
        Np, P, N = len(idx["parent_tok"]), idx["n_pages"], len(idx["token_parent"])
        self.n_parents = ctypes.c_int32(Np)
        self.n_pages = ctypes.c_int32(P)
        self.parent_tok = np.full(np_cap, -1, np.int32); self.parent_tok[:Np] = idx["parent_tok"]
        self.parent_keys = np.zeros((np_cap, d)); self.parent_keys[:Np] = idx["parent_keys"]
        self.parent_e = np.zeros(np_cap); self.parent_e[:Np] = idx["parent_e"]
        self.page_parent = np.full(page_cap, -1, np.int32); self.page_parent[:P] = idx["page_parent"]
        self.page_len = np.zeros(page_cap, np.int32); self.page_len[:P] = idx["page_len"]
        self.page_tokens = np.full((page_cap, S), -1, np.int32); self.page_tokens[:P] = idx["page_tokens"]
        self.pool_k = np.zeros((page_cap, S, d)); self.pool_k[:P] = idx["pool_k"]
        self.pool_v = np.zeros((page_cap, S, d)); self.pool_v[:P] = idx["pool_v"]
        self.token_parent = np.full(n_cap, -1, np.int32); self.token_parent[:N] = idx["token_parent"]
        self.token_page = np.full(n_cap, -1, np.int32); self.token_page[:N] = idx["token_page"]
        self.token_slot = np.full(n_cap, -1, np.int32); self.token_slot[:N] = idx["token_slot"]
        self.np_cap, self.page_cap, self.n_cap = np_cap, page_cap, n_cap

    def insert(self, k_new, v_new, pos: int, *, seed: int, layer: int, seq: int, head: int, thresh: int,
               parent: int = -1):
        """One insert (step a11).  parent >= 0 replaces the nearest-parent
        search by that parent (a test that follows a device's choice at a
        checked fp32 near-tie); a promoted token ignores it."""
        k = _f64(k_new)
        v = _f64(v_new)
        rc = _load().orc_insert(seed, layer, seq, head, thresh, self.d, self.S, self.M2, _p(k), _p(v), pos, parent,
                                self.np_cap, ctypes.byref(self.n_parents), _p(self.parent_tok),
                                _p(self.parent_keys), _p(self.parent_e),
                                self.page_cap, ctypes.byref(self.n_pages), _p(self.page_parent),
                                _p(self.page_len), _p(self.page_tokens), _p(self.pool_k), _p(self.pool_v),
                                self.n_cap, _p(self.token_parent), _p(self.token_page), _p(self.token_slot))
        _check(rc, "insert")

    def as_dict(self) -> dict:
        Np, P = self.n_parents.value, self.n_pages.value
        return dict(S=self.S, M2=self.M2, parent_tok=self.parent_tok[:Np], parent_keys=self.parent_keys[:Np],
                    parent_e=self.parent_e[:Np], n_pages=P, page_parent=self.page_parent[:P],
                    page_len=self.page_len[:P], page_tokens=self.page_tokens[:P], pool_k=self.pool_k[:P],
                    pool_v=self.pool_v[:P], token_parent=self.token_parent, token_page=self.token_page,
                    token_slot=self.token_slot)


def run_units(fn, items, threads: int | None = None):
    """Run fn(item) over independent units on a thread pool.

    The C calls release the GIL, so units run in parallel on host cores.
    Returns the results in item order and the thread count used.
    """
    items = list(items)
    threads = max(1, min(threads or os.cpu_count() or 1, len(items) or 1))
    _load()
    if threads == 1:
        return [fn(x) for x in items], 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items)), threads
