"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
on seeded workloads and compare every output with the CPU oracle.

Comparison rules (the reading of the pages' tolerance statement):
  * integer outputs (promotion, page tables, selections, copies) are compared
    bit-exactly;
  * a parent assignment may differ from the oracle's only at a near-tie: the
    oracle's lifted squared distance to the GPU's parent exceeds the best one
    by at most 2e-6 * M^2 (a 1e-6 relative tie in the lifted inner product
    k'.p', whose scale is |k'|^2 = M^2);
  * a selected page set may differ only through parents whose scores lie
    within 1e-6 * |q| * M of the k-th page's score;
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


class DeviceRun:
    """One layer built and decoded on the GPU, with host copies of everything."""

    def __init__(self, w: workloads.Workload, layer: int = 0, assign: str = "auto", **cfg_kw):
        self.w = w
        self.cfg = cfg_of(w, layer=layer, **cfg_kw)
        self.layer = layer
        self.K, self.V = workloads.batch_kv(w, layer)
        dt = self.cfg.torch_dtype
        self.Kd, self.Vd = to_dev(self.K, dt), to_dev(self.V, dt)
        self.idx = ice.Index(self.cfg)
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
        self.h = {f: getattr(self.idx, f).float().cpu().numpy() if f == "parent_keys" else getattr(self.idx, f).cpu().numpy()
                  for f in ice.INDEX_FIELDS if f not in ("pool_k", "pool_v")}

    def pool(self, u):
        P = int(self.h["n_pages"][u])
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

    def __init__(self, w: workloads.Workload, layer: int = 0, **cfg_kw):
        self.w = w
        self.cfg = cfg_of(w, layer=layer, **cfg_kw)
        self.layer = layer
        self.Kd, self.Vd, self.C = workloads.batch_kv_device(w, layer)
        self.K, self.V = _UnitArrays(self.Kd), _UnitArrays(self.Vd)
        self.idx = ice.Index(self.cfg)
        self.params = self.cfg.params()
        self.ws = ice.workspace(ice.ice_build_workspace_bytes(self.params))
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ice.ice_build_index(self.params, self.Kd, self.Vd, self.idx, self.ws, self.err)
        self.status = ice.ice_check(self.err)
        self.h = {f: _UnitRows(getattr(self.idx, f)) for f in ice.INDEX_FIELDS if f not in ("pool_k", "pool_v")}

    def queries(self, step: int = 0):
        assert step == 0
        Qd = workloads.batch_queries_device(self.w, self.C, self.layer)
        return Qd.float().cpu().numpy(), Qd


# ------------------------------------------------------------ comparisons --
def lifted_d2(K, e, j, t):
    """Oracle-precision lifted squared distance between tokens j and t."""
    dk = K[j].astype(np.float64) - K[t].astype(np.float64)
    return float(dk @ dk + (e[j] - e[t]) ** 2)


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
    mism = js[tp_gpu[js] != tp_ora[js]]
    for j in mism:
        a = lifted_d2(K, e, j, pt[tp_gpu[j]])
        o = lifted_d2(K, e, j, pt[tp_ora[j]])
        assert a - o <= 2 * TIE_REL * M2, (u, j, tp_gpu[j], tp_ora[j], a, o)
    assert len(mism) <= max(2, len(js) // 2000), (u, len(mism))
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
    head, union = oracle.select(q, pkeys, H["page_parent"][u, :Ps], k_pages)
    union = np.concatenate([union, np.arange(Ps, P, dtype=union.dtype)])
    if not np.array_equal(got, union):
        # near-tie protocol: differences only through parents tied with the boundary
        _, M2, _ = oracle.lift(run.K[b, h].astype(np.float64))
        allowed = set(union.tolist())
        required = set()
        for hh in range(g):
            s = pkeys @ q[hh]
            ps = s[H["page_parent"][u, :Ps]]
            kth = ps[head[hh][min(k_pages, Ps) - 1]]
            tol = TIE_REL * np.linalg.norm(q[hh]) * np.sqrt(M2)
            near = np.where(np.abs(ps - kth) <= tol)[0]
            allowed |= set(near.tolist())
            required |= set(np.where(ps > kth + tol)[0].tolist())
        gs = set(got.tolist())
        assert required <= gs and gs <= allowed, (u, sorted(gs ^ set(union.tolist())))
    assert np.all(np.diff(got) > 0)
    # gather: exact copies of the selected pages
    gi = torch.as_tensor(got, dtype=torch.long, device=buf.kbuf.device)
    pk_sel = run.idx.pool_k[u].index_select(0, gi).float().cpu().numpy()
    pv_sel = run.idx.pool_v[u].index_select(0, gi).float().cpu().numpy()
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
