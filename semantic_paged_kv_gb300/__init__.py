"""Python binding of the IceCache GB300 library (libice.so, C ABI in include/ice.h).

Argument marshalling only: every function below has the name of the C entry
point it calls, turns torch tensors into raw device pointers and the current
torch CUDA stream into a cudaStream_t, and raises IceError on a non-zero
status.  Every step of the hot path runs in the library's CUDA kernels; there
is no CPU or PyTorch fallback, and importing this package fails loudly when
libice.so has not been built (``python semantic_paged_kv_gb300/build.py``).

PyTorch serves only as the allocator of device memory and as the source of
streams.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libice.so")

ICE_OK, ICE_ERR_INVALID_ARG, ICE_ERR_CUDA, ICE_ERR_OOM, ICE_ERR_CAPACITY, ICE_ERR_TIMEOUT, ICE_ERR_UNSUPPORTED = range(7)
ICE_BF16, ICE_FP32 = 0, 1
HEAD_DIM, PAGE_SIZE = 128, 16


class IceError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[{status}] {msg}")
        self.status = status


class IceParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_tokens", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("n_levels", ctypes.c_int32), ("promote_thresh", ctypes.c_uint64),
                ("seed", ctypes.c_uint64), ("layer", ctypes.c_int32), ("np_cap", ctypes.c_int32),
                ("page_cap", ctypes.c_int32), ("n_cap", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("n_window", ctypes.c_int32)]


INDEX_FIELDS = ["n_parents", "n_pages", "n_indexed", "m2", "parent_tok", "parent_keys", "parent_e", "parent_corr",
                "parent_first_page", "parent_last_page", "parent_n_pages", "page_parent", "page_len", "page_next",
                "page_tokens", "token_parent", "token_page", "token_slot", "pool_k", "pool_v",
                "n_nodes2", "node2", "parent2", "child_start", "children"]


class IceIndex(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in INDEX_FIELDS]


_lib = None


def load() -> ctypes.CDLL:
    """Load libice.so from this package directory (never from elsewhere)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the IceCache CUDA library first "
                          "(python semantic_paged_kv_gb300/build.py or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    pp, pi = ctypes.POINTER(IceParams), ctypes.POINTER(IceIndex)
    sigs = {
        "ice_status_string": ([i32], ctypes.c_char_p),
        "ice_last_error": ([], ctypes.c_char_p),
        "ice_version": ([], ctypes.c_char_p),
        "ice_check": ([P, P], i32),
        "ice_page_bound": ([i32, i32, i32], i32),
        "ice_default_capacities": ([pp], i32),
        "ice_index_bytes": ([pp, i32, ctypes.POINTER(sz)], i32),
        "ice_index_layout": ([pp, i32, P, pi], i32),
        "ice_positional_pages": ([i32, i32, i32, i32], i32),
        "ice_build_workspace_bytes": ([pp, ctypes.POINTER(sz)], i32),
        "ice_build_index": ([pp, P, P, pi, P, sz, P, P], i32),
        "ice_build_lift_promote": ([pp, P, pi, P, sz, P, P], i32),
        "ice_build_assign": ([pp, P, pi, P, sz, P, P], i32),
        "ice_build_assign_simt": ([pp, P, pi, P, sz, P, P], i32),
        "ice_build_pack": ([pp, P, P, pi, P, sz, P, P], i32),
        "ice_build_index_reuse": ([pp, P, P, pi, pi, P, sz, P, P], i32),
        "ice_decode_workspace_bytes": ([pp, i32, i32, ctypes.POINTER(sz)], i32),
        "ice_select_pages": ([pp, pi, P, i32, P, P, i32, P, sz, P, P], i32),
        "ice_gather_pages": ([pp, pi, P, P, i32, P, P, P, P], i32),
        "ice_sparse_attn_decode": ([pp, P, P, P, P, P, i32, f32, P, P, sz, P], i32),
        "ice_decode_step": ([pp, pi, P, i32, P, P, i32, P, P, P, f32, P, P, sz, P, P], i32),
        "ice_decode_plan": ([pp, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
        "ice_sparse_attn_decode_noalloc": ([pp, P, P, P, P, P, i32, f32, P, P], i32),
        "ice_insert_workspace_bytes": ([pp, ctypes.POINTER(sz)], i32),
        "ice_insert_tokens": ([pp, pi, P, P, P, sz, P, P], i32),
        "ice_host_pool_create": ([sz, sz, i32, ctypes.POINTER(P)], i32),
        "ice_host_pool_destroy": ([P], i32),
        "ice_host_pool_pointers": ([P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P)], i32),
        "ice_host_pool_staging_bytes": ([pp, i32], sz),
        "ice_host_pool_gather_h2d": ([P, pp, P, P, P, i32, P, sz, P], i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def exported_symbols() -> list[str]:
    return ["ice_status_string", "ice_last_error", "ice_version", "ice_check", "ice_page_bound", "ice_positional_pages",
            "ice_default_capacities", "ice_index_bytes", "ice_index_layout",
            "ice_build_workspace_bytes", "ice_build_index", "ice_build_lift_promote", "ice_build_assign",
            "ice_build_assign_simt", "ice_build_pack", "ice_build_index_reuse", "ice_decode_workspace_bytes",
            "ice_select_pages",
            "ice_gather_pages", "ice_sparse_attn_decode", "ice_sparse_attn_decode_noalloc", "ice_decode_step",
            "ice_decode_plan",
            "ice_insert_workspace_bytes", "ice_insert_tokens", "ice_host_pool_create", "ice_host_pool_destroy",
            "ice_host_pool_pointers", "ice_host_pool_staging_bytes", "ice_host_pool_gather_h2d"]


# ----------------------------------------------------------- marshalling --
def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int):
    if status != ICE_OK:
        lib = load()
        raise IceError(status, lib.ice_last_error().decode())


def promote_threshold(p: float) -> int:
    return int(math.floor(p * 4294967296.0))


@dataclasses.dataclass
class Config:
    """Shapes of one layer's index (mirrors ice_params)."""
    batch: int
    n_q_heads: int
    n_kv_heads: int
    n_tokens: int
    dtype: int = ICE_BF16
    promote_p: float = 1.0 / 16.0
    seed: int = 0
    layer: int = 0
    np_cap: int | None = None
    page_cap: int | None = None
    n_cap: int | None = None
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    n_levels: int = 2
    n_sink: int = 0    # first tokens kept as positional pages (not indexed)
    n_window: int = 0  # last tokens of the build kept as positional pages (not indexed)

    def __post_init__(self):
        if self.n_cap is None:
            self.n_cap = max(self.n_tokens, 1)
        if self.np_cap is None:
            # the library's default capacities (ice_default_capacities)
            d = self._params(np_cap=0, page_cap=0)
            _check(load().ice_default_capacities(ctypes.byref(d)))
            self.np_cap = d.np_cap
            if self.page_cap is None:
                self.page_cap = d.page_cap
        if self.page_cap is None:
            self.page_cap = max(1, ice_page_bound(self.n_cap, self.np_cap, self.page_size) + self.n_pos)

    @property
    def n_pos(self) -> int:
        """Positional (sink and window) pages of a unit."""
        return int(load().ice_positional_pages(self.n_tokens, self.n_sink, self.n_window, self.page_size))

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def units(self) -> int:
        return self.batch * self.n_kv_heads

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == ICE_BF16 else torch.float32

    def params(self) -> IceParams:
        return self._params()

    def _params(self, **over) -> IceParams:
        f = {**dict(np_cap=self.np_cap, page_cap=self.page_cap, n_cap=self.n_cap), **over}
        return IceParams(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim, self.n_tokens, self.page_size,
                         self.dtype, self.n_levels, promote_threshold(self.promote_p), self.seed, self.layer,
                         f["np_cap"], f["page_cap"], f["n_cap"], self.n_sink, self.n_window)


class Index:
    """Device arrays of one layer's index in one slab of device memory
    allocated with torch (caller-owned memory in the C ABI's terms), sized
    by ice_index_bytes and carved by ice_index_layout; each array is a torch
    view into the slab.  With a host pool the pool arrays are the pool's
    device-mapped pointers instead."""

    def __init__(self, cfg: Config, device="cuda", host_pool=None):
        U, Np, Pc, Nc, S, d = cfg.units, cfg.np_cap, cfg.page_cap, cfg.n_cap, cfg.page_size, cfg.head_dim
        i32, dt = torch.int32, cfg.torch_dtype
        shapes = {"n_parents": (i32, (U,)), "n_pages": (i32, (U,)), "n_indexed": (i32, (U,)),
                  "m2": (torch.float64, (U,)), "parent_tok": (i32, (U, Np)), "parent_keys": (dt, (U, Np, d)),
                  "parent_e": (torch.float32, (U, Np)), "parent_corr": (torch.float32, (U, Np)),
                  "parent_first_page": (i32, (U, Np)), "parent_last_page": (i32, (U, Np)),
                  "parent_n_pages": (i32, (U, Np)), "page_parent": (i32, (U, Pc)), "page_len": (i32, (U, Pc)),
                  "page_next": (i32, (U, Pc)), "page_tokens": (i32, (U, Pc, S)), "token_parent": (i32, (U, Nc)),
                  "token_page": (i32, (U, Nc)), "token_slot": (i32, (U, Nc)), "pool_k": (dt, (U, Pc, S, d)),
                  "pool_v": (dt, (U, Pc, S, d)), "n_nodes2": (i32, (U,)), "node2": (i32, (U, Np)),
                  "parent2": (i32, (U, Np)), "child_start": (i32, (U, Np + 1)), "children": (i32, (U, Np))}
        self.cfg = cfg
        params = cfg.params()
        with_pool = host_pool is None
        n = ctypes.c_size_t(0)
        _check(load().ice_index_bytes(ctypes.byref(params), int(with_pool), ctypes.byref(n)))
        self.slab = torch.zeros(n.value, dtype=torch.uint8, device=device)
        st = IceIndex()
        _check(load().ice_index_layout(ctypes.byref(params), int(with_pool), self.slab.data_ptr(), ctypes.byref(st)))
        base = self.slab.data_ptr()
        for f in INDEX_FIELDS:
            ptr = getattr(st, f)
            if ptr is None:
                setattr(self, f, None)
                continue
            t, shape = shapes[f]
            off = ptr - base
            nb = math.prod(shape) * torch.empty((), dtype=t).element_size()
            assert 0 <= off and off + nb <= n.value
            setattr(self, f, self.slab[off:off + nb].view(t).view(shape))
        if host_pool is not None:  # pages live in the pinned host pool (device-mapped pointers)
            self.host_pool = host_pool
            st.pool_k, st.pool_v = host_pool.k_dev, host_pool.v_dev
        self._struct = st

    @property
    def struct(self) -> IceIndex:
        return self._struct


# ------------------------------------------------------- entry points -----
def ice_version() -> str:
    return load().ice_version().decode()


def ice_status_string(s: int) -> str:
    return load().ice_status_string(s).decode()


def ice_page_bound(n_tokens: int, n_parents: int, page_size: int = PAGE_SIZE) -> int:
    return int(load().ice_page_bound(n_tokens, n_parents, page_size))


def ice_check(err_dev, stream=None) -> int:
    """Synchronise, read and clear the device error word; returns its status."""
    return int(load().ice_check(_ptr(err_dev), _stream(stream)))


def ice_build_workspace_bytes(params: IceParams) -> int:
    n = ctypes.c_size_t(0)
    _check(load().ice_build_workspace_bytes(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def ice_decode_workspace_bytes(params: IceParams, budget_tokens: int, max_sel: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().ice_decode_workspace_bytes(ctypes.byref(params), budget_tokens, max_sel, ctypes.byref(n)))
    return n.value


def _build_call(name, params, K, V, index, ws, err, stream):
    fn = getattr(load(), name)
    ix = index.struct if isinstance(index, Index) else index
    args = [ctypes.byref(params), _ptr(K)]
    if V is not None:
        args.append(_ptr(V))
    args += [ctypes.byref(ix), _ptr(ws), ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0,
             _ptr(err), _stream(stream)]
    _check(fn(*args))


def ice_build_index(params, K, V, index, ws, err, stream=None):
    _build_call("ice_build_index", params, K, V, index, ws, err, stream)


def ice_build_lift_promote(params, K, index, ws, err, stream=None):
    _build_call("ice_build_lift_promote", params, K, None, index, ws, err, stream)


def ice_build_assign(params, K, index, ws, err, stream=None):
    _build_call("ice_build_assign", params, K, None, index, ws, err, stream)


def ice_build_assign_simt(params, K, index, ws, err, stream=None):
    _build_call("ice_build_assign_simt", params, K, None, index, ws, err, stream)


def ice_build_pack(params, K, V, index, ws, err, stream=None):
    _build_call("ice_build_pack", params, K, V, index, ws, err, stream)


def ice_build_index_reuse(params, K, V, prev, index, ws, err, stream=None):
    """Build `index` for this layer's K, V on `prev`'s parents, assignment and
    pages (the inter-layer index reuse)."""
    px = prev.struct if isinstance(prev, Index) else prev
    ix = index.struct if isinstance(index, Index) else index
    _check(load().ice_build_index_reuse(ctypes.byref(params), _ptr(K), _ptr(V), ctypes.byref(px), ctypes.byref(ix),
                                        _ptr(ws), _nbytes(ws), _ptr(err), _stream(stream)))


def ice_insert_workspace_bytes(params: IceParams) -> int:
    n = ctypes.c_size_t(0)
    _check(load().ice_insert_workspace_bytes(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def ice_insert_tokens(params, index, k_new, v_new, ws, err, stream=None):
    ix = index.struct if isinstance(index, Index) else index
    _check(load().ice_insert_tokens(ctypes.byref(params), ctypes.byref(ix), _ptr(k_new), _ptr(v_new), _ptr(ws),
                                    _nbytes(ws), _ptr(err), _stream(stream)))


class HostPool:
    """The library-owned pinned host page pool (ice_host_pool_*)."""

    def __init__(self, cfg: "Config", max_sel: int, n_threads: int = 8):
        esz = 2 if cfg.dtype == ICE_BF16 else 4
        self.cfg = cfg
        self.pool_bytes = cfg.units * cfg.page_cap * cfg.page_size * cfg.head_dim * esz
        self.staging_bytes = int(load().ice_host_pool_staging_bytes(ctypes.byref(cfg.params()), max_sel))
        h = ctypes.c_void_p()
        _check_plain(load().ice_host_pool_create(self.pool_bytes, self.staging_bytes, n_threads, ctypes.byref(h)))
        self.handle = h
        kd, vd, kh, vh = (ctypes.c_void_p() for _ in range(4))
        _check_plain(load().ice_host_pool_pointers(h, ctypes.byref(kd), ctypes.byref(vd), ctypes.byref(kh),
                                                   ctypes.byref(vh)))
        self.k_dev, self.v_dev, self.k_host, self.v_host = kd.value, vd.value, kh.value, vh.value

    def host_array(self, which: str):
        """numpy view of a host pool [U, page_cap, S, d] (storage dtype bits)."""
        import numpy as np
        cfg = self.cfg
        n = self.pool_bytes // (2 if cfg.dtype == ICE_BF16 else 4)
        ct = ctypes.c_uint16 if cfg.dtype == ICE_BF16 else ctypes.c_float
        ptr = ctypes.cast(self.k_host if which == "k" else self.v_host, ctypes.POINTER(ct))
        return np.ctypeslib.as_array(ptr, shape=(n,)).reshape(cfg.units, cfg.page_cap, cfg.page_size, cfg.head_dim)

    def close(self):
        if self.handle is not None:
            load().ice_host_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check_plain(status: int):
    if status != ICE_OK:
        raise IceError(status, ice_status_string(status))


def ice_host_pool_gather_h2d(pool: HostPool, params, sel_pages_host, sel_count_host, page_len_host, max_sel, dst,
                             stream=None):
    """sel_pages_host etc. are host (CPU) tensors; dst a device uint8 tensor."""
    _check_plain(load().ice_host_pool_gather_h2d(pool.handle, ctypes.byref(params), _ptr(sel_pages_host),
                                                 _ptr(sel_count_host), _ptr(page_len_host), max_sel, _ptr(dst),
                                                 _nbytes(dst), _stream(stream)))


def _nbytes(t) -> int:
    return t.numel() * t.element_size() if isinstance(t, torch.Tensor) else 0


def ice_select_pages(params, index, Q, budget_tokens, sel_pages, sel_count, ws, err, stream=None):
    ix = index.struct if isinstance(index, Index) else index
    _check(load().ice_select_pages(ctypes.byref(params), ctypes.byref(ix), _ptr(Q), budget_tokens, _ptr(sel_pages),
                                   _ptr(sel_count), sel_pages.shape[-1], _ptr(ws), _nbytes(ws), _ptr(err),
                                   _stream(stream)))


def ice_gather_pages(params, index, sel_pages, sel_count, kbuf, vbuf, buf_len, stream=None):
    ix = index.struct if isinstance(index, Index) else index
    _check(load().ice_gather_pages(ctypes.byref(params), ctypes.byref(ix), _ptr(sel_pages), _ptr(sel_count),
                                   sel_pages.shape[-1], _ptr(kbuf), _ptr(vbuf), _ptr(buf_len), _stream(stream)))


def ice_sparse_attn_decode(params, Q, kbuf, vbuf, buf_len, sel_count, scale, O, ws, stream=None):
    _check(load().ice_sparse_attn_decode(ctypes.byref(params), _ptr(Q), _ptr(kbuf), _ptr(vbuf), _ptr(buf_len),
                                         _ptr(sel_count), buf_len.shape[-1], float(scale), _ptr(O), _ptr(ws),
                                         _nbytes(ws), _stream(stream)))


def ice_sparse_attn_decode_noalloc(params, Q, kbuf, vbuf, buf_len, sel_count, scale, O, stream=None):
    """ice_sparse_attn_decode without a workspace: scratch in the library's
    static device array (see ice.h for its limit and sharing rules)."""
    _check(load().ice_sparse_attn_decode_noalloc(ctypes.byref(params), _ptr(Q), _ptr(kbuf), _ptr(vbuf), _ptr(buf_len),
                                                 _ptr(sel_count), buf_len.shape[-1], float(scale), _ptr(O),
                                                 _stream(stream)))


def ice_decode_step(params, index, Q, budget_tokens, sel_pages, sel_count, kbuf, vbuf, buf_len, scale, O, ws, err,
                    stream=None):
    ix = index.struct if isinstance(index, Index) else index
    _check(load().ice_decode_step(ctypes.byref(params), ctypes.byref(ix), _ptr(Q), budget_tokens, _ptr(sel_pages),
                                  _ptr(sel_count), sel_pages.shape[-1], _ptr(kbuf), _ptr(vbuf), _ptr(buf_len),
                                  float(scale), _ptr(O), _ptr(ws), _nbytes(ws), _ptr(err), _stream(stream)))


(ICE_PLAN_CLUSTER_BF16, ICE_PLAN_CLUSTER, ICE_PLAN_SCORE_SELECT, ICE_PLAN_SCORE_TOPK, ICE_PLAN_SIMT,
 ICE_PLAN_DESCENT) = 1, 2, 3, 4, 5, 6
ICE_PLAN_ATTN_MMA, ICE_PLAN_ATTN_SIMT = 1, 2


def ice_decode_plan(params, budget_tokens: int, max_sel: int) -> tuple[int, int]:
    """(step plan, attention plan) of ice_decode_step for this shape."""
    a, b = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load().ice_decode_plan(ctypes.byref(params), budget_tokens, max_sel, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


# ----------------------------------------------------- buffer helpers -----
def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled, 256-byte aligned device workspace (torch's allocator
    aligns to 512); decode workspaces must start zeroed (see ice.h)."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def max_selected(cfg: Config, budget_tokens: int) -> int:
    k = -(-budget_tokens // cfg.page_size)
    return max(1, min(cfg.group * k + cfg.n_pos, cfg.page_cap))


class DecodeBuffers:
    """Outputs of one decode step for a config and budget."""

    def __init__(self, cfg: Config, budget_tokens: int, device="cuda"):
        U, S, d = cfg.units, cfg.page_size, cfg.head_dim
        self.max_sel = max_selected(cfg, budget_tokens)
        self.sel_pages = torch.full((U, self.max_sel), -1, dtype=torch.int32, device=device)
        self.sel_count = torch.zeros(U, dtype=torch.int32, device=device)
        self.kbuf = torch.zeros((U, self.max_sel, S, d), dtype=cfg.torch_dtype, device=device)
        self.vbuf = torch.zeros((U, self.max_sel, S, d), dtype=cfg.torch_dtype, device=device)
        self.buf_len = torch.zeros((U, self.max_sel), dtype=torch.int32, device=device)
        self.O = torch.zeros((cfg.batch, cfg.n_q_heads, d), dtype=torch.float32, device=device)
        self.ws = workspace(ice_decode_workspace_bytes(cfg.params(), budget_tokens, self.max_sel), device)
