"""Error behaviour of the C ABI's entry points, as include/ice.h states it:
every argument is checked on the host before anything is launched, and a
bad one returns its status with a message in ice_last_error().

Each case breaks exactly one argument of an otherwise well-formed call whose
pointers are host addresses (a numpy buffer), so the call must return at its
host-side check.  The file runs only where no CUDA device is present: with a
device, a missing check would send those host addresses to a kernel."""
import ctypes

import numpy as np
import pytest
import torch

import semantic_paged_kv_gb300 as ice

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="host addresses stand in for device pointers")

CFG = dict(batch=1, n_q_heads=8, n_kv_heads=2, n_tokens=100)
_BUF = np.zeros(1 << 22, np.uint8)  # 4 MB of host memory behind every fake pointer
_BASE = (_BUF.ctypes.data + 255) & ~255


def _addr(i: int) -> int:
    """The i-th 4 KB slot of the buffer (256-byte aligned)."""
    return _BASE + 4096 * i


def _params(**kw):
    p = ice.Config(**CFG).params()
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _index(**null):
    """An index whose arrays are host addresses; the fields named in `null` are NULL."""
    ix = ice.IceIndex(*[_addr(i) for i in range(len(ice.INDEX_FIELDS))])
    for f in null:
        setattr(ix, f, None)
    return ix


WS = _addr(100)
WS_BYTES = 1 << 20
K, V, Q, O = _addr(400), _addr(500), _addr(600), _addr(700)
SEL, CNT, KB, VB, BL, ERR = _addr(800), _addr(810), _addr(820), _addr(840), _addr(860), _addr(870)


def _build(p=None, k=K, v=V, ix=None, ws=WS, ws_bytes=WS_BYTES):
    return ice.load().ice_build_index(ctypes.byref(p or _params()), k, v, ctypes.byref(ix or _index()), ws, ws_bytes,
                                      ERR, None)


def _select(p=None, ix=None, q=Q, budget=256, sel=SEL, cnt=CNT, max_sel=64):
    return ice.load().ice_select_pages(ctypes.byref(p or _params()), ctypes.byref(ix or _index()), q, budget, sel,
                                       cnt, max_sel, WS, WS_BYTES, ERR, None)


def _step(o=O, kb=KB, vb=VB, bl=BL, q=Q):
    return ice.load().ice_decode_step(ctypes.byref(_params()), ctypes.byref(_index()), q, 256, SEL, CNT, 64, kb, vb,
                                      bl, 0.088, o, WS, WS_BYTES, ERR, None)


def _insert(p=None, k=K):
    return ice.load().ice_insert_tokens(ctypes.byref(p or _params()), ctypes.byref(_index()), k, V, WS, WS_BYTES,
                                        ERR, None)


def _attn(q=Q, kb=KB, max_sel=64):
    return ice.load().ice_sparse_attn_decode(ctypes.byref(_params()), q, kb, VB, BL, CNT, max_sel, 0.088, O, WS,
                                             WS_BYTES, None)


def _noalloc(max_sel=64, o=O):
    return ice.load().ice_sparse_attn_decode_noalloc(ctypes.byref(_params()), Q, KB, VB, BL, CNT, max_sel, 0.088, o,
                                                     None)


def _gather(kb=KB, max_sel=64):
    return ice.load().ice_gather_pages(ctypes.byref(_params()), ctypes.byref(_index()), SEL, CNT, max_sel, kb, VB, BL,
                                       None)


INV, UNS = ice.ICE_ERR_INVALID_ARG, ice.ICE_ERR_UNSUPPORTED
_cfg = ice.Config(**CFG)
WANT = min(_cfg.group * 16, _cfg.page_cap)  # the smallest max_sel a budget of 256 tokens accepts
CASES = [
    ("build: an index array NULL", lambda: _build(ix=_index(page_len=1)), INV, "array pointer is NULL"),
    ("build: K NULL", lambda: _build(k=None), INV, "K must be"),
    ("build: K misaligned", lambda: _build(k=K + 8), INV, "K must be"),
    ("build: V NULL, before any stage", lambda: _build(v=None), INV, "V must be"),
    ("build: workspace misaligned", lambda: _build(ws=WS + 16), INV, "256-byte aligned"),
    ("build: workspace too small", lambda: _build(ws_bytes=1024), INV, "workspace has"),
    ("build: three levels without level-2 arrays", lambda: _build(p=_params(n_levels=3), ix=_index(children=1)),
     INV, "three-level index needs"),
    ("build: parent_keys misaligned", lambda: _build(ix=_misaligned_keys()), INV, "16-byte aligned"),
    ("select: Q NULL", lambda: _select(q=None), INV, "must be non-NULL"),
    ("select: sel_count NULL", lambda: _select(cnt=None), INV, "must be non-NULL"),
    ("select: max_sel below min(g * k, page_cap)", lambda: _select(max_sel=WANT - 1), INV, f"max_sel ({WANT - 1})"),
    ("select: max_sel 0", lambda: _select(max_sel=0), INV, "max_sel must be >= 1"),
    ("select: negative budget", lambda: _select(budget=-16), INV, "budget_tokens must be >= 0"),
    ("select: descent with more than 32 pages a head", lambda: _select(p=_params(n_levels=3), budget=1024,
                                                                      max_sel=512), UNS, "at most 32 pages"),
    ("step: O NULL", lambda: _step(o=None), INV, "non-NULL O"),
    ("step: buffers partly NULL", lambda: _step(vb=None), INV, "all non-NULL or all NULL"),
    ("step: kbuf misaligned", lambda: _step(kb=KB + 4), INV, "16-byte aligned"),
    ("insert: k_new misaligned", lambda: _insert(k=K + 2), INV, "k_new and v_new"),
    ("insert: sink pages", lambda: _insert(p=_params(n_sink=4)), UNS, "sink or window"),
    ("insert: three levels", lambda: _insert(p=_params(n_levels=3)), UNS, "two levels"),
    ("attention: Q NULL", lambda: _attn(q=None), INV, "non-NULL Q"),
    ("attention: kbuf misaligned", lambda: _attn(kb=KB + 8), INV, "16-byte aligned"),
    ("attention (allocation-free): max_sel 0", lambda: _noalloc(max_sel=0), INV, "max_sel must be >= 1"),
    ("attention (allocation-free): O NULL", lambda: _noalloc(o=None), INV, "non-NULL Q"),
    ("gather: kbuf NULL", lambda: _gather(kb=None), INV, "non-NULL buffers"),
    ("gather: max_sel 0", lambda: _gather(max_sel=0), INV, "non-NULL buffers"),
    ("check: error word NULL", lambda: ice.load().ice_check(None, None), INV, "err_dev is NULL"),
]


def _misaligned_keys():
    ix = _index()
    ix.parent_keys = _addr(3) + 8
    return ix


@pytest.mark.parametrize("what,call,status,msg", CASES, ids=[c[0] for c in CASES])
def test_bad_argument_is_refused_on_the_host(what, call, status, msg):
    assert call() == status, ice.load().ice_last_error().decode()
    assert msg in ice.load().ice_last_error().decode()


def test_well_formed_host_checks_pass_up_to_the_device():
    """The same calls with nothing broken get past every host check and stop
    only at the device (there is none here): the cases above fail for the
    argument they break and nothing else."""
    for call in (lambda: _build(), lambda: _select(), lambda: _step(), lambda: _insert(), lambda: _attn(),
                 lambda: _gather()):
        st = call()
        assert st == ice.ICE_ERR_CUDA, (st, ice.load().ice_last_error().decode())


@pytest.mark.parametrize("batch,n_q,n_kv,budget", [(8, 32, 32, 256), (8, 32, 32, 64), (16, 64, 8, 64)])
def test_noalloc_accepts_documented_shapes(batch, n_q, n_kv, budget):
    """The allocation-free attention's capacity check passes the LongChat-7B
    shape at batch 8 (256 units, g = 1) and the Qwen3-32B shape at batch 16
    with budget 64 (its scratch holds only the attention's ticket words and
    partials); without a device the call then fails on its first CUDA call,
    not on capacity."""
    cfg = ice.Config(batch=batch, n_q_heads=n_q, n_kv_heads=n_kv, n_tokens=100000)
    p = cfg.params()
    max_sel = ice.max_selected(cfg, budget)
    st = ice.load().ice_sparse_attn_decode_noalloc(ctypes.byref(p), Q, KB, VB, BL, CNT, max_sel, 0.088, O, None)
    assert st != ice.ICE_ERR_CAPACITY, ice.load().ice_last_error().decode()
    assert st == ice.ICE_ERR_CUDA
