"""The GPU parity checks themselves, on the CPU: do they notice a difference?

The comparison helpers of the GPU tests (parity_util.check_build_unit,
check_decode_unit) are fed the oracle's own index and decode outputs dressed
as device outputs (CPU tensors in the layout the library writes): they must
pass.  Then one output at a time is changed the way a kernel bug would
change it (a token under a farther parent, two tokens swapped between pages,
a pool value, a promoted token, M^2, a selected page, a gathered row, a page
length, the attention output) and the same helper must fail.  Nothing here
runs the CUDA library."""
import types

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import cfg_of, check_build_unit, check_decode_unit

W = workloads.WORKLOADS["tiny"].scaled(n_tokens=700)
BUDGET = 64


class _Run:
    """What the helpers read from a device run, filled from the oracle (one unit)."""

    def __init__(self, n_sink: int = 0, n_window: int = 0):
        w = self.w = W
        self.cfg = cfg_of(w, layer=0, n_sink=n_sink, n_window=n_window)
        self.layer = 0
        self.K, self.V = workloads.batch_kv(w, 0)
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

    def decode(self):
        """(Q, buffers) as ice_decode_step leaves them, from the oracle's decode."""
        cfg, g = self.cfg, self.cfg.group
        Q = workloads.batch_queries(self.w, 0, 0)
        dec = oracle.decode_unit(self.ref, Q[0, :g], BUDGET)
        max_sel, S, d = g * (BUDGET // cfg.page_size) + cfg.n_pos, cfg.page_size, cfg.head_dim
        n = len(dec["sel_pages"])
        sel = torch.full((1, max_sel), -1, dtype=torch.int32)
        sel[0, :n] = torch.from_numpy(dec["sel_pages"])
        kbuf, vbuf = torch.zeros((1, max_sel, S, d)), torch.zeros((1, max_sel, S, d))
        kbuf[0, :n], vbuf[0, :n] = torch.from_numpy(dec["kbuf"]), torch.from_numpy(dec["vbuf"])
        blen = torch.zeros((1, max_sel), dtype=torch.int32)
        blen[0, :n] = torch.from_numpy(np.asarray(dec["buf_len"]))
        O = torch.from_numpy(dec["out"]).float().reshape(1, g, d)
        buf = types.SimpleNamespace(sel_pages=sel, sel_count=torch.tensor([n], dtype=torch.int32), kbuf=kbuf,
                                    vbuf=vbuf, buf_len=blen, O=O)
        return Q, buf


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
