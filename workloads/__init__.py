"""Seeded synthetic workloads for the IceCache hot path.

This module only draws input data (keys, values, queries, new tokens for the
incremental insert) and describes workload shapes.  It holds none of the
method's arithmetic, so both the CUDA library's tests/benchmark and the CPU
oracle consume the same arrays from here.

Every array is drawn in float32 from numpy's PCG64 and rounded once to the
workload's storage dtype (bf16 round-to-nearest-even, or kept as fp32); the
returned float32 arrays hold exactly the stored values, so widening them to
double for the oracle is exact.

Shapes follow the model head layouts the IceCache pages evaluate
(Llama-3.1-8B, Mistral-7B, LongChat-7B, Qwen3-32B) with synthetic Gaussian-
mixture keys standing in for real KV caches (no model weights or datasets are
used).
"""
from __future__ import annotations

import dataclasses

import numpy as np

HEAD_DIM = 128
PAGE_SIZE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    n_tokens: int
    layers: int
    dtype: str               # "bf16" | "fp32"
    centres: int             # Gaussian-mixture centres per KV head
    budgets: tuple           # token budgets
    seed: int
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    promote_p: float = 1.0 / 16.0
    spread: float = 0.3      # key / query spread around a centre
    needle: bool = False     # plant one key aligned with a query head
    lognormal_sigma: float = 0.0  # per-token key-norm scale exp(sigma * xi)
    decode_steps: int = 1    # decode steps (each with one inserted token when > 1)
    host_pool: bool = False  # page pool held in pinned host memory

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def units(self) -> int:
        return self.batch * self.n_kv_heads

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 1, 2048, 1, "fp32", 32, (64,), seed=0),
    "llama31_8b_16k": Workload("llama31_8b_16k", 1, 32, 8, 16384, 1, "bf16", 256, (64, 128, 256),
                               seed=1, needle=True),
    "mistral_7b_36k": Workload("mistral_7b_36k", 1, 32, 8, 36864, 32, "bf16", 1024, (256,), seed=2,
                               decode_steps=128),
    "longchat_7b_100k": Workload("longchat_7b_100k", 1, 32, 32, 100000, 32, "bf16", 4096, (64, 256),
                                 seed=3, lognormal_sigma=0.5),
    "qwen3_32b_100k": Workload("qwen3_32b_100k", 16, 64, 8, 100000, 64, "bf16", 4096, (256,), seed=4,
                               host_pool=True),
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def _rng(w: Workload, layer: int, seq: int, head: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, layer, seq, head, stream]))


def unit_centres(w: Workload, layer: int, seq: int, head: int) -> np.ndarray:
    """The mixture centres of one (seq, layer, KV head), N(0, I)."""
    return _rng(w, layer, seq, head, 0).standard_normal((w.centres, w.head_dim), dtype=np.float32)


def unit_kv(w: Workload, layer: int, seq: int, head: int, n_tokens: int | None = None):
    """Keys and values of one unit: K = centre + spread * N(0,I) (times a
    log-normal per-token scale when set), V ~ N(0, I).  Returns float32 arrays
    holding storage-dtype values, shape [N, d]."""
    N = w.n_tokens if n_tokens is None else n_tokens
    C = unit_centres(w, layer, seq, head)
    r = _rng(w, layer, seq, head, 1)
    lab = r.integers(0, w.centres, size=N)
    K = C[lab] + w.spread * r.standard_normal((N, w.head_dim), dtype=np.float32)
    if w.lognormal_sigma > 0:
        K *= np.exp(w.lognormal_sigma * r.standard_normal((N, 1), dtype=np.float32))
    V = r.standard_normal((N, w.head_dim), dtype=np.float32)
    if w.needle and N > 0:
        q0 = unit_queries(w, layer, seq, head)[0].astype(np.float64)
        qhat = q0 / np.linalg.norm(q0)
        pos = int(needle_position(w, layer, seq, head, N))
        med = float(np.median(np.linalg.norm(K.astype(np.float64), axis=1)))
        K[pos] = (2.0 * med * qhat + 0.05 * r.standard_normal(w.head_dim)).astype(np.float32)
    return to_storage(K, w.dtype), to_storage(V, w.dtype)


def needle_position(w: Workload, layer: int, seq: int, head: int, n_tokens: int | None = None) -> int:
    N = w.n_tokens if n_tokens is None else n_tokens
    return int(_rng(w, layer, seq, head, 3).integers(0, max(N, 1)))


def unit_queries(w: Workload, layer: int, seq: int, head: int, step: int = 0) -> np.ndarray:
    """The g query heads of one KV group: each a seeded centre of the unit's
    mixture plus spread * N(0, I).  Returns [g, d] float32 storage values."""
    C = unit_centres(w, layer, seq, head)
    r = _rng(w, layer, seq, head, 100 + step)
    lab = r.integers(0, w.centres, size=w.group)
    q = C[lab] + w.spread * r.standard_normal((w.group, w.head_dim), dtype=np.float32)
    return to_storage(q, w.dtype)


def unit_new_tokens(w: Workload, layer: int, seq: int, head: int, steps: int):
    """Keys/values of `steps` new tokens drawn from the same mixture."""
    C = unit_centres(w, layer, seq, head)
    r = _rng(w, layer, seq, head, 2)
    lab = r.integers(0, w.centres, size=steps)
    K = C[lab] + w.spread * r.standard_normal((steps, w.head_dim), dtype=np.float32)
    if w.lognormal_sigma > 0:
        K *= np.exp(w.lognormal_sigma * r.standard_normal((steps, 1), dtype=np.float32))
    V = r.standard_normal((steps, w.head_dim), dtype=np.float32)
    return to_storage(K, w.dtype), to_storage(V, w.dtype)


def batch_kv(w: Workload, layer: int = 0):
    """K, V for all units of one layer: float32 [B, Hkv, N, d]."""
    K = np.empty((w.batch, w.n_kv_heads, w.n_tokens, w.head_dim), np.float32)
    V = np.empty_like(K)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            K[b, h], V[b, h] = unit_kv(w, layer, b, h)
    return K, V


def batch_queries(w: Workload, layer: int = 0, step: int = 0) -> np.ndarray:
    """Q for all query heads: float32 [B, Hq, d]; query head h*g + i belongs
    to KV head h."""
    Q = np.empty((w.batch, w.n_q_heads, w.head_dim), np.float32)
    g = w.group
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            Q[b, h * g:(h + 1) * g] = unit_queries(w, layer, b, h, step)
    return Q


# ------------------------------------------------------------------------------
# Device-side draws of the same mixtures, for timing at full size (100k-token
# contexts, batch 16), where drawing on the host takes tens of seconds.  Same
# recipe as unit_kv / unit_queries (per-unit N(0, I) centres, spread noise,
# log-normal norms when set, N(0, I) values), drawn from torch's generator on
# the device instead of PCG64, so the values differ from the host draws.  The
# timing runs use them, and so do the full-size parity tests, which copy the
# units they check back to the host for the oracle.
def _torch_gen(w: Workload, layer: int, stream: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(((w.seed * 1_000_003 + layer) * 1_000_003 + stream) & 0x7FFFFFFFFFFFFFFF)
    return g


def batch_kv_device(w: Workload, layer: int = 0, device="cuda"):
    """K, V [B, Hkv, N, d] in the workload's storage dtype, drawn on `device`."""
    import torch
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    B, H, N, d = w.batch, w.n_kv_heads, w.n_tokens, w.head_dim
    g = _torch_gen(w, layer, 0, device)
    C = torch.randn((B * H, w.centres, d), generator=g, device=device)
    K = torch.empty((B * H, N, d), dtype=dt, device=device)
    V = torch.empty((B * H, N, d), dtype=dt, device=device)
    for u in range(B * H):  # one unit at a time keeps the fp32 temporaries small
        lab = torch.randint(0, w.centres, (N,), generator=g, device=device)
        k = C[u][lab] + w.spread * torch.randn((N, d), generator=g, device=device)
        if w.lognormal_sigma > 0:
            k *= torch.exp(w.lognormal_sigma * torch.randn((N, 1), generator=g, device=device))
        K[u] = k.to(dt)
        V[u] = torch.randn((N, d), generator=g, device=device).to(dt)
    return K.view(B, H, N, d), V.view(B, H, N, d), C


def batch_queries_device(w: Workload, centres, layer: int = 0, device="cuda"):
    """Q [B, Hq, d]: query head h*g + i is a centre of KV head h's mixture
    plus spread noise (centres as returned by batch_kv_device)."""
    import torch
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    B, H, gq, d = w.batch, w.n_kv_heads, w.group, w.head_dim
    g = _torch_gen(w, layer, 1, device)
    lab = torch.randint(0, w.centres, (B * H, gq), generator=g, device=device)
    q = torch.gather(centres, 1, lab[..., None].expand(-1, -1, d)) + \
        w.spread * torch.randn((B * H, gq, d), generator=g, device=device)
    return q.reshape(B, H * gq, d).to(dt)
