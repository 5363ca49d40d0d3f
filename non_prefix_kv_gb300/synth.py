"""Seeded synthetic inputs shared by the tests, the CPU oracle's callers and the benchmark.

This module draws random numbers and lays out shapes; it holds none of the method's
arithmetic (no RoPE, norm, projection, deviation or selection).  Every array is drawn
from ``numpy.random.default_rng([seed, purpose])`` so the same (seed, purpose) pair gives
the same values on any machine.

Model family: a pre-norm Llama-style decoder without biases (RMSNorm, RoPE, SwiGLU FFN).
Weight layout is "output-major": every projection matrix is stored [out_features,
in_features] row-major, so a projection is ``y = x @ W.T``.

Per-layer tensors:
  attn_norm  [d]                       RMSNorm gain before attention
  wqkv       [(H + 2*Hkv) * hd, d]     rows 0..H*hd-1 = Wq, then Wk (Hkv*hd rows), then Wv
  wo         [d, H * hd]
  ffn_norm   [d]
  w_gate_up  [2 * F, d]                rows 0..F-1 = W_gate, rows F..2F-1 = W_up
  w_down     [d, F]
Model-level: embed [vocab, d], final_norm [d], w_lm [vocab, d].
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np

# purpose codes for default_rng([seed, purpose])
P_WEIGHTS = 1
P_EMBED = 2
P_TOKENS = 3
P_NOISE = 4          # free-form test tensors
P_ORDER = 100        # + request index: per-request chunk order


@dataclass(frozen=True)
class ModelShape:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    rope_base: float = 1.0e4
    rms_eps: float = 1.0e-5
    dtype: str = "f32"            # "f32" or "bf16": storage type on the device
    shared_layers: bool = False   # every layer uses layer 0's weights
    w_std: float = 0.02
    emb_std: float = 1.0

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_width(self) -> int:
        return self.q_width + 2 * self.kv_width

    @property
    def params_per_layer(self) -> int:
        d, F = self.d_model, self.d_ff
        return d * self.qkv_width + self.q_width * d + 3 * d * F


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    chunk_len: int                 # tokens per chunk
    n_distinct: int                # distinct chunk contents in the pool
    order: tuple                   # pool index of each chunk slot, in sequence order
    n_query: int                   # uncached suffix tokens
    ratio: float                   # HKVD recompute ratio r
    check_layer: int = 1
    gradual: bool = False
    n_requests: int = 1
    seed: int = 0
    note: str = ""

    @property
    def n_cached(self) -> int:
        return self.chunk_len * len(self.order)

    @property
    def n_tokens(self) -> int:
        return self.n_cached + self.n_query


TINY_F32 = ModelShape(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64,
                      d_ff=688, vocab=1024, dtype="f32")
LLAMA7B = ModelShape(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32, head_dim=128,
                     d_ff=11008, vocab=32000, dtype="bf16")
LLAMA13B = ModelShape(n_layers=40, d_model=5120, n_heads=40, n_kv_heads=40, head_dim=128,
                      d_ff=13824, vocab=32000, dtype="bf16")
YI34B = ModelShape(n_layers=60, d_model=7168, n_heads=56, n_kv_heads=8, head_dim=128,
                   d_ff=20480, vocab=64000, rope_base=5.0e6, dtype="bf16")

WORKLOADS = {
    # 2 layers, 3 chunks x 128 + 32 query tokens = 416, fp32, r = 15 %
    "tiny_f32": Workload("tiny_f32", TINY_F32, chunk_len=128, n_distinct=3, order=(0, 1, 2),
                         n_query=32, ratio=0.15),
    # one Llama-2-7B-shaped layer's weights run as a shared-weight stack of three layers:
    # layer 0 = pre-check, layer 1 = check (HKVD selection), layer 2 = steady.
    # 6 chunks x 640 + 256 query tokens = 4096, bf16, r = 15 %
    "llama7b_layer_4k": Workload("llama7b_layer_4k",
                                 replace(LLAMA7B, n_layers=3, shared_layers=True),
                                 chunk_len=640, n_distinct=6, order=(0, 1, 2, 3, 4, 5),
                                 n_query=256, ratio=0.15),
    # 32 layers, 8 chunks x 480 + 256; slots 6 and 7 repeat chunks 1 and 3; gradual filtering
    "llama7b_32_4k": Workload("llama7b_32_4k", LLAMA7B, chunk_len=480, n_distinct=6,
                              order=(0, 1, 2, 3, 4, 5, 1, 3), n_query=256, ratio=0.15,
                              gradual=True),
    "llama13b_40_8k": Workload("llama13b_40_8k", LLAMA13B, chunk_len=640, n_distinct=12,
                               order=tuple(range(12)), n_query=512, ratio=0.15),
    "yi34b_60_16k_b4": Workload("yi34b_60_16k_b4", YI34B, chunk_len=640, n_distinct=40,
                                order=tuple(range(24)), n_query=1024, ratio=0.15,
                                n_requests=4),
}


def rng(seed: int, purpose: int) -> np.random.Generator:
    return np.random.default_rng([seed, purpose])


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    Storage conversion only: every value the device sees in a bf16 run is exactly the
    float32 returned here, so both sides start from identical numbers.
    """
    out = np.array(a, dtype=np.float32, copy=True, order="C")
    u = out.view(np.uint32)
    # finite inputs never overflow 32 bits here: |u| <= 0xFF7FFFFF, + 0x8000
    lsb = (u >> 16) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u &= np.uint32(0xFFFF0000)
    return out


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of values that are already bf16-representable."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    a = a.astype(np.float32)
    return round_bf16(a) if dtype == "bf16" else a


def normal(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def make_layer_weights(shape: ModelShape, g: np.random.Generator, gains: str = "ones") -> dict:
    d, F = shape.d_model, shape.d_ff
    s = shape.w_std
    w = {
        "wqkv": _store(normal(g, (shape.qkv_width, d), s), shape.dtype),
        "wo": _store(normal(g, (d, shape.q_width), s), shape.dtype),
        "w_gate_up": _store(normal(g, (2 * F, d), s), shape.dtype),
        "w_down": _store(normal(g, (d, F), s), shape.dtype),
    }
    if gains == "ones":
        w["attn_norm"] = np.ones(d, np.float32)
        w["ffn_norm"] = np.ones(d, np.float32)
    else:  # non-unit gains for unit tests of the norm path
        w["attn_norm"] = _store(1.0 + normal(g, (d,), 0.1), shape.dtype)
        w["ffn_norm"] = _store(1.0 + normal(g, (d,), 0.1), shape.dtype)
    return w


def make_model(shape: ModelShape, seed: int = 0, gains: str = "ones") -> dict:
    """Random-init weights: matrices N(0, w_std), embeddings N(0, emb_std), gains 1."""
    gw = rng(seed, P_WEIGHTS)
    n_distinct_layers = 1 if shape.shared_layers else shape.n_layers
    distinct = [make_layer_weights(shape, gw, gains) for _ in range(n_distinct_layers)]
    layers = [distinct[0 if shape.shared_layers else i] for i in range(shape.n_layers)]
    ge = rng(seed, P_EMBED)
    embed = _store(normal(ge, (shape.vocab, shape.d_model), shape.emb_std), shape.dtype)
    final_norm = np.ones(shape.d_model, np.float32)
    w_lm = _store(normal(gw, (shape.vocab, shape.d_model), shape.w_std), shape.dtype)
    return {"shape": shape, "layers": layers, "embed": embed, "final_norm": final_norm,
            "w_lm": w_lm}


@dataclass
class Request:
    """One blended-prefill request: chunk slots drawn from a pool, then a query suffix."""
    chunk_tokens: List[np.ndarray]     # pool: token ids of each distinct chunk
    order: List[int]                   # pool index per slot
    query_tokens: np.ndarray
    chunk_len: int

    @property
    def tokens(self) -> np.ndarray:
        parts = [self.chunk_tokens[i] for i in self.order] + [self.query_tokens]
        return np.concatenate(parts).astype(np.int32)

    @property
    def n_cached(self) -> int:
        return self.chunk_len * len(self.order)

    @property
    def chunk_starts(self) -> List[int]:
        return [m * self.chunk_len for m in range(len(self.order))]


def make_requests(wl: Workload, seed: Optional[int] = None) -> List[Request]:
    """Token ids uniform in [0, vocab); chunk order shuffled per request when the pool is
    larger than the slot count (the shared-pool workload), else the workload's order."""
    seed = wl.seed if seed is None else seed
    gt = rng(seed, P_TOKENS)
    V = wl.shape.vocab
    pool = [gt.integers(0, V, size=wl.chunk_len, dtype=np.int64).astype(np.int32)
            for _ in range(wl.n_distinct)]
    reqs = []
    for b in range(wl.n_requests):
        q = gt.integers(0, V, size=wl.n_query, dtype=np.int64).astype(np.int32)
        if wl.n_distinct > len(wl.order):
            order = list(rng(seed, P_ORDER + b).permutation(wl.n_distinct)[:len(wl.order)])
        else:
            order = list(wl.order)
        reqs.append(Request(pool, [int(o) for o in order], q, wl.chunk_len))
    return reqs


def test_tensor(shape, seed: int, purpose: int = P_NOISE, std: float = 1.0,
                dtype: str = "f32") -> np.ndarray:
    return _store(normal(rng(seed, purpose), shape, std), dtype)
