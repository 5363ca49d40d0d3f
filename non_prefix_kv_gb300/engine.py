"""Request driver for blended prefill: device-resident weights, the chunk-KV pool, and the
per-layer loop of the CacheBlend pipeline (CacheBlend explainer,
0h-n0.github.io/posts/paper-2312-03052, §Pipelining: fetch a layer's chunk KV, run the
layer's partial prefill, synchronize).  Marshalling and host bookkeeping only: every
arithmetic step runs in libcacheblend's kernels."""
from __future__ import annotations

import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import binding as B
from .synth import ModelShape


def torch_dtype(shape: ModelShape):
    return torch.bfloat16 if shape.dtype == "bf16" else torch.float32


def make_dims(shape: ModelShape) -> B.cb_dims:
    return B.cb_dims(shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.d_ff, shape.vocab,
                     float(shape.rope_base), float(shape.rms_eps), B.CB_BF16 if shape.dtype == "bf16" else B.CB_F32)


class DeviceModel:
    """Weights on the device in the shape's storage dtype."""

    def __init__(self, shape: ModelShape, layers: List[dict], embed, final_norm, w_lm, unit_gains=None):
        """unit_gains: per layer (attn_norm, ffn_norm) flags, True where that norm's gains are
        all one; the library is then given NULL for it (unit gains), which lets the bf16 path
        fold the norm into the neighbouring GEMMs."""
        self.shape = shape
        self.dims = make_dims(shape)
        self.layers = layers
        self.embed, self.final_norm, self.w_lm = embed, final_norm, w_lm
        unit_gains = unit_gains or [(False, False)] * len(layers)
        self.layers_c = [B.cb_layer_w(0 if ug[0] else l["attn_norm"].data_ptr(), l["wqkv"].data_ptr(),
                                      l["wo"].data_ptr(), 0 if ug[1] else l["ffn_norm"].data_ptr(),
                                      l["w_gate_up"].data_ptr(), l["w_down"].data_ptr())
                         for l, ug in zip(layers, unit_gains)]

    @classmethod
    def from_host(cls, model: dict, device="cuda") -> "DeviceModel":
        """Upload a synth.make_model() dict (values already representable in the dtype)."""
        shape = model["shape"]
        dt = torch_dtype(shape)

        def up(a):
            return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device).to(dt)

        cache = {}
        layers = []
        for l in model["layers"]:
            if id(l) not in cache:
                cache[id(l)] = {k: up(v) for k, v in l.items()}
            layers.append(cache[id(l)])
        unit = [(bool(np.all(np.asarray(l["attn_norm"]) == 1)), bool(np.all(np.asarray(l["ffn_norm"]) == 1)))
                for l in model["layers"]]
        return cls(shape, layers, up(model["embed"]), up(model["final_norm"]), up(model["w_lm"]), unit)

    @classmethod
    def random_on_device(cls, shape: ModelShape, seed: int = 0, device="cuda") -> "DeviceModel":
        """Random-init weights drawn on the device (seeded torch CUDA generator) for shapes
        too large to draw on the host: matrices N(0, w_std), embeddings N(0, emb_std),
        gains 1."""
        dt = torch_dtype(shape)
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000003 + 1)
        d, F = shape.d_model, shape.d_ff

        def normal(*sz, std):
            return (torch.randn(*sz, generator=g, device=device, dtype=torch.float32) * std).to(dt)

        n_distinct = 1 if shape.shared_layers else shape.n_layers
        distinct = []
        for _ in range(n_distinct):
            distinct.append({
                "attn_norm": torch.ones(d, device=device, dtype=dt),
                "wqkv": normal(shape.qkv_width, d, std=shape.w_std),
                "wo": normal(d, shape.q_width, std=shape.w_std),
                "ffn_norm": torch.ones(d, device=device, dtype=dt),
                "w_gate_up": normal(2 * F, d, std=shape.w_std),
                "w_down": normal(d, F, std=shape.w_std),
            })
        layers = [distinct[0 if shape.shared_layers else i] for i in range(shape.n_layers)]
        embed = normal(shape.vocab, d, std=shape.emb_std)
        w_lm = normal(shape.vocab, d, std=shape.w_std)
        # the norm gains are ones by construction
        return cls(shape, layers, embed, torch.ones(d, device=device, dtype=dt), w_lm,
                   [(True, True)] * shape.n_layers)


@dataclass
class ChunkPool:
    """Per-layer K/V of every distinct chunk, precomputed alone at local positions 0..n-1."""
    k: List[torch.Tensor]          # per layer [rows, Hkv*hd]
    v: List[torch.Tensor]
    offsets: List[int]             # first pool row of each chunk
    lens: List[int]


    def layer_tensors(self, l: int) -> List[torch.Tensor]:
        return [self.k[l], self.v[l]]


@dataclass
class ChunkPoolQ8:
    """The chunk-KV pool as 8-bit per-channel codes (CacheGen explainer,
    0h-n0.github.io/posts/paper-2401-12191, §Step 1): per layer the K and V codes
    [rows, Hkv*hd] uint8 and, per chunk, the scale/zero of every channel [n_chunks, Hkv*hd]."""
    kq: List[torch.Tensor]
    vq: List[torch.Tensor]
    ks: List[torch.Tensor]
    kz: List[torch.Tensor]
    vs: List[torch.Tensor]
    vz: List[torch.Tensor]
    offsets: List[int]
    lens: List[int]

    @classmethod
    def from_pool(cls, pool: ChunkPool, dims: B.cb_dims) -> "ChunkPoolQ8":
        W = pool.k[0].shape[1]
        nc = len(pool.lens)
        dev = pool.k[0].device
        L = len(pool.k)
        q = cls([torch.empty_like(pool.k[l], dtype=torch.uint8) for l in range(L)],
                [torch.empty_like(pool.v[l], dtype=torch.uint8) for l in range(L)],
                *[[torch.empty(nc, W, dtype=torch.float32, device=dev) for _ in range(L)] for _ in range(4)],
                list(pool.offsets), list(pool.lens))
        for l in range(L):
            for c, (off, n) in enumerate(zip(pool.offsets, pool.lens)):
                B.cb_kv_quantize(pool.k[l][off:off + n], n, W, dims.dtype, q.kq[l][off:off + n], q.ks[l][c], q.kz[l][c])
                B.cb_kv_quantize(pool.v[l][off:off + n], n, W, dims.dtype, q.vq[l][off:off + n], q.vs[l][c], q.vz[l][c])
        return q

    def layer_tensors(self, l: int) -> List[torch.Tensor]:
        return [self.kq[l], self.vq[l], self.ks[l], self.kz[l], self.vs[l], self.vz[l]]


class BlendEngine:
    def __init__(self, dm: DeviceModel, n_tok_max: int, max_pos: Optional[int] = None, device="cuda"):
        self.dm = dm
        self.device = device
        s = dm.shape
        self.max_pos = int(max_pos or n_tok_max)
        self.cos_sin = torch.empty(self.max_pos * s.head_dim, dtype=torch.float32, device=device)
        B.cb_rope_table(self.cos_sin, self.max_pos, s.head_dim, float(s.rope_base))
        self.ws = torch.empty(B.cb_workspace_bytes(dm.dims, n_tok_max, n_tok_max), dtype=torch.uint8,
                              device=device)
        self.n_tok_max = n_tok_max
        # inputs shorter than this are prefilled in full: the blend's fixed overhead (pre-check
        # and check layers) outweighs its savings there ([CB-A] §configuration parameters,
        # minimum token count for blending, 256)
        self.min_tokens = 256
        # device-resident chunk KV is re-positioned on this stream beside the layers, one
        # event per layer (run_blend(..., overlap_assembly=True))
        self.asm_stream = torch.cuda.Stream(device=device)
        self.asm_done = [torch.cuda.Event() for _ in range(dm.shape.n_layers)]
        # check and gradual layers expand the selected rows' K/V on this stream beside the
        # selected queries' GEMM (run_blend(..., aux_expansion=True))
        self.aux_stream = torch.cuda.Stream(device=device)
        self.aux_events = (torch.cuda.Event(), torch.cuda.Event())
        for ev in self.aux_events:       # torch creates the CUDA event on its first record
            ev.record(self.aux_stream)

    # ---- precompute (offline: KV^pre) ------------------------------------------------------
    def precompute_pool(self, chunk_tokens: Sequence[np.ndarray]) -> ChunkPool:
        s = self.dm.shape
        lens = [len(t) for t in chunk_tokens]
        offs = list(np.cumsum([0] + lens[:-1]))
        rows = int(sum(lens))
        dt = torch_dtype(s)
        k = [torch.empty(rows, s.kv_width, dtype=dt, device=self.device) for _ in range(s.n_layers)]
        v = [torch.empty(rows, s.kv_width, dtype=dt, device=self.device) for _ in range(s.n_layers)]
        for t, off, n in zip(chunk_tokens, offs, lens):
            tok = torch.from_numpy(np.asarray(t, np.int32)).to(self.device)
            B.cb_full_prefill(self.dm.dims, self.dm.layers_c, self.dm.embed, tok, n, 0,
                              [kk[off:off + n] for kk in k], [vv[off:off + n] for vv in v], None, None,
                              self.cos_sin, self.max_pos, self.ws)
        return ChunkPool(k, v, [int(o) for o in offs], lens)

    def full_prefill(self, tokens: torch.Tensor, k_out, v_out, h_last, x_all=None, pos0: int = 0):
        B.cb_full_prefill(self.dm.dims, self.dm.layers_c, self.dm.embed, tokens, tokens.numel(), pos0, k_out,
                          v_out, h_last, x_all, self.cos_sin, self.max_pos, self.ws)


class Request:
    """Device state of one blended-prefill request: the row layout (cached chunk slots and
    uncached spans), token ids, the blended K/V cache of every layer, hidden-row buffers.

    Default layout: the chunks of `order` back to back, then the uncached query suffix.
    With `segments` (each an int chunk id or an array of uncached token ids: a system
    prompt, separators, query spans, in any order) the uncached rows are given to the
    library as a forced-row mask; `tokens` is then the whole input in segment order."""

    def __init__(self, eng: BlendEngine, pool, order: Sequence[int], tokens: np.ndarray, segments=None, kv=None):
        """kv: optional (K, V) lists of per-layer [N, Hkv*hd] tensors to use as this
        request's blended cache (e.g. views into a batch's shared caches)."""
        s = eng.dm.shape
        dev = eng.device
        dt = torch_dtype(s)
        self.eng, self.pool = eng, pool
        self.N = int(len(tokens))
        if segments is None:
            segments = list(order) + ([np.zeros(self.N - int(sum(pool.lens[c] for c in order)), np.int32)]
                                      if self.N > sum(pool.lens[c] for c in order) else [])
            general = False
        else:
            general = True
        self.segments = list(segments)
        self.order = [g for g in self.segments if isinstance(g, (int, np.integer))]
        src, delta, qrow = [], [], []
        self.runs = []                                # (first blended row, first cached index, rows)
        cached = np.zeros(self.N, bool)
        start = 0
        for g in self.segments:
            if isinstance(g, (int, np.integer)):
                n = pool.lens[g]
                if self.runs and self.runs[-1][0] + self.runs[-1][2] == start:
                    r0, c0, m = self.runs[-1]
                    self.runs[-1] = (r0, c0, m + n)
                else:
                    self.runs.append((start, len(src), n))
                src.extend(range(pool.offsets[g], pool.offsets[g] + n))
                delta.extend([start] * n)             # p - p' = slot start (p' = local position)
                qrow.extend([int(g)] * n)             # chunk of the row (8-bit pool tables)
                cached[start:start + n] = True
            else:
                n = len(g)
            start += n
        if start != self.N:
            raise ValueError(f"segments cover {start} rows, tokens {self.N}")
        self.n_cached = int(cached.sum())             # the HKVD budget counts these rows
        forced = ~cached
        forced[self.N - 1] = True
        self.n_forced = int(forced.sum())
        self.forced_mask = torch.from_numpy(forced.astype(np.uint8)).to(dev) if general else None
        self.src_host = np.asarray(src, np.int64)
        self.src_row = torch.tensor(src, dtype=torch.int32, device=dev)
        self.delta = torch.tensor(delta, dtype=torch.int32, device=dev)
        self.qrow = torch.tensor(qrow, dtype=torch.int32, device=dev)
        self.n_pool_rows = int(sum(pool.lens))
        self.tokens_host = check_token_ids(tokens, s.vocab)
        self.tokens = torch.from_numpy(self.tokens_host).to(dev)
        if kv is not None:
            self.K, self.V = list(kv[0]), list(kv[1])
        else:
            self.K = [torch.zeros(self.N, s.kv_width, dtype=dt, device=dev) for _ in range(s.n_layers)]
            self.V = [torch.zeros(self.N, s.kv_width, dtype=dt, device=dev) for _ in range(s.n_layers)]
        self.x = [torch.empty(self.N, s.d_model, dtype=dt, device=dev) for _ in range(2)]
        # each hidden-row buffer's partial sums of squares (left by the layer that wrote it, so
        # the next layer's norm folds into its GEMMs); at most 2 * ceil(d / 192) per row
        self.ssq = [torch.empty(2 * -(-s.d_model // 192) * self.N, dtype=torch.float32, device=dev)
                    for _ in range(2)]
        self.s = [torch.empty(self.N, dtype=torch.int32, device=dev) for _ in range(2)]
        self.scores = torch.empty(self.N, dtype=torch.float32, device=dev)
        self.token = torch.zeros(1, dtype=torch.int32, device=dev)
        self.sel_hist: List[torch.Tensor] = []
        self.m_hist: List[int] = []

    start_rows = None      # device int32 rows entering the first layer (None: every row)
    start_tokens = None

    def pool_ranges(self, n_rows: int):
        """Pool rows feeding the request's first n_rows cached slots, as (first row, rows)
        ranges of consecutive pool rows."""
        return contiguous_ranges(self.src_host[:n_rows])

    def plan(self, ratios: Sequence[Optional[float]], check_layer: int = 1, gradual: bool = False):
        return layer_plan(self.eng.dm.shape, self.N, self.n_cached, ratios, check_layer, gradual,
                          n_forced=self.n_forced)

    def prefix_cache_plan(self):
        """The prefix-caching comparison workload: only the cached rows before the first
        uncached row are reused (a true prefix, exact), every later row is recomputed at
        every layer.  Sets the first layer's rows and returns the all-steady plan."""
        first = int(np.argmax(self.forced_mask.cpu().numpy() != 0)) if self.forced_mask is not None else \
            min(self.n_cached, self.N - 1)
        rows = np.arange(first, self.N, dtype=np.int32)
        self.start_rows = torch.from_numpy(rows).to(self.tokens.device)
        self.start_tokens = torch.from_numpy(self.tokens_host[first:].copy()).to(self.tokens.device)
        return [(B.CB_LAYER_STEADY, 0)] * self.eng.dm.shape.n_layers


def check_token_ids(tokens, vocab: int) -> np.ndarray:
    """Token ids as int32, each in [0, vocab) (the embedding lookup's rows); raises otherwise.
    The device gather checks them again against the table height."""
    t = np.asarray(tokens)
    if t.ndim != 1 or (t.size and (int(t.min()) < 0 or int(t.max()) >= vocab)):
        raise ValueError(f"token ids must be a 1-D array of values in [0, {vocab})")
    return t.astype(np.int32)


def contiguous_ranges(rows) -> list:
    """(first, count) runs of consecutive values in a row list, in list order."""
    src = np.asarray(rows, np.int64)
    if len(src) == 0:
        return []
    cut = np.nonzero(np.diff(src) != 1)[0] + 1
    return [(int(a[0]), int(len(a))) for a in np.split(src, cut)]


def precheck_split_rows(shape: ModelShape, n_tok: int, n_cached: int, link_gbs: float, gemm_tflops: float,
                        hbm_gbs: float, store_esz: Optional[int] = None) -> int:
    """How many cached rows of the pre-check layer to load (the rest have their K/V
    recomputed): the load controller's balance ([CB-A] §Pipelining and load controller)
    applied at that layer, where recomputing is exact up to rounding (R5).  Loading X rows
    over the host link and re-positioning them should take as long as the work queued ahead
    of the layer's attention: RMSNorm and Q for every row, K/V for the other N - X rows.
    Both sides are linear in X; the result is where they meet, rounded down to 64 rows.
    store_esz: bytes per stored K/V element on the host (default: the compute dtype's; 1 for
    an 8-bit store, whose decode is part of the re-positioning pass)."""
    s = shape
    esz = 2 if s.dtype == "bf16" else 4
    sesz = esz if store_esz is None else store_esz
    N, d, qc, W = n_tok, s.d_model, s.q_width, s.kv_width
    R, L, H = gemm_tflops * 1e12, link_gbs * 1e9, hbm_gbs * 1e9
    t_q = 2.0 * N * d * qc / R + 2.0 * N * d * esz / H
    c = 2.0 * d * 2 * W / R
    l = 2.0 * W * sesz / L + 2.0 * W * (sesz + esz) / H
    x = int((t_q + N * c) / (c + l)) // 64 * 64
    return max(1, min(n_cached, x))


def layer_plan(shape: ModelShape, n_tok: int, n_cached: int, ratios: Sequence[Optional[float]],
               check_layer: int = 1, gradual: bool = False, n_forced: Optional[int] = None):
    """Host bookkeeping of the per-layer mode and HKVD budget (k and |S| are known before
    any launch, so the loop never waits on the device).  n_cached is the budget's base (the
    cached rows); n_forced the always-recomputed rows (default: the rows after the cached
    prefix, and at least the last row)."""
    if n_forced is None:
        n_forced = n_tok - min(n_cached, n_tok - 1)
    f0 = n_tok - n_forced                  # candidates at the check layer
    plan = []
    m_in = n_tok
    for l in range(shape.n_layers):
        if l < check_layer:
            plan.append((B.CB_LAYER_PRECHECK, 0))
            m_in = n_tok
        elif l == check_layer:
            k = B.cb_hkvd_budget(n_cached, ratios[l], f0)
            plan.append((B.CB_LAYER_CHECK, k))
            m_in = k + n_forced
        elif gradual:
            n_cand = m_in - n_forced
            k = B.cb_hkvd_budget(n_cached, ratios[l], n_cand)
            plan.append((B.CB_LAYER_GRADUAL, k))
            m_in = k + n_forced
        else:
            plan.append((B.CB_LAYER_STEADY, 0))
    return plan


class HostPool:
    """A chunk-KV pool (bf16 or 8-bit) mirrored in pinned host memory (the storage tier of
    the pages' design), with a side stream and one event per layer for layer-ahead loading
    into the device pool."""

    def __init__(self, pool):
        self.pool = pool
        n_layers = len(pool.k) if isinstance(pool, ChunkPool) else len(pool.kq)
        self.dev = [pool.layer_tensors(l) for l in range(n_layers)]
        self.host = [[t.cpu().pin_memory() for t in ts] for ts in self.dev]
        self.side = torch.cuda.Stream()
        self.done = [torch.cuda.Event() for _ in range(n_layers)]
        for ev in self.done:          # torch creates the CUDA event on its first record
            ev.record(self.side)
        self.nbytes = sum(t.numel() * t.element_size() for ts in self.host for t in ts)

    def copy_layer(self, l: int, ranges=None):
        """Queue layer l's copy on the side stream: the whole layer, or only the given
        (first pool row, rows) ranges of its K and V rows (bf16/fp32 values, or 8-bit codes;
        an 8-bit pool's per-chunk scale/zero tables are copied whole)."""
        n_rows = self.dev[l][0].shape[0]
        for i, (h, d) in enumerate(zip(self.host[l], self.dev[l])):
            row_indexed = i < 2   # K and V rows (values or codes); the rest are per-chunk tables
            if ranges is None or not row_indexed:
                B.cb_prefetch_layer(d, h, h.numel() * h.element_size(), self.side, self.done[l])
            else:
                assert h.shape[0] == n_rows
                rb = h.shape[1] * h.element_size()
                for r0, n in ranges:
                    B.cb_prefetch_layer(d[r0:r0 + n], h[r0:r0 + n], n * rb, self.side, self.done[l])

    def begin(self, stream):
        """Loads queued from here on start once `stream`'s prior work is done."""
        self.side.wait_stream(stream)

    def load_layer(self, l: int, after_copy=None, ranges=None):
        """Queue layer l's copy (only the given row ranges, if any); after_copy(l,
        side_stream) enqueues more work on the landed layer (the re-positioning) before the
        layer's event is recorded."""
        self.copy_layer(l, ranges)
        if after_copy is not None:
            after_copy(l, self.side)
            self.done[l].record(self.side)

    def prefetch_all(self, stream, after_copy=None, skip=(), partial=None):
        """Queue every layer's copy (but those in skip; only some rows of the layers in
        partial: {layer: ranges}) on the side stream once `stream`'s prior work is done."""
        self.begin(stream)
        for l in range(len(self.host)):
            if l not in skip:
                self.load_layer(l, after_copy, (partial or {}).get(l))


class FileStore:
    """A chunk-KV pool (bf16 or 8-bit) kept in one file, the storage tier below pinned host
    memory: every layer's tensors back to back in HostPool order, written once (offline).
    read_layer(l) brings one layer into the HostPool's pinned buffers with cb_file_read."""

    def __init__(self, path: str, host_pool: HostPool, n_threads: int = 8):
        self.path, self.hp, self.n_threads = path, host_pool, n_threads
        self.layout = []
        off = 0
        with open(path, "wb") as f:
            for hs in host_pool.host:
                ent = []
                for h in hs:
                    b = h.numel() * h.element_size()
                    f.write(h.reshape(-1).view(torch.uint8).numpy().tobytes())
                    ent.append((off, b))
                    off += b
                self.layout.append(ent)
        self.nbytes = off

    def read_layer(self, l: int):
        for (off, b), h in zip(self.layout[l], self.hp.host[l]):
            B.cb_file_read(self.path, off, h, b, self.n_threads)


class RequestGraph:
    """One request shape captured as a CUDA graph, from the token ids in pinned host memory
    to the first-token id in pinned host memory: the token upload, every layer's chunk-KV
    load and re-positioning on the loading stream (when a host pool is given), the layers,
    the lm_head and the read-back.  A request of the same sizes replays it after the host
    refreshes the token ids (run(tokens)); another chunk layout of the same sizes refreshes
    the request's row maps (src_row, delta) in place first."""

    def __init__(self, req: Request, plan, host_pool: Optional[HostPool] = None, stream=None,
                 recompute_precheck_kv: bool = False, precheck_load_rows: Optional[int] = None):
        self.req, self.plan, self.host_pool = req, plan, host_pool
        self.recompute = recompute_precheck_kv
        self.split = precheck_load_rows
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.host_tokens = torch.from_numpy(req.tokens_host.copy()).pin_memory()
        self.out = torch.empty(1, dtype=torch.int32).pin_memory()
        for _ in range(2):               # first calls set kernel attributes and tensor maps
            self._enqueue()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._enqueue()
        self.stream.synchronize()

    def _enqueue(self):
        with torch.cuda.stream(self.stream):
            B.cb_copy_async(self.req.tokens, self.host_tokens, self.req.N * 4, self.stream)
            run_blend(self.req, self.plan, host_pool=self.host_pool, stream=self.stream,
                      recompute_precheck_kv=self.recompute, precheck_load_rows=self.split)
            B.cb_copy_async(self.out, self.req.token, 4, self.stream)

    def run(self, tokens=None) -> int:
        if tokens is not None:
            t = check_token_ids(tokens, self.req.eng.dm.shape.vocab)
            if t.shape != (self.req.N,):
                raise ValueError(f"a captured request takes exactly {self.req.N} token ids")
            self.host_tokens.numpy()[:] = t
        with torch.cuda.stream(self.stream):      # a graph replays on the current stream
            self.graph.replay()
        self.stream.synchronize()
        return int(self.out.item())


def run_blend(req: Request, plan, dev_mode: int = B.CB_DEV_KV, sel_override=None, keep_history=False,
              assemble: bool = True, stream=None, host_pool: Optional[HostPool] = None,
              file_store: Optional[FileStore] = None, recompute_precheck_kv: bool = False,
              precheck_load_rows: Optional[int] = None, overlap_assembly: bool = True,
              layer_events: Optional[list] = None, upto: Optional[int] = None, x_out_last=None, s_out_last=None,
              aux_expansion: bool = True, fold_norms: bool = True):
    """One blended prefill: re-position the chunk KV of every layer, run the layer plan,
    then the lm_head argmax.  Returns the number of rows carried out of the last layer.

    With host_pool, every layer's chunk KV is copied from pinned host memory and
    re-positioned on a side stream, all layers queued up front; layer l waits for its own
    layer's event only where it first touches the cached rows (in the pre-check layer after
    its Q and uncached-row K/V GEMMs), so loading overlaps recompute.

    With file_store (whose host pool is used), a loader thread reads each layer from the
    file into pinned memory and then queues that layer's copy and re-positioning; the layer
    loop waits on the host for the layer's read before queueing the layer (the pages'
    generator pipeline: fetch layer l+1 while layer l computes).

    recompute_precheck_kv: the pre-check layers compute K/V for every row instead of using
    the chunk caches, which agree with it up to rounding there (R5); their chunk KV is then
    neither loaded nor re-positioned (a third of the host bytes of a three-layer stack).

    overlap_assembly (device-resident pool only; default on): the re-positioning runs on the
    engine's assembly stream, queued layer by layer between the layers, and each layer waits
    for its own layer's event at its first cached-row access, instead of all of it up front
    on the layers' stream (32-layer 7B-shape step 12.25 -> 12.15 ms; no change at 3 layers).

    layer_events: a list that receives (layer, start, end) CUDA events recorded on the
    layers' stream around each layer (timing only).

    precheck_load_rows: the pre-check layers use the chunk caches for the first X cached
    rows only and compute K/V for the rest (R5 again); only those X rows of their chunk KV
    are loaded and re-positioned.  precheck_split_rows() picks the X at which the load
    ends with the GEMMs that precede the layer's attention.

    aux_expansion (default on): check and gradual layers expand the selected rows' K/V on
    the engine's aux stream beside the selected queries' GEMM.

    fold_norms (default on): each layer hands its output rows' sums of squares to the next,
    so that with unit attention-norm gains (bf16) the next layer folds its norm into its
    Q/K/V GEMMs instead of running a norm pass.

    upto: run layers [0, upto) only and skip the lm_head (every layer's chunk KV is still
    re-positioned); the last of them writes its rows to x_out_last / s_out_last when given.
    Returns that layer's row count."""
    eng = req.eng
    dm = eng.dm
    s = dm.shape
    dims = dm.dims
    esz = 2 if s.dtype == "bf16" else 4
    if req.N < eng.min_tokens:
        # too short to blend: a full prefill of the request (every row, every layer)
        if host_pool is not None or file_store is not None:
            raise ValueError("requests shorter than min_tokens are prefilled in full and load no chunk KV")
        B.cb_full_prefill(dims, dm.layers_c, dm.embed, req.tokens, req.N, 0, req.K, req.V, None, req.x[0],
                          eng.cos_sin, eng.max_pos, eng.ws, stream)
        if keep_history:
            rows = torch.arange(req.N, dtype=torch.int32, device=req.tokens.device)
            req.sel_hist, req.m_hist = [rows] * s.n_layers, [req.N] * s.n_layers
        req.m_last, req.x_last = req.N, req.x[0]
        B.cb_lmhead_argmax(req.x[0][req.N - 1], dm.final_norm, dm.w_lm, dims, None, req.token, eng.ws, stream)
        return req.N
    pre = {l for l, (mode, _) in enumerate(plan) if mode == B.CB_LAYER_PRECHECK}
    split = None
    if precheck_load_rows is not None:
        split = int(precheck_load_rows)
        if req.forced_mask is not None or recompute_precheck_kv or not 0 < split <= req.n_cached:
            raise ValueError("precheck_load_rows needs the default layout, 0 < X <= n_cached and no "
                             "recompute_precheck_kv")

    def assemble_layer(l, st):
        # one re-positioning pass per run of adjacent chunk slots (pre-check layers with a
        # split: the rows below it only)
        lim = split if (split is not None and l in pre) else None
        for r0, c0, n in req.runs:
            if lim is not None:
                if r0 >= lim:
                    continue
                n = min(n, lim - r0)
            kd, vd = req.K[l][r0:r0 + n], req.V[l][r0:r0 + n]
            src, dl = req.src_row[c0:c0 + n], req.delta[c0:c0 + n]
            if isinstance(req.pool, ChunkPoolQ8):
                p = req.pool
                B.cb_rope_shift_q8(kd, vd, p.kq[l], p.vq[l], p.ks[l], p.kz[l], p.vs[l], p.vz[l], src,
                                   req.n_pool_rows, req.qrow[c0:c0 + n], len(p.lens), dl, n, dims, eng.cos_sin,
                                   eng.max_pos, st)
            else:
                B.cb_rope_shift(kd, vd, req.pool.k[l], req.pool.v[l], src, dl, n, dims, eng.cos_sin, eng.max_pos,
                                st)

    skip = set(pre) if recompute_precheck_kv else set()
    partial = {l: req.pool_ranges(split) for l in pre} if split is not None else {}
    ready, errors, loader, queue_loads = None, [], None, None
    if file_store is not None:
        host_pool = file_store.hp
    if host_pool is not None and host_pool.pool is not req.pool:
        raise ValueError("host_pool must mirror the request's pool")
    if file_store is not None:
        hp = host_pool
        hp.side.synchronize()              # the pinned buffers are no longer being copied from
        hp.side.wait_stream(torch.cuda.current_stream() if stream is None else stream)
        ready = [threading.Event() for _ in range(s.n_layers)]

        def load():
            try:
                # this thread's calls size and launch work for the engine's device
                torch.cuda.set_device(hp.side.device)
                for l in range(s.n_layers):
                    if l in skip:
                        ready[l].set()
                        continue
                    file_store.read_layer(l)
                    hp.copy_layer(l, partial.get(l))
                    if assemble:
                        assemble_layer(l, hp.side)
                        hp.done[l].record(hp.side)
                    ready[l].set()
            except BaseException as e:      # surfaced by the layer loop
                errors.append(e)
                for ev in ready:
                    ev.set()

        loader = threading.Thread(target=load, daemon=True)
        loader.start()
    elif host_pool is not None:
        # the loads are queued in layer order, interleaved with the layers: layer 0's before
        # anything else, layer l+1's right after layer l has been queued (the host runs far
        # ahead of the device, so every load still starts as soon as the previous one ends,
        # and the first layer's launches are not held back behind the later layers' calls)
        host_pool.begin(torch.cuda.current_stream() if stream is None else stream)
        queued = [0]

        def queue_loads(upto):
            while queued[0] < min(upto, s.n_layers):
                l = queued[0]
                if l not in skip:
                    host_pool.load_layer(l, assemble_layer if assemble else None, partial.get(l))
                queued[0] += 1
        queue_loads(1)

    # a first layer that runs every row reads its input rows in place from the embedding table
    # (row map = the token ids); otherwise the rows are gathered first
    embed_in_place = req.start_rows is None and plan[0][0] == B.CB_LAYER_PRECHECK
    if embed_in_place:
        m_in, s_in = req.N, None
    elif req.start_rows is None:
        B.cb_gather_rows(req.x[0], dm.embed, req.tokens, req.N, s.d_model * esz, stream)
        m_in, s_in = req.N, None
    else:
        # the first layer starts from a subset of rows (e.g. everything after a reused prefix)
        m_in = int(req.start_rows.numel())
        B.cb_gather_rows(req.x[0], dm.embed, req.start_tokens, m_in, s.d_model * esz, stream)
        s_in = req.start_rows
    asm_ready = None
    if assemble and host_pool is None:
        if overlap_assembly:
            main = torch.cuda.current_stream() if stream is None else stream
            eng.asm_stream.wait_stream(main)
            asm_ready = {}
            queued = [0]

            def queue_loads(upto):
                while queued[0] < min(upto, s.n_layers):
                    l = queued[0]
                    if l not in skip:
                        assemble_layer(l, eng.asm_stream)
                        eng.asm_done[l].record(eng.asm_stream)
                        asm_ready[l] = eng.asm_done[l]
                    queued[0] += 1
            queue_loads(1)
        else:
            for l in range(s.n_layers):
                if l not in skip:
                    assemble_layer(l, stream)
    cur = 0
    ssq_parts = 0                       # statistics of req.x[cur] (none for the first layer)
    if keep_history:
        req.sel_hist, req.m_hist, req.score_hist = [], [], []
    for l, (mode, k) in enumerate(plan):
        if upto is not None and l >= upto:
            break
        last = upto is not None and l == upto - 1
        if ready is not None:
            ready[l].wait()
            if errors:
                loader.join()
                raise errors[0]
        ov = None if sel_override is None else sel_override.get(l)
        if layer_events is not None:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(torch.cuda.current_stream() if stream is None else stream)
        first = embed_in_place and l == 0
        parts_out = [0]
        m_out = B.cb_blend_layer(dims, dm.layers_c[l], mode, dm.embed if first else req.x[cur], s_in, m_in, req.N,
                                 req.n_cached,
                                 req.K[l], req.V[l], eng.cos_sin, eng.max_pos, k, dev_mode, ov,
                                 x_out_last if (last and x_out_last is not None) else req.x[1 - cur],
                                 s_out_last if (last and s_out_last is not None) else req.s[1 - cur],
                                 req.scores if mode in (B.CB_LAYER_CHECK, B.CB_LAYER_GRADUAL) else None,
                                 eng.ws, stream,
                                 kv_ready=(asm_ready.get(l) if asm_ready is not None else
                                           None if (host_pool is None or l in skip) else host_pool.done[l]),
                                 forced_mask=req.forced_mask, n_forced=req.n_forced, recompute_kv=l in skip,
                                 recompute_from=split if (split is not None and l in pre) else 0,
                                 x_rows=req.tokens if first else None, n_x_rows=s.vocab if first else 0,
                                 aux=((eng.aux_stream,) + eng.aux_events
                                      if aux_expansion and mode in (B.CB_LAYER_CHECK, B.CB_LAYER_GRADUAL) else None),
                                 x_out_ssq=None if (last or not fold_norms) else req.ssq[1 - cur],
                                 ssq_parts_out=parts_out,
                                 x_in_ssq=req.ssq[cur] if (ssq_parts and not first) else None,
                                 x_in_ssq_parts=ssq_parts)
        if layer_events is not None:
            ev[1].record(torch.cuda.current_stream() if stream is None else stream)
            layer_events.append((l, ev[0], ev[1]))
        cur = 1 - cur
        s_in = req.s[cur]
        m_in = m_out
        ssq_parts = parts_out[0]
        if queue_loads is not None:
            queue_loads(l + 2)
        if keep_history:
            req.sel_hist.append(req.s[cur][:m_out].clone())
            req.m_hist.append(m_out)
            req.score_hist.append(req.scores.clone() if mode in (B.CB_LAYER_CHECK, B.CB_LAYER_GRADUAL) else None)
    if upto is not None and queue_loads is not None:
        queue_loads(s.n_layers)          # the layers run later (by a batch) still need their KV
    if loader is not None:
        loader.join()
    if asm_ready is not None:
        # join the assembly stream (each layer already waited for its own re-positioning)
        (torch.cuda.current_stream() if stream is None else stream).wait_stream(eng.asm_stream)
    if upto is not None:
        return m_in
    req.m_last = m_in
    req.x_last = req.x[cur]
    h_last = req.x[cur][m_in - 1]
    B.cb_lmhead_argmax(h_last, dm.final_norm, dm.w_lm, dims, None, req.token, eng.ws, stream)
    return m_in


class RequestBatch:
    """Independent requests of the same length over one chunk pool, run together (the
    batch of the Yi-34B-shaped workload).  Each layer's blended caches of the R requests are
    one [R * N, Hkv*hd] tensor (request r's rows at [r N, (r + 1) N)).  The layers up to the
    check layer run per request; from there on (fixed mode: every later layer keeps the
    check layer's rows) the selected rows of all requests are one set of GEMM rows, so each
    steady layer reads its weights once for the whole batch (cb_blend_steady_batch)."""

    def __init__(self, eng: BlendEngine, pool, orders: Sequence[Sequence[int]], tokens_list: Sequence[np.ndarray]):
        s = eng.dm.shape
        dev = eng.device
        dt = torch_dtype(s)
        N = {len(t) for t in tokens_list}
        if len(N) != 1:
            raise ValueError("the requests of a batch must have the same length")
        self.N = N.pop()
        self.R = len(tokens_list)
        self.eng = eng
        self.K = [torch.zeros(self.R * self.N, s.kv_width, dtype=dt, device=dev) for _ in range(s.n_layers)]
        self.V = [torch.zeros(self.R * self.N, s.kv_width, dtype=dt, device=dev) for _ in range(s.n_layers)]
        self.reqs = []
        for r, (order, toks) in enumerate(zip(orders, tokens_list)):
            sl = slice(r * self.N, (r + 1) * self.N)
            self.reqs.append(Request(eng, pool, order, toks, kv=([k[sl] for k in self.K], [v[sl] for v in self.V])))
        self.X = None
        self.S = None
        self.ws = None

    def _buffers(self, m_total: int):
        s = self.eng.dm.shape
        if self.X is None or self.X[0].shape[0] < m_total:
            dt = torch_dtype(s)
            dev = self.eng.device
            self.X = [torch.empty(m_total, s.d_model, dtype=dt, device=dev) for _ in range(2)]
            self.S = torch.empty(m_total, dtype=torch.int32, device=dev)
            self.ws = torch.empty(B.cb_workspace_bytes(self.eng.dm.dims, m_total, m_total), dtype=torch.uint8,
                                  device=dev)


def run_blend_batch(batch: RequestBatch, plan, stream=None) -> List[int]:
    """One blended prefill of every request of the batch: per request the pre-check and the
    check layer (HKVD selection), then every steady layer once for all requests' selected
    rows, then each request's lm_head argmax (into req.token).
    Returns the rows each request carries out of the last layer."""
    eng = batch.eng
    dm = eng.dm
    s = dm.shape
    modes = [m for m, _ in plan]
    if B.CB_LAYER_CHECK not in modes:
        raise ValueError("a batched blend needs a check layer")
    c = modes.index(B.CB_LAYER_CHECK)
    if any(m != B.CB_LAYER_STEADY for m in modes[c + 1:]):
        raise ValueError("layers after the check layer must be steady (fixed mode) in a batched blend")
    if any(r.forced_mask is not None for r in batch.reqs):
        raise ValueError("a batched blend takes the default layout (chunks, then the query)")
    m_r = [plan[c][1] + r.n_forced for r in batch.reqs]
    row0 = [0]
    for m in m_r:
        row0.append(row0[-1] + m)
    batch._buffers(row0[-1])
    for r, req in enumerate(batch.reqs):
        m = run_blend(req, plan, stream=stream, upto=c + 1, x_out_last=batch.X[0][row0[r]:row0[r + 1]],
                      s_out_last=batch.S[row0[r]:row0[r + 1]], fold_norms=False)
        if m != m_r[r]:
            raise RuntimeError(f"request {r}: {m} rows out of the check layer, {m_r[r]} expected")
    cur = 0
    for l in range(c + 1, s.n_layers):
        B.cb_blend_steady_batch(dm.dims, dm.layers_c[l], row0, batch.X[cur], batch.S, batch.N, batch.K[l], batch.V[l],
                                eng.cos_sin, eng.max_pos, batch.X[1 - cur], batch.ws, stream)
        cur = 1 - cur
    for r, req in enumerate(batch.reqs):
        req.m_last = m_r[r]
        req.x_last = batch.X[cur][row0[r]:row0[r + 1]]
        B.cb_lmhead_argmax(req.x_last[m_r[r] - 1], dm.final_norm, dm.w_lm, dm.dims, None, req.token, eng.ws, stream)
    return m_r
