"""CPU oracle for CacheBlend selective KV recompute.  TEST INFRASTRUCTURE ONLY.

Only the test-suite, the package's smoke check and the benchmark's CPU-baseline leg may
import this module.  The product path (the CUDA library and its binding) never calls it.

Plain, slow, float64 numpy.  Loops are written for readability, not speed.  It shares no
code with the CUDA path; its inputs come from the seeded generator module only.

Sources (cited by short tag in each docstring):
  [CB-A]  "論文解説: CacheBlend — RAGシステム向けKV Cache融合による高速LLMサービング"
          (0h-n0.github.io/posts/paper-2312-03052)
  [CB-B]  "CacheBlend: Fast Large Language Model Serving for RAG with Cached Knowledge
          Fusion" explainer (abeam.tech, 2026-09-20-cacheblend-rag-cached-knowledge-fusion)
  [PC]    "論文解説: Prompt Cache — モジュラーAttention再利用による低レイテンシ推論"
          (0h-n0.github.io/posts/paper-2402-01008)
  [CG]    "論文解説: CacheGen — KVキャッシュ圧縮とストリーミングで長文コンテキストのLLM推論を
          高速化" (0h-n0.github.io/posts/paper-2401-12191)

Readings taken where the pages are silent or disagree (each is listed with its reason in
the design notes of the repository):
  R1  Queries are recomputed only for the selected rows (cost proportional to r); the
      page's "Q for all tokens" applies to the pre-check layer, which runs every row.
  R2  Deviation at the check layer = squared L2 distance between the layer's freshly
      computed K (and V) and the cached, re-rotated K (and V), summed over all KV heads.
  R3  Chunks are precomputed at local positions 0..n-1 and re-rotated by their start.
      RoPE pairs are interleaved (2i, 2i+1); theta_i = base^(-2i/head_dim).
  R4  The budget counts cached rows only: k = floor(N_c * r), at least 1 when r > 0,
      capped by the number of candidates.  Uncached rows and the last row are forced in.
  R5  The check layer is layer index 1 (0-based); layer 0 runs every row but reuses the
      re-rotated cached K/V, which at layer 0 equal a full prefill's up to rounding.
  R6  Gradual filtering: r_l = r + (r1 - r) * 2^-(l - c), r1 = min(1, 1.5 r); only the
      rows of S_l have their K/V overwritten.
  R7  Ties in top-k go to the lower row index; the selected rows are returned ascending.
  R8  RMSNorm eps = 1e-5, no biases, untied lm_head, argmax ties to the lowest index.
  (R9-R11 concern the benchmark's layer stack, the weight layout and the RoPE table of the
  CUDA path; they do not change what the oracle computes.)
  R12 8-bit chunk KV: per channel of one chunk's K (or V) of one layer, zero = min over
      the chunk's rows, scale = (max - min) / 255 floored at 1e-8, code = round half to
      even of (x - zero) / scale; the code is decided in float32 (the pages fix no
      precision), one IEEE operation per step, so both sides decide it bit for bit.
  R13 Uncached spans anywhere (system prompt, separators, query): every uncached row and
      the last row are forced; the budget counts the cached rows; the pre-check layer
      recomputes K/V of the uncached rows only.

Parity status of each function is stated in its docstring ("pinned by" / "parity
unpinned").
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------------------
def rope_theta(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d), i in [0, d/2)  ([CB-A] §RoPE, rotation matrix R(m);
    [PC] §RoPE position adjustment, theta_j).  d is the head dimension (R3).
    Pinned by: golden values for hand-computed theta (tests/golden/rope_points.txt)."""
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(base), -2.0 * i / head_dim)


def rope_rotate(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate each interleaved pair (x[2i], x[2i+1]) of the last axis by angle pos*theta_i:
        (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos)
    ([CB-A] §RoPE, R(m) applied to a 2-vector).  x: [n, heads, hd] (or [n, hd]);
    pos: scalar or [n] (any integer, negative allowed = inverse rotation).
    Pinned by: golden unit-vector rotations, R(a)R(b) = R(a+b), R(p)^T R(p) = I,
    the relative-position identity of the score."""
    x = np.asarray(x, dtype=F64)
    hd = x.shape[-1]
    theta = rope_theta(hd, base)
    pos = np.asarray(pos, dtype=F64)
    ang = pos.reshape(pos.shape + (1,) * (x.ndim - 1 - pos.ndim) + (1,)) * theta \
        if pos.ndim else pos * theta
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def rope_shift(k_pre: np.ndarray, delta, base: float) -> np.ndarray:
    """Re-position cached keys: k(p) = R(p - p') k(p')  ([PC] §RoPE position adjustment).
    delta = p - p' per row (or scalar).  Values are copied unchanged by the caller.
    Pinned by: R(delta) R(p') k == R(p' + delta) k (rotation from scratch)."""
    return rope_rotate(k_pre, delta, base)


# ----------------------------------------------------------------------------------------
# Model pieces (pre-norm decoder, R8)
# ----------------------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g, per row.
    Pinned by: constant rows (closed form), scale invariance."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=F64)


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z).  Pinned by: silu(0)=0, silu(z)->z for large z, silu(-z) = silu(z) - z."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x @ W^T with W stored [out, in].  Pinned by a one-hot weight (closed form)."""
    return np.asarray(x, dtype=F64) @ np.asarray(w, dtype=F64).T


def project_qkv(layer: dict, a: np.ndarray, pos, shape, want=("q", "k", "v")):
    """q, k, v projections of normalised rows a [n, d], RoPE applied to q and k at the
    given positions ([CB-A] §Selective recomputation, Step 2).  Returns a dict of
    q [n, H, hd], k [n, Hkv, hd], v [n, Hkv, hd] (only the requested ones)."""
    H, Hkv, hd = shape.n_heads, shape.n_kv_heads, shape.head_dim
    wq = layer["wqkv"][: H * hd]
    wk = layer["wqkv"][H * hd: (H + Hkv) * hd]
    wv = layer["wqkv"][(H + Hkv) * hd:]
    out = {}
    n = a.shape[0]
    if "q" in want:
        out["q"] = rope_rotate(linear(a, wq).reshape(n, H, hd), pos, shape.rope_base)
    if "k" in want:
        out["k"] = rope_rotate(linear(a, wk).reshape(n, Hkv, hd), pos, shape.rope_base)
    if "v" in want:
        out["v"] = linear(a, wv).reshape(n, Hkv, hd)
    return out


def attend(q: np.ndarray, q_pos: Sequence[int], K: np.ndarray, V: np.ndarray,
           k_pos: Optional[Sequence[int]] = None) -> np.ndarray:
    """Causal softmax attention of selected queries over the whole KV
    ([CB-A] §Selective recomputation, Step 4; [CB-B] §技術の仕組み: the selected tokens
    attend over the entire input).  Query j at position p_j sees every key whose position
    is <= p_j.  GQA: query head h reads KV head floor(h * Hkv / H).
    q [M, H, hd], K/V [N, Hkv, hd]; returns o [M, H*hd].
    Pinned by: single visible key -> V row; zero query -> mean of visible V rows;
    brute-force softmax on tiny inputs."""
    q = np.asarray(q, F64)
    K = np.asarray(K, F64)
    V = np.asarray(V, F64)
    M, H, hd = q.shape
    Hkv = K.shape[1]
    if k_pos is None:
        k_pos = np.arange(K.shape[0])
    k_pos = np.asarray(k_pos)
    scale = 1.0 / math.sqrt(hd)
    o = np.zeros((M, H, hd), F64)
    for j in range(M):
        vis = np.nonzero(k_pos <= q_pos[j])[0]
        for h in range(H):
            g = (h * Hkv) // H
            s = K[vis, g, :] @ q[j, h] * scale
            s = s - s.max()
            w = np.exp(s)
            w = w / w.sum()
            o[j, h] = w @ V[vis, g, :]
    return o.reshape(M, H * hd)


def out_ffn(layer: dict, x_rows: np.ndarray, o: np.ndarray, shape) -> np.ndarray:
    """h = x + o Wo^T;  y = h + (SiLU(b Wg^T) * (b Wu^T)) Wd^T with b = RMSNorm(h)
    ([CB-A] §Selective recomputation, Step 4 "next layer's input"; SwiGLU FFN)."""
    F = shape.d_ff
    h = np.asarray(x_rows, F64) + linear(o, layer["wo"])
    b = rmsnorm(h, layer["ffn_norm"], shape.rms_eps)
    gate = linear(b, layer["w_gate_up"][:F])
    up = linear(b, layer["w_gate_up"][F:])
    return h + linear(silu(gate) * up, layer["w_down"])


def layer_forward(layer: dict, x: np.ndarray, pos, shape) -> Dict[str, np.ndarray]:
    """Plain decoder layer over a contiguous row range (used by full prefill)."""
    a = rmsnorm(x, layer["attn_norm"], shape.rms_eps)
    p = project_qkv(layer, a, pos, shape)
    o = attend(p["q"], pos, p["k"], p["v"], k_pos=pos)
    return {"x": out_ffn(layer, x, o, shape), "k": p["k"], "v": p["v"]}


def full_prefill(model: dict, tokens: np.ndarray, pos0: int = 0) -> Dict[str, object]:
    """Standard causal prefill of a token range at positions pos0..pos0+n-1: KV^full when
    run over the whole input, KV^pre when run over one chunk alone at local positions
    ([CB-A] §KV cache definitions).  Returns per-layer K/V [n, Hkv, hd], every layer's
    hidden rows and the last hidden row.
    Pinned by: the true-prefix identity and causality (rows <= j depend on tokens <= j)."""
    shape = model["shape"]
    tokens = np.asarray(tokens)
    pos = pos0 + np.arange(len(tokens))
    x = np.asarray(model["embed"], F64)[tokens]
    Ks, Vs, xs = [], [], [x]
    for layer in model["layers"]:
        r = layer_forward(layer, x, pos, shape)
        Ks.append(r["k"])
        Vs.append(r["v"])
        x = r["x"]
        xs.append(x)
    return {"K": Ks, "V": Vs, "x": xs, "h_last": x[-1]}


def lm_head_argmax(model: dict, h_last: np.ndarray):
    """First token of the answer: argmax(RMSNorm(h) W_lm^T), lowest index on ties (R8).
    Pinned by: a hand-built case (one-hot lm_head rows, a non-unit final-norm gain,
    closed-form logits, a tie between equal rows)."""
    shape = model["shape"]
    b = rmsnorm(np.asarray(h_last, F64)[None, :], model["final_norm"], shape.rms_eps)
    logits = linear(b, model["w_lm"])[0]
    return int(np.argmax(logits)), logits


# ----------------------------------------------------------------------------------------
# HKVD selection
# ----------------------------------------------------------------------------------------
def kv_deviation(k_new, k_ref, v_new=None, v_ref=None) -> np.ndarray:
    """Per-token squared L2 deviation  s_j = sum (K_new[j] - K_ref[j])^2 (+ same for V)
    ([CB-A] §KV deviation definition and §HKVD selection code: sum of squared differences
    over the feature axis; R2: no square root, which is monotone).
    Pinned by: zero for identical rows, closed form for constant offsets."""
    k_new = np.asarray(k_new, F64).reshape(len(k_new), -1)
    k_ref = np.asarray(k_ref, F64).reshape(len(k_ref), -1)
    s = np.sum((k_new - k_ref) ** 2, axis=1)
    if v_new is not None:
        v_new = np.asarray(v_new, F64).reshape(len(v_new), -1)
        v_ref = np.asarray(v_ref, F64).reshape(len(v_ref), -1)
        s = s + np.sum((v_new - v_ref) ** 2, axis=1)
    return s


def budget(n_cached_candidates_total: int, ratio: float, n_candidates: Optional[int] = None) -> int:
    """HKVD budget k = floor(N_c * r) evaluated in double; at least 1 when r > 0 (the
    page's max(int(N * r), 1)); exactly 0 when r == 0; capped by the candidate count
    ([CB-A] §HKVD selection code; R4).  Pinned by: golden budget table."""
    if ratio <= 0.0:
        return 0
    k = int(math.floor(float(n_cached_candidates_total) * float(ratio)))
    k = max(k, 1)
    if n_candidates is not None:
        k = min(k, n_candidates)
    return k


def topk_rows(scores: np.ndarray, cand: Sequence[int], k: int) -> np.ndarray:
    """The k candidates with the largest score, ties to the lower row index, returned in
    ascending row order ([CB-A] §HKVD selection code: top-k then sort by position; R7).
    Implemented as a full sort by (score desc, row asc).
    Pinned by: brute force over all k-subsets on tiny inputs."""
    cand = np.asarray(cand, dtype=np.int64)
    scores = np.asarray(scores)
    if k <= 0:
        return np.zeros(0, np.int64)
    if np.any(~np.isfinite(scores)):
        raise ValueError("non-finite deviation score")
    order = sorted(range(len(cand)), key=lambda i: (-float(scores[i]), int(cand[i])))
    return np.sort(cand[order[:k]])


def ratio_schedule(r: float, n_layers: int, check_layer: int, gradual: bool,
                   r1_factor: float = 1.5) -> List[Optional[float]]:
    """Per-layer ratio: None for layers before the check layer; r at the check layer and
    after it in fixed mode; in gradual mode r_c = r1 = min(1, r1_factor*r) decaying toward
    r as r + (r1 - r) 2^-(l-c) ([CB-A] §Gradual filtering; R6).  The pages give no numbers,
    only the shape.  Pinned by: that shape (r1 >= r and <= 1, never increasing, never
    below r, tending to r; constant r in fixed mode) and non-increasing budgets."""
    out: List[Optional[float]] = []
    r1 = min(1.0, r1_factor * r)
    for l in range(n_layers):
        if l < check_layer:
            out.append(None)
        elif not gradual:
            out.append(r)
        else:
            out.append(r + (r1 - r) * 2.0 ** (-(l - check_layer)))
    return out


# ----------------------------------------------------------------------------------------
# Blend
# ----------------------------------------------------------------------------------------
def precompute_chunks(model: dict, chunk_tokens: Sequence[np.ndarray]) -> List[dict]:
    """KV^pre: each distinct chunk prefilled alone at local positions 0..n-1
    ([CB-A] §KV cache definitions; [CB-B] §チャンク単位でKVを保存する)."""
    return [full_prefill(model, t, 0) for t in chunk_tokens]


def assemble(model: dict, chunk_kv: Sequence[dict], order: Sequence[int], n_query: int):
    """Concatenate the chunks' KV in request order, keys re-rotated by their chunk's start
    s_m ([PC] §RoPE position adjustment; [CB-B] position correction at load time).
    Rows N_c..N-1 (the query suffix) are left zero: they are computed, never cached."""
    shape = model["shape"]
    lens = [chunk_kv[c]["K"][0].shape[0] for c in order]
    n_cached = int(sum(lens))
    N = n_cached + n_query
    K = [np.zeros((N, shape.n_kv_heads, shape.head_dim), F64) for _ in range(shape.n_layers)]
    V = [np.zeros_like(K[0]) for _ in range(shape.n_layers)]
    start = 0
    for c, n in zip(order, lens):
        for l in range(shape.n_layers):
            K[l][start:start + n] = rope_shift(chunk_kv[c]["K"][l], start, shape.rope_base)
            V[l][start:start + n] = chunk_kv[c]["V"][l]
        start += n
    return K, V, n_cached


def assemble_segments(model: dict, chunk_kv: Sequence[dict], segments: Sequence):
    """Lay out a request made of segments: an int is a cached chunk (its KV re-rotated by
    its slot's start, as in assemble), an array of token ids is uncached text (a system
    prompt, a separator, a query) whose rows are computed, never cached ([CB-A] §vLLM
    integration: separators between chunks; R13: any number of uncached spans).
    Returns K, V per layer with the cached rows filled, and the per-row cached mask."""
    shape = model["shape"]
    lens = [chunk_kv[g]["K"][0].shape[0] if isinstance(g, (int, np.integer)) else len(g) for g in segments]
    N = int(sum(lens))
    K = [np.zeros((N, shape.n_kv_heads, shape.head_dim), F64) for _ in range(shape.n_layers)]
    V = [np.zeros_like(K[0]) for _ in range(shape.n_layers)]
    cached = np.zeros(N, bool)
    start = 0
    for g, n in zip(segments, lens):
        if isinstance(g, (int, np.integer)):
            for l in range(shape.n_layers):
                K[l][start:start + n] = rope_shift(chunk_kv[g]["K"][l], start, shape.rope_base)
                V[l][start:start + n] = chunk_kv[g]["V"][l]
            cached[start:start + n] = True
        start += n
    return K, V, cached


def blend(model: dict, chunk_kv: Sequence[dict], order: Sequence[int], tokens: np.ndarray,
          ratios: Sequence[Optional[float]], check_layer: int = 1, gradual: bool = False,
          dev_mode: str = "kv", sel_override: Optional[Dict[int, np.ndarray]] = None,
          segments: Optional[Sequence] = None):
    """CacheBlend selective KV recompute, layer by layer
    ([CB-A] §Selective recomputation Steps 1-4, §HKVD selection, §Gradual filtering;
    [CB-B] §技術の仕組み).

    tokens: the whole input (chunks in order, then the query suffix).
    segments: optional general layout (see assemble_segments) replacing order + suffix:
              every uncached row is forced, the budget counts cached rows.
    ratios: per-layer ratio (None before the check layer), see ratio_schedule.
    sel_override: optional {layer: top-k row set} replacing the HKVD choice at that layer
                  (teacher forcing: the forced rows are still added).
    Returns dict with the blended K/V per layer, hidden rows per layer, the selected row
    sets and scores per layer, the last hidden row and the first token.

    Pinned by: r=1 equals full prefill; r=0 equals the re-rotated concatenation for cached
    rows and a suffix prefill over that fixed past for the query rows.  The HKVD choice at
    0 < r < 1 has no printed worked example: those values are parity unpinned beyond the
    invariants.
    """
    shape = model["shape"]
    L = shape.n_layers
    N = len(tokens)
    if segments is None:
        n_chunk_rows = sum(chunk_kv[c]["K"][0].shape[0] for c in order)
        K, V, n_cached = assemble(model, chunk_kv, order, N - n_chunk_rows)
        cached = np.arange(N) < n_cached
    else:
        K, V, cached = assemble_segments(model, chunk_kv, segments)
        assert len(cached) == N
        n_cached = int(cached.sum())
    forced = set(np.nonzero(~cached)[0].tolist()) | {N - 1}
    forced_sorted = np.array(sorted(forced), dtype=np.int64)

    x = np.asarray(model["embed"], F64)[np.asarray(tokens)]   # hidden rows of S
    S = np.arange(N)                                          # rows currently carried
    hist = {"S": [], "scores": [], "cand": [], "x": []}
    for l in range(L):
        layer = model["layers"][l]
        a = rmsnorm(x, layer["attn_norm"], shape.rms_eps)
        if l < check_layer:
            # pre-check layer: every row; cached rows keep the re-rotated cache (R5)
            p = project_qkv(layer, a, S, shape)
            unc = np.nonzero(~cached[S])[0]
            K[l][S[unc]] = p["k"][unc]
            V[l][S[unc]] = p["v"][unc]
            o = attend(p["q"], S, K[l], V[l])
            x = out_ffn(layer, x, o, shape)
            hist["S"].append(S.copy()); hist["scores"].append(None); hist["cand"].append(None)
        elif l == check_layer or gradual:
            # check (or gradual) layer: fresh K/V for the carried rows, deviation vs cache
            p = project_qkv(layer, a, S, shape, want=("k", "v"))
            cand_pos = np.array([i for i, r in enumerate(S) if cached[r] and r not in forced],
                                dtype=np.int64)
            cand = S[cand_pos]
            if dev_mode == "kv":
                sc = kv_deviation(p["k"][cand_pos], K[l][cand], p["v"][cand_pos], V[l][cand])
            else:
                sc = kv_deviation(p["k"][cand_pos], K[l][cand])
            k_l = budget(n_cached, ratios[l], len(cand))
            if sel_override is not None and l in sel_override:
                T = np.asarray(sel_override[l], np.int64)
            else:
                T = topk_rows(sc, cand, k_l)
            S_new = np.array(sorted(set(T.tolist()) | forced), dtype=np.int64)
            keep = np.searchsorted(S, S_new)                  # positions of S_new inside S
            K[l][S_new] = p["k"][keep]                         # Step 3: KV expansion
            V[l][S_new] = p["v"][keep]
            q = project_qkv(layer, a[keep], S_new, shape, want=("q",))["q"]
            o = attend(q, S_new, K[l], V[l])
            x = out_ffn(layer, x[keep], o, shape)
            hist["S"].append(S_new.copy()); hist["scores"].append(sc); hist["cand"].append(cand)
            S = S_new
        else:
            # steady layer, fixed mode: S_l = S_c
            p = project_qkv(layer, a, S, shape)
            K[l][S] = p["k"]
            V[l][S] = p["v"]
            o = attend(p["q"], S, K[l], V[l])
            x = out_ffn(layer, x, o, shape)
            hist["S"].append(S.copy()); hist["scores"].append(None); hist["cand"].append(None)
        hist["x"].append(x.copy())
    h_last = x[-1]
    tok, logits = lm_head_argmax(model, h_last)
    return {"K": K, "V": V, "S": hist["S"], "scores": hist["scores"], "cand": hist["cand"],
            "x": hist["x"], "h_last": h_last, "token": tok, "logits": logits,
            "n_cached": n_cached, "forced": forced_sorted}


# ----------------------------------------------------------------------------------------
# 8-bit per-channel chunk KV ([CG] §Step 1 per-channel quantization; entropy coding out)
# ----------------------------------------------------------------------------------------
F32 = np.float32


def kv_quantize(x, bits: int = 8):
    """Per-channel asymmetric quantization of one chunk's K (or V) of one layer ([CG] §Step 1:
    per channel c, z_c = min over tokens, s_c = (max - min) / (2^b - 1); code =
    round((x - z_c) / s_c)).  R12: float32, one rounding per operation, half to even, codes
    clipped to [0, 2^b - 1], the scale floored at 1e-8 (the page's listing clamps it so a
    constant channel does not divide by zero).
    Returns (codes uint8 [n, C], scale f32 [C], zero f32 [C]) for x [n, ...] (C = the
    trailing size).
    Pinned by: integer-valued channels with unit and even scales (codes = values, halves to
    even), min -> 0 and max -> 2^b - 1, the round-trip bound |x^ - x| <= s/2 (+ float32
    rounding), constant channels."""
    x2 = np.asarray(x, F32).reshape(len(x), -1)
    levels = F32(2 ** bits - 1)
    zero = x2.min(axis=0)
    scale = np.maximum((x2.max(axis=0) - zero) / levels, F32(1e-8)).astype(F32)
    codes = np.clip(np.rint((x2 - zero) / scale), 0, levels).astype(np.uint8)
    return codes, scale, zero


def kv_dequantize(codes, scale, zero) -> np.ndarray:
    """x^ = code * s + z in float32, the product rounded before the sum ([CG] decode step)."""
    return (np.asarray(codes, F32) * np.asarray(scale, F32)).astype(F32) + np.asarray(zero, F32)


def quantize_chunks(chunk_kv: Sequence[dict]) -> List[dict]:
    """The chunk store kept as 8-bit codes: every chunk's K and V of every layer quantized
    per channel, then decoded again (what the blend sees after loading)."""
    out = []
    for kv in chunk_kv:
        d = dict(kv)
        for key in ("K", "V"):
            layers = []
            for t in kv[key]:
                q, sc, z = kv_quantize(t)
                layers.append(kv_dequantize(q, sc, z).astype(F64).reshape(t.shape))
            d[key] = layers
        out.append(d)
    return out


# ----------------------------------------------------------------------------------------
# Cost-model helpers ([CB-A] §Pipelining and load controller; KV size per [CacheGen] page)
# ----------------------------------------------------------------------------------------
def kv_bytes(n_layers: int, n_tokens: int, n_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """K and V for every layer: 2 * L * S * H * d_h * elem_bytes."""
    return 2 * n_layers * n_tokens * n_kv_heads * head_dim * elem_bytes


def t_load(per_token_kv_bytes: float, n_tokens: int, throughput_bytes_per_s: float) -> float:
    """T_load = PerTokenKVSize * L / Throughput(D), L = input tokens ([CB-A] §load controller)."""
    return per_token_kv_bytes * n_tokens / throughput_bytes_per_s


def optimal_ratio(r_min: float, t_load_s: float, t_prefill_s: float) -> float:
    """r* = max(r_min, T_load / T_prefill)  ([CB-A] §load controller)."""
    return max(r_min, t_load_s / t_prefill_s)
