"""Thin ctypes binding of libcacheblend.so: the C entry points under the same names,
taking torch tensors (device memory) and marshalling them to raw pointers.  No arithmetic
of the method happens here; every step runs in the library's CUDA kernels.  Raises
CBError on any non-zero status.  Fails loudly when the library has not been built."""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

from . import build as _build

CB_OK = 0
CB_F32, CB_BF16 = 0, 1
CB_DEV_KV, CB_DEV_K = 0, 1
CB_LAYER_PRECHECK, CB_LAYER_CHECK, CB_LAYER_STEADY, CB_LAYER_GRADUAL = 0, 1, 2, 3
STATUS_NAMES = {0: "CB_OK", 1: "CB_ERR_INVALID_ARG", 2: "CB_ERR_SHAPE", 3: "CB_ERR_DTYPE",
                4: "CB_ERR_WORKSPACE", 5: "CB_ERR_NONFINITE", 6: "CB_ERR_CUDA", 7: "CB_ERR_TIMEOUT",
                8: "CB_ERR_UNSUPPORTED", 9: "CB_ERR_DEVICE", 10: "CB_ERR_IO"}


class CBError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class cb_layer_opts(C.Structure):
    _fields_ = [("forced_mask", C.c_void_p), ("n_forced", C.c_int32), ("kv_ready", C.c_void_p),
                ("recompute_kv", C.c_int32), ("recompute_from", C.c_int32), ("x_rows", C.c_void_p),
                ("n_x_rows", C.c_int64), ("aux_stream", C.c_void_p), ("aux_fork", C.c_void_p),
                ("aux_join", C.c_void_p), ("x_out_ssq", C.c_void_p), ("x_out_ssq_parts_host", C.POINTER(C.c_int32)),
                ("x_in_ssq", C.c_void_p), ("x_in_ssq_parts", C.c_int32)]


class cb_dims(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ff", C.c_int32), ("vocab", C.c_int32),
                ("rope_base", C.c_double), ("rms_eps", C.c_float), ("dtype", C.c_int32)]


class cb_layer_w(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("wqkv", C.c_void_p), ("wo", C.c_void_p),
                ("ffn_norm", C.c_void_p), ("w_gate_up", C.c_void_p), ("w_down", C.c_void_p)]


class cb_prof_record(C.Structure):
    _fields_ = [("kind", C.c_int32), ("aux", C.c_int32), ("m", C.c_int64), ("n", C.c_int64), ("k", C.c_int64),
                ("flops", C.c_double), ("bytes", C.c_double), ("ms", C.c_float), ("span_ms", C.c_float)]


PROF_KINDS = {0: "rope_shift", 1: "copy_rows", 2: "rmsnorm", 3: "gemm", 4: "attention", 5: "deviation",
              6: "topk", 7: "index", 8: "lmhead_gemv", 9: "argmax", 10: "rope_table", 11: "kv_quantize"}

_P = C.c_void_p
_I32 = C.c_int32
_I64 = C.c_int64
_SZ = C.c_size_t
_PROTOS = {
    "cb_status_string": (C.c_char_p, [C.c_int]),
    "cb_last_error_message": (C.c_char_p, []),
    "cb_last_cuda_error": (C.c_char_p, []),
    "cb_sync": (C.c_int, [_P, C.c_double]),
    "cb_workspace_bytes": (C.c_int, [C.POINTER(cb_dims), _I64, _I64, C.POINTER(_SZ)]),
    "cb_hkvd_budget": (_I64, [_I64, C.c_double, _I64]),
    "cb_gradual_ratio": (C.c_double, [C.c_double, _I32, _I32, C.c_double]),
    "cb_load_controller_ratio": (C.c_double, [C.c_double, C.c_double, C.c_double]),
    "cb_rope_table": (C.c_int, [_P, _I32, _I32, C.c_double, _P]),
    "cb_shutdown": (None, []),
    "cb_rope_shift": (C.c_int, [_P, _P, _P, _P, _P, _I64, _P, _I64, C.POINTER(cb_dims), _P, _I32, _P]),
    "cb_kv_deviation_topk": (C.c_int, [_P, _P, _I64, _P, _P, _I64, _P, _P, _I32, _I32, _I32, C.POINTER(cb_dims),
                                       _P, _P, _P, _SZ, _P]),
    "cb_kv_deviation_topk_noalloc": (C.c_int, [_P, _P, _I64, _P, _P, _I64, _P, _P, _I32, _I32, _I32,
                                               C.POINTER(cb_dims), _P, _P, _P]),
    "cb_topk_from_scores": (C.c_int, [_P, _P, _I32, _I32, _P, _P, _SZ, _P]),
    "cb_gather_rows": (C.c_int, [_P, _P, _I64, _P, _I64, _I64, _P]),
    "cb_scatter_kv": (C.c_int, [_P, _P, _I64, _P, _P, _I64, _P, _P, _I64, C.POINTER(cb_dims), _P]),
    "cb_selective_qkv": (C.c_int, [_P, _I64, _P, _P, _I32, C.POINTER(cb_dims), C.POINTER(cb_layer_w), _P, _I32,
                                   _P, _P, _P, _P, _SZ, _P]),
    "cb_partial_attention": (C.c_int, [_P, _P, _I32, _P, _P, _I64, C.POINTER(cb_dims), _P, _P, _SZ, _P]),
    "cb_o_proj_ffn": (C.c_int, [_P, _P, _I32, C.POINTER(cb_dims), C.POINTER(cb_layer_w), _P, _P, _SZ, _P]),
    "cb_blend_layer": (C.c_int, [C.POINTER(cb_dims), C.POINTER(cb_layer_w), _I32, _P, _P, _I32, _I64, _I64,
                                 _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, C.POINTER(_I32), _P,
                                 C.POINTER(cb_layer_opts), _P, _SZ, _P]),
    "cb_blend_steady_batch": (C.c_int, [C.POINTER(cb_dims), C.POINTER(cb_layer_w), _I32, C.POINTER(_I32), _P, _P,
                                        _I64, _P, _P, _P, _I32, _P, _P, _SZ, _P]),
    "cb_full_prefill": (C.c_int, [C.POINTER(cb_dims), _I32, C.POINTER(cb_layer_w), _P, _P, _I32, _I32,
                                  C.POINTER(_P), C.POINTER(_P), _P, _P, _P, _I32, _P, _SZ, _P]),
    "cb_lmhead_argmax": (C.c_int, [_P, _P, _P, C.POINTER(cb_dims), _P, _P, _P, _SZ, _P]),
    "cb_linear": (C.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _P]),
    "cb_kv_quantize": (C.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _P]),
    "cb_file_read": (C.c_int, [C.c_char_p, C.c_uint64, _P, _SZ, _I32]),
    "cb_selftest_wait": (C.c_int, [_I32, _I32, _P]),
    "cb_copy_async": (C.c_int, [_P, _P, _SZ, _P]),
    "cb_rmsnorm": (C.c_int, [_P, _P, _I64, _P, _I64, _I32, _P, C.c_float, _I32, _I32, _P]),
    "cb_io_error_message": (C.c_char_p, []),
    "cb_rope_shift_q8": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _I32, _P, _I64,
                                   C.POINTER(cb_dims), _P, _I32, _P]),
    "cb_prefetch_layer": (C.c_int, [_P, _P, _SZ, _P, _P]),
    "cb_stream_wait": (C.c_int, [_P, _P]),
    "cb_kernel_launch_count": (_I64, []),
    "cb_profile_begin": (C.c_int, [_I32]),
    "cb_profile_begin_spans": (C.c_int, [_I32]),
    "cb_profile_end": (C.c_int, [C.POINTER(cb_prof_record), _I32, C.POINTER(_I32)]),
}

_LIB = None


def lib():
    """Load the in-tree library (never builds implicitly on the call path)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with non_prefix_kv_gb300.build.build()")
        L = C.CDLL(path)
        for name, (res, args) in _PROTOS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != CB_OK:
        raise CBError(fn, st, lib().cb_last_error_message().decode(errors="replace"))


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def cb_last_cuda_error() -> str:
    """The last failing CUDA runtime call on this thread ("" if none)."""
    return lib().cb_last_cuda_error().decode(errors="replace")


# ---- host helpers -------------------------------------------------------------------------
def cb_hkvd_budget(n_cached: int, ratio: float, n_cand: int) -> int:
    return int(lib().cb_hkvd_budget(n_cached, ratio, n_cand))


def cb_gradual_ratio(r: float, layer: int, check_layer: int, r1_factor: float = 1.5) -> float:
    return float(lib().cb_gradual_ratio(r, layer, check_layer, r1_factor))


def cb_load_controller_ratio(r_min: float, t_load_s: float, t_prefill_s: float) -> float:
    return float(lib().cb_load_controller_ratio(r_min, t_load_s, t_prefill_s))


def cb_workspace_bytes(dims: cb_dims, n_tok: int, m_max: int) -> int:
    out = _SZ(0)
    _check("cb_workspace_bytes", lib().cb_workspace_bytes(C.byref(dims), n_tok, m_max, C.byref(out)))
    return int(out.value)


def cb_sync(stream=None, timeout_s: float = 60.0) -> None:
    _check("cb_sync", lib().cb_sync(_stream(stream), timeout_s))


def cb_shutdown() -> None:
    lib().cb_shutdown()


def _rows(t, n: Optional[int]) -> int:
    """Row count of a buffer for the index checks: given, or the tensor's first dimension."""
    if n is not None:
        return int(n)
    if t is None or isinstance(t, int):
        raise ValueError("the row count of a raw pointer must be given")
    return int(t.shape[0])


# ---- device entry points --------------------------------------------------------------------
def cb_rope_table(cos_sin, max_pos: int, head_dim: int, base: float, stream=None):
    _check("cb_rope_table", lib().cb_rope_table(_ptr(cos_sin), max_pos, head_dim, base, _stream(stream)))


def cb_rope_shift(k_dst, v_dst, k_src, v_src, src_row, delta, n_rows: int, dims: cb_dims, cos_sin,
                  max_pos: int, stream=None, n_src_rows: Optional[int] = None):
    """n_src_rows: rows of k_src/v_src (default: k_src's first dimension)."""
    _check("cb_rope_shift", lib().cb_rope_shift(_ptr(k_dst), _ptr(v_dst), _ptr(k_src), _ptr(v_src),
                                                _ptr(src_row), _rows(k_src, n_src_rows), _ptr(delta), n_rows,
                                                C.byref(dims), _ptr(cos_sin), max_pos, _stream(stream)))


def cb_kv_deviation_topk(k_new, v_new, k_ref, v_ref, new_row, ref_row, n_cand: int, k: int, dev_mode: int,
                         dims: cb_dims, scores, sel, ws, stream=None, n_new_rows: Optional[int] = None,
                         n_ref_rows: Optional[int] = None):
    """n_new_rows / n_ref_rows: rows of k_new and k_ref (default: their first dimension)."""
    _check("cb_kv_deviation_topk", lib().cb_kv_deviation_topk(
        _ptr(k_new), _ptr(v_new), _rows(k_new, n_new_rows), _ptr(k_ref), _ptr(v_ref), _rows(k_ref, n_ref_rows),
        _ptr(new_row), _ptr(ref_row), n_cand, k, dev_mode, C.byref(dims), _ptr(scores), _ptr(sel), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def cb_kv_deviation_topk_noalloc(k_new, v_new, k_ref, v_ref, new_row, ref_row, n_cand: int, k: int,
                                 dev_mode: int, dims: cb_dims, scores, sel, stream=None,
                                 n_new_rows: Optional[int] = None, n_ref_rows: Optional[int] = None):
    """Same as cb_kv_deviation_topk, with the scratch in the library's fixed device array
    (for callers that cannot allocate; at most 65536 candidates; overlapping calls race)."""
    _check("cb_kv_deviation_topk_noalloc", lib().cb_kv_deviation_topk_noalloc(
        _ptr(k_new), _ptr(v_new), _rows(k_new, n_new_rows), _ptr(k_ref), _ptr(v_ref), _rows(k_ref, n_ref_rows),
        _ptr(new_row), _ptr(ref_row), n_cand, k, dev_mode, C.byref(dims), _ptr(scores), _ptr(sel),
        _stream(stream)))


def cb_topk_from_scores(scores, cand, n_cand: int, k: int, sel, ws, stream=None):
    _check("cb_topk_from_scores", lib().cb_topk_from_scores(_ptr(scores), _ptr(cand), n_cand, k, _ptr(sel),
                                                            _ptr(ws), _nbytes(ws), _stream(stream)))


def cb_gather_rows(dst, src, idx, n: int, row_bytes: int, stream=None, n_src_rows: Optional[int] = None):
    """n_src_rows: rows of src that idx may address (default: src's first dimension)."""
    _check("cb_gather_rows", lib().cb_gather_rows(_ptr(dst), _ptr(src), _rows(src, n_src_rows), _ptr(idx), n,
                                                  row_bytes, _stream(stream)))


def cb_scatter_kv(k_cache, v_cache, k_rows, v_rows, dst_idx, src_idx, n: int, dims: cb_dims, stream=None,
                  n_cache_rows: Optional[int] = None, n_src_rows: Optional[int] = None):
    _check("cb_scatter_kv", lib().cb_scatter_kv(_ptr(k_cache), _ptr(v_cache), _rows(k_cache, n_cache_rows),
                                                _ptr(k_rows), _ptr(v_rows), _rows(k_rows, n_src_rows),
                                                _ptr(dst_idx), _ptr(src_idx), n, C.byref(dims),
                                                _stream(stream)))


def cb_selective_qkv(x, rows, pos, M: int, dims: cb_dims, w: cb_layer_w, cos_sin, max_pos: int, q, k, v,
                     ws, stream=None, n_x_rows: Optional[int] = None):
    _check("cb_selective_qkv", lib().cb_selective_qkv(
        _ptr(x), _rows(x, n_x_rows), _ptr(rows), _ptr(pos), M, C.byref(dims), C.byref(w), _ptr(cos_sin), max_pos,
        _ptr(q), _ptr(k), _ptr(v), _ptr(ws), _nbytes(ws), _stream(stream)))


def cb_partial_attention(q, q_pos, M: int, k_cache, v_cache, n_kv: int, dims: cb_dims, out, ws=None,
                         stream=None):
    _check("cb_partial_attention", lib().cb_partial_attention(
        _ptr(q), _ptr(q_pos), M, _ptr(k_cache), _ptr(v_cache), n_kv, C.byref(dims), _ptr(out), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def cb_o_proj_ffn(attn, x_res, M: int, dims: cb_dims, w: cb_layer_w, x_out, ws, stream=None):
    _check("cb_o_proj_ffn", lib().cb_o_proj_ffn(_ptr(attn), _ptr(x_res), M, C.byref(dims), C.byref(w),
                                                _ptr(x_out), _ptr(ws), _nbytes(ws), _stream(stream)))


def cb_blend_layer(dims: cb_dims, w: cb_layer_w, mode: int, x_in, s_in, m_in: int, n_tok: int, n_cached: int,
                   k_cache, v_cache, cos_sin, max_pos: int, k_budget: int, dev_mode: int, sel_override,
                   x_out, s_out, scores_out, ws, stream=None, kv_ready=None, forced_mask=None,
                   n_forced: int = 0, recompute_kv: bool = False, recompute_from: int = 0, x_rows=None,
                   n_x_rows: int = 0, aux=None, x_out_ssq=None, ssq_parts_out: Optional[list] = None, x_in_ssq=None,
                   x_in_ssq_parts: int = 0) -> int:
    """kv_ready: a torch.cuda.Event (or raw cudaEvent_t) the layer waits for just before it
    first touches the cached rows, or None.  forced_mask/n_forced: uncached rows anywhere
    (a uint8 device tensor over the tokens, marking the last row too), or None.
    recompute_from: PRECHECK only, recompute K/V from this row on (0: off).
    x_rows / n_x_rows: PRECHECK only, input row i is x_in[x_rows[i]] (e.g. x_in = the embedding
    table, x_rows = the token ids).
    aux: (stream, fork event, join event) for the CHECK/GRADUAL KV expansion beside the Q GEMM,
    or None.
    x_out_ssq: a float32 device buffer that receives the output rows' partial sums of squares;
    their count is stored in ssq_parts_out[0].  x_in_ssq / x_in_ssq_parts: the same from the
    call that produced x_in (lets the bf16 path with unit attention-norm gains skip the norm)."""
    m_out = _I32(0)
    opts = None
    parts = _I32(0)
    if (kv_ready is not None or forced_mask is not None or recompute_kv or recompute_from or x_rows is not None
            or aux is not None or x_out_ssq is not None or x_in_ssq is not None):
        ev = kv_ready if (kv_ready is None or isinstance(kv_ready, int)) else kv_ready.cuda_event
        ax = (None, None, None) if aux is None else (_stream(aux[0]), _event(aux[1]), _event(aux[2]))
        opts = C.byref(cb_layer_opts(_ptr(forced_mask), n_forced if forced_mask is not None else 0, ev,
                                     1 if recompute_kv else 0, int(recompute_from), _ptr(x_rows),
                                     int(n_x_rows) if x_rows is not None else 0, *ax, _ptr(x_out_ssq),
                                     C.pointer(parts) if x_out_ssq is not None else None, _ptr(x_in_ssq),
                                     int(x_in_ssq_parts) if x_in_ssq is not None else 0))
    _check("cb_blend_layer", lib().cb_blend_layer(
        C.byref(dims), C.byref(w), mode, _ptr(x_in), _ptr(s_in), m_in, n_tok, n_cached, _ptr(k_cache),
        _ptr(v_cache), _ptr(cos_sin), max_pos, k_budget, dev_mode, _ptr(sel_override), _ptr(x_out),
        _ptr(s_out), C.byref(m_out), _ptr(scores_out), opts, _ptr(ws), _nbytes(ws), _stream(stream)))
    if ssq_parts_out is not None:
        ssq_parts_out[:] = [int(parts.value)]
    return int(m_out.value)


def cb_blend_steady_batch(dims: cb_dims, w: cb_layer_w, row0: Sequence[int], x_in, s_in, n_tok: int, k_cache,
                          v_cache, cos_sin, max_pos: int, x_out, ws, stream=None):
    """One steady layer of len(row0) - 1 requests at once (request r: rows [row0[r], row0[r+1]))."""
    arr = (C.c_int32 * len(row0))(*[int(v) for v in row0])
    _check("cb_blend_steady_batch", lib().cb_blend_steady_batch(
        C.byref(dims), C.byref(w), len(row0) - 1, arr, _ptr(x_in), _ptr(s_in), n_tok, _ptr(k_cache), _ptr(v_cache),
        _ptr(cos_sin), max_pos, _ptr(x_out), _ptr(ws), _nbytes(ws), _stream(stream)))


def cb_full_prefill(dims: cb_dims, layers: Sequence[cb_layer_w], embed, tokens, n: int, pos0: int,
                    k_out: Sequence, v_out: Sequence, h_last, x_all, cos_sin, max_pos: int, ws, stream=None):
    L = len(layers)
    arr_w = (cb_layer_w * L)(*layers)
    arr_k = (C.c_void_p * L)(*[_ptr(t) for t in k_out])
    arr_v = (C.c_void_p * L)(*[_ptr(t) for t in v_out])
    _check("cb_full_prefill", lib().cb_full_prefill(
        C.byref(dims), L, arr_w, _ptr(embed), _ptr(tokens), n, pos0, arr_k, arr_v, _ptr(h_last), _ptr(x_all),
        _ptr(cos_sin), max_pos, _ptr(ws), _nbytes(ws), _stream(stream)))


def cb_lmhead_argmax(h, final_norm, w_lm, dims: cb_dims, logits, token, ws, stream=None):
    _check("cb_lmhead_argmax", lib().cb_lmhead_argmax(_ptr(h), _ptr(final_norm), _ptr(w_lm), C.byref(dims),
                                                      _ptr(logits), _ptr(token), _ptr(ws), _nbytes(ws),
                                                      _stream(stream)))


def cb_linear(x, w, y, M: int, N: int, K: int, dtype: int, stream=None):
    _check("cb_linear", lib().cb_linear(_ptr(x), _ptr(w), _ptr(y), M, N, K, dtype, _stream(stream)))


def cb_file_read(path: str, offset: int, dst, nbytes: int, n_threads: int = 8):
    """Read nbytes of the file at offset into dst (a pinned host tensor or raw pointer)."""
    st = lib().cb_file_read(path.encode(), offset, _ptr(dst), nbytes, n_threads)
    if st != CB_OK:
        raise CBError("cb_file_read", st, lib().cb_io_error_message().decode(errors="replace"))


def cb_rmsnorm(out, x, rows, n: int, d: int, gain, eps: float, dtype_in: int, dtype_out: int, stream=None,
               n_x_rows: Optional[int] = None):
    _check("cb_rmsnorm", lib().cb_rmsnorm(_ptr(out), _ptr(x), _rows(x, n_x_rows), _ptr(rows), n, d, _ptr(gain),
                                          eps, dtype_in, dtype_out, _stream(stream)))


def cb_copy_async(dst, src, nbytes: int, stream=None):
    _check("cb_copy_async", lib().cb_copy_async(_ptr(dst), _ptr(src), nbytes, _stream(stream)))


def cb_selftest_wait(max_polls: int, arrive: bool, stream=None):
    _check("cb_selftest_wait", lib().cb_selftest_wait(max_polls, 1 if arrive else 0, _stream(stream)))


def cb_kv_quantize(x, n_rows: int, W: int, dtype: int, codes, scale, zero, stream=None):
    _check("cb_kv_quantize", lib().cb_kv_quantize(_ptr(x), n_rows, W, dtype, _ptr(codes), _ptr(scale), _ptr(zero),
                                                  _stream(stream)))


def cb_rope_shift_q8(k_dst, v_dst, k_codes, v_codes, k_scale, k_zero, v_scale, v_zero, src_row, n_src_rows: int,
                     qrow, n_qrows: int, delta, n_rows: int, dims: cb_dims, cos_sin, max_pos: int, stream=None):
    _check("cb_rope_shift_q8", lib().cb_rope_shift_q8(
        _ptr(k_dst), _ptr(v_dst), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(k_zero), _ptr(v_scale),
        _ptr(v_zero), _ptr(src_row), n_src_rows, _ptr(qrow), n_qrows, _ptr(delta), n_rows, C.byref(dims),
        _ptr(cos_sin), max_pos, _stream(stream)))


def cb_kernel_launch_count() -> int:
    return int(lib().cb_kernel_launch_count())


def cb_profile_begin(max_records: int = 4096):
    _check("cb_profile_begin", lib().cb_profile_begin(max_records))


def cb_profile_begin_spans(max_records: int = 4096):
    _check("cb_profile_begin_spans", lib().cb_profile_begin_spans(max_records))


def cb_profile_end(max_records: int = 4096):
    """Returns a list of dicts {kind, aux, m, n, k, flops, bytes, ms, span_ms}, one per launch."""
    arr = (cb_prof_record * max_records)()
    n = _I32(0)
    _check("cb_profile_end", lib().cb_profile_end(arr, max_records, C.byref(n)))
    return [{"kind": PROF_KINDS.get(r.kind, str(r.kind)), "aux": r.aux, "m": r.m, "n": r.n, "k": r.k,
             "flops": r.flops, "bytes": r.bytes, "ms": r.ms, "span_ms": r.span_ms} for r in arr[:n.value]]


def _event(ev) -> int:
    return ev if isinstance(ev, int) else ev.cuda_event


def cb_prefetch_layer(dev_dst, pinned_src, nbytes: int, side_stream, done_event):
    _check("cb_prefetch_layer", lib().cb_prefetch_layer(_ptr(dev_dst), _ptr(pinned_src), nbytes,
                                                        _stream(side_stream), _event(done_event)))


def cb_stream_wait(stream, event):
    _check("cb_stream_wait", lib().cb_stream_wait(_stream(stream), _event(event)))
