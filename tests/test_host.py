"""CPU-only checks of the C ABI: the library loads, exports every entry point the header
declares, its host-side helpers agree with the oracle, and argument validation rejects bad
calls before any launch (no GPU is touched by these calls)."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import oracle.cacheblend_oracle as O
from non_prefix_kv_gb300 import binding as B
from non_prefix_kv_gb300 import build as nb
from tests.conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "cacheblend.h")


@pytest.fixture(scope="module")
def lib():
    nb.build()
    return B.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cb_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_symbols()
    for n in ["cb_rope_shift", "cb_kv_deviation_topk", "cb_gather_rows", "cb_selective_qkv",
              "cb_partial_attention", "cb_scatter_kv", "cb_blend_layer", "cb_full_prefill"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(nb.LIB)
    missing = [n for n in declared_symbols() if not hasattr(raw, n)]
    assert not missing, missing
    # and the binding wraps every one of them under the same name
    for n in declared_symbols():
        assert n in B._PROTOS


def test_budget_matches_oracle(lib):
    for n, r, k in read_golden("budget_table.txt"):
        assert B.cb_hkvd_budget(int(n), float(r), 1 << 40) == int(k)
    g = np.random.default_rng(0)
    for _ in range(2000):
        n = int(g.integers(0, 20000))
        r = float(g.choice([0.0, 1.0, g.random(), 0.05, 0.1, 0.15, 0.18]))
        cand = int(g.integers(0, n + 1))
        assert B.cb_hkvd_budget(n, r, cand) == O.budget(n, r, cand)
    assert B.cb_hkvd_budget(10, 1.5, 10) == -1
    assert B.cb_hkvd_budget(10, -0.1, 10) == -1


def test_gradual_schedule_matches_oracle(lib):
    for r in [0.05, 0.15, 0.18, 0.7, 1.0]:
        sched = O.ratio_schedule(r, 32, 1, True)
        for l in range(32):
            got = B.cb_gradual_ratio(r, l, 1, 1.5)
            if sched[l] is None:
                assert got == -1.0
            else:
                assert got == sched[l]


def test_load_controller(lib):
    assert B.cb_load_controller_ratio(0.15, 0.016, 0.020) == O.optimal_ratio(0.15, 0.016, 0.020)
    assert B.cb_load_controller_ratio(0.15, 0.001, 0.020) == 0.15


def test_status_strings(lib):
    for code in range(11):
        assert lib.cb_status_string(code)
    assert lib.cb_status_string(99) == b"unknown status"


def _dims(**kw):
    base = dict(d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, d_ff=688, vocab=1024, rope_base=1e4,
                rms_eps=1e-5, dtype=B.CB_F32)
    base.update(kw)
    return B.cb_dims(**base)


def test_workspace_query_and_dims_validation(lib):
    n = B.cb_workspace_bytes(_dims(), 416, 416)
    assert n > 416 * 256 * 4
    with pytest.raises(B.CBError) as e:
        B.cb_workspace_bytes(_dims(dtype=7), 416, 416)
    assert e.value.status == 3
    with pytest.raises(B.CBError) as e:
        B.cb_workspace_bytes(_dims(n_kv_heads=3), 416, 416)
    assert e.value.status == 2
    with pytest.raises(B.CBError) as e:
        B.cb_workspace_bytes(_dims(head_dim=48), 416, 416)
    assert e.value.status == 8


FAKE = 0x10000   # never dereferenced: every call below fails validation before launching


def test_entry_points_reject_bad_arguments_before_launch(lib):
    d = _dims()
    w = B.cb_layer_w(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    st = lib.cb_rope_shift(FAKE, None, FAKE, FAKE, None, 10, None, 10, ctypes.byref(d), FAKE, 100, None)
    assert st == 1        # delta NULL
    st = lib.cb_rope_shift(FAKE, FAKE, FAKE, None, None, 10, FAKE, 10, ctypes.byref(d), FAKE, 100, None)
    assert st == 1        # v_dst without v_src
    st = lib.cb_rope_shift(FAKE, FAKE, FAKE, FAKE, None, 9, FAKE, 10, ctypes.byref(d), FAKE, 100, None)
    assert st == 2        # no row map and fewer source rows than destination rows
    st = lib.cb_kv_deviation_topk(FAKE, FAKE, 10, FAKE, FAKE, 10, None, None, 10, 11, 0, ctypes.byref(d), None,
                                  FAKE, FAKE, 1 << 20, None)
    assert st == 2        # k > n_cand
    st = lib.cb_kv_deviation_topk(FAKE, FAKE, 10, FAKE, FAKE, 9, None, None, 10, 5, 0, ctypes.byref(d), None,
                                  FAKE, FAKE, 1 << 20, None)
    assert st == 2        # no ref_row map and fewer cached rows than candidates
    st = lib.cb_topk_from_scores(FAKE, None, 100, 5, FAKE, FAKE, 16, None)
    assert st == 4        # workspace too small
    st = lib.cb_gather_rows(FAKE, FAKE, 3, None, 3, 6, None)
    assert st == 2        # row_bytes not a multiple of 4
    st = lib.cb_gather_rows(FAKE, FAKE, 2, None, 3, 8, None)
    assert st == 2        # no index and fewer source rows than rows to copy
    st = lib.cb_scatter_kv(FAKE, FAKE, -1, FAKE, FAKE, 10, FAKE, None, 3, ctypes.byref(d), None)
    assert st == 2        # negative cache height
    st = lib.cb_rmsnorm(FAKE, FAKE, 4, None, 5, 64, FAKE, ctypes.c_float(1e-5), B.CB_BF16, B.CB_BF16, None)
    assert st == 2        # no row map and fewer input rows than outputs
    m_out = ctypes.c_int32(-1)
    args = lambda mode, m_in, k, ws_bytes=1 << 40: (ctypes.byref(d), ctypes.byref(w), mode, FAKE, None, m_in, 416,
                                                   384, FAKE, FAKE, FAKE, 416, k, 0, None, FAKE + 64, FAKE,
                                                   ctypes.byref(m_out), None, None, FAKE, ws_bytes, None)
    assert lib.cb_blend_layer(*args(B.CB_LAYER_CHECK, 416, 385)) == 2     # k > candidates (384)
    assert lib.cb_blend_layer(*args(B.CB_LAYER_CHECK, 400, 5)) == 2       # CHECK needs all rows
    assert lib.cb_blend_layer(*args(B.CB_LAYER_PRECHECK, 416, 0, 100)) == 4
    assert lib.cb_blend_layer(*args(9, 416, 0)) == 1
    # recompute_from: PRECHECK only, within [0, n_cached] (384 cached rows)
    def with_opts(mode, m_in, k, rfrom, rkv=0):
        o = B.cb_layer_opts(None, 0, None, rkv, rfrom)
        a = list(args(mode, m_in, k))
        a[19] = ctypes.byref(o)
        return lib.cb_blend_layer(*a)
    assert with_opts(B.CB_LAYER_CHECK, 416, 5, 128) == 1
    assert with_opts(B.CB_LAYER_PRECHECK, 416, 0, 385) == 2
    assert with_opts(B.CB_LAYER_PRECHECK, 416, 0, -1) == 2
    assert with_opts(B.CB_LAYER_PRECHECK, 416, 0, 128, rkv=1) == 1
    o = B.cb_layer_opts(None, 0, None, 0, 0, None, 0, FAKE, None, None)
    a = list(args(B.CB_LAYER_CHECK, 416, 5))
    a[19] = ctypes.byref(o)
    assert lib.cb_blend_layer(*a) == 1   # aux stream without its two events
    assert m_out.value == -1          # nothing reported for a rejected call
    st = lib.cb_blend_layer(ctypes.byref(d), ctypes.byref(w), 0, FAKE, None, 416, 416, 384, FAKE, FAKE, FAKE,
                            100, 0, 0, None, FAKE + 64, FAKE, ctypes.byref(m_out), None, None, FAKE, 1 << 40, None)
    assert st == 2                    # rope table shorter than the sequence
    assert b"rope table" in lib.cb_last_error_message()
    st = lib.cb_linear(FAKE, FAKE, FAKE, 4, 24, 64, B.CB_BF16, None)
    assert st == 8                    # bf16 N % 16


def test_cuda_failures_are_reported_with_the_failing_call(lib):
    """A failing CUDA runtime call comes back as CB_ERR_CUDA, and cb_last_cuda_error names
    the error and the call.  Without a GPU, cb_sync's stream query is such a call."""
    import torch
    st = lib.cb_sync(None, ctypes.c_double(1.0))
    if torch.cuda.is_available():
        assert st == 0
    else:
        assert st == 6
        msg = B.cb_last_cuda_error()
        assert "cudaStreamQuery" in msg and "cuda" in msg.lower()


def test_misaligned_buffers_are_refused_before_launch(lib):
    """Device buffers the kernels move in 16-byte vectors must start on a 16-byte boundary:
    a misaligned one is refused on the host (CB_ERR_INVALID_ARG, nothing launched) instead of
    faulting on the GPU.  The row copies need only 4 bytes."""
    d = _dims()
    odd = FAKE + 8          # 8-byte aligned, not 16
    st = lib.cb_rmsnorm(FAKE, odd, 4, None, 4, 64, FAKE, ctypes.c_float(1e-5), B.CB_BF16, B.CB_BF16, None)
    assert st == 1 and b"16-byte" in lib.cb_last_error_message()
    st = lib.cb_rope_shift(odd, None, FAKE, None, None, 10, FAKE, 10, ctypes.byref(d), FAKE, 100, None)
    assert st == 1
    st = lib.cb_linear(FAKE, odd, FAKE, 4, 32, 64, B.CB_BF16, None)
    assert st == 1
    w = B.cb_layer_w(None, FAKE, odd, None, FAKE, FAKE)
    st = lib.cb_o_proj_ffn(FAKE, FAKE, 4, ctypes.byref(d), ctypes.byref(w), FAKE + 64, FAKE, 1 << 30, None)
    assert st == 1 and b"layer weights" in lib.cb_last_error_message()
    w = B.cb_layer_w(None, FAKE, FAKE, None, FAKE, FAKE)
    st = lib.cb_o_proj_ffn(FAKE, odd, 4, ctypes.byref(d), ctypes.byref(w), FAKE + 64, FAKE, 1 << 30, None)
    assert st == 1 and b"o_proj_ffn" in lib.cb_last_error_message()
    st = lib.cb_partial_attention(odd, FAKE, 4, FAKE, FAKE, 16, ctypes.byref(d), FAKE, None, 0, None)
    assert st == 1
    st = lib.cb_gather_rows(FAKE, FAKE + 2, 3, None, 3, 8, None)
    assert st == 1 and b"4-byte" in lib.cb_last_error_message()
    m_out = ctypes.c_int32(-1)
    st = lib.cb_blend_layer(ctypes.byref(d), ctypes.byref(w), B.CB_LAYER_PRECHECK, odd, None, 416, 416, 384, FAKE,
                            FAKE, FAKE, 416, 0, 0, None, FAKE + 64, FAKE, ctypes.byref(m_out), None, None, FAKE,
                            1 << 40, None)
    assert st == 1 and m_out.value == -1


def test_shutdown_releases_state_and_the_library_stays_usable(lib):
    """cb_shutdown empties the per-device caches; every later call rebuilds what it needs."""
    d = _dims()
    before = B.cb_workspace_bytes(d, 416, 416)
    B.cb_shutdown()
    B.cb_shutdown()                      # twice in a row is harmless
    assert B.cb_workspace_bytes(d, 416, 416) == before
    assert B.cb_hkvd_budget(3840, 0.15, 3840) == 576
    st = lib.cb_gather_rows(FAKE, FAKE, 3, None, 3, 6, None)
    assert st == 2 and b"row_bytes" in lib.cb_last_error_message()


def test_layer_plan_sizes_match_oracle_selection(lib):
    from non_prefix_kv_gb300 import engine as E
    from non_prefix_kv_gb300 import synth
    wl = synth.WORKLOADS["llama7b_32_4k"]
    ratios = O.ratio_schedule(wl.ratio, wl.shape.n_layers, 1, True)
    plan = E.layer_plan(wl.shape, wl.n_tokens, wl.n_cached, ratios, gradual=True)
    n_forced = wl.n_tokens - wl.n_cached
    m = wl.n_tokens
    for l, (mode, k) in enumerate(plan):
        if l == 0:
            assert mode == B.CB_LAYER_PRECHECK
            continue
        n_cand = wl.n_cached if l == 1 else m - n_forced
        assert k == O.budget(wl.n_cached, ratios[l], n_cand)
        m = k + n_forced
    assert plan[1][1] == O.budget(3840, min(1.0, 1.5 * 0.15))


def test_file_read_ranges_threads_and_errors(lib, tmp_path):
    """The storage-tier reader returns exactly the requested byte range for any split over
    threads (pieces of at least 4 MB), and reports missing files and short files as
    CB_ERR_IO without touching the destination beyond the range."""
    g = np.random.default_rng(3)
    data = g.integers(0, 256, (9 << 20) + 12345, dtype=np.uint8)
    path = tmp_path / "store.bin"
    data.tofile(path)
    for off, n, nt in [(0, len(data), 1), (0, len(data), 8), (777, (6 << 20) + 3, 3), (len(data) - 5, 5, 4),
                       (123, 0, 2)]:
        buf = np.full(n + 16, 0xAB, np.uint8)
        B.cb_file_read(str(path), off, buf.ctypes.data, n, nt)
        np.testing.assert_array_equal(buf[:n], data[off:off + n])
        assert np.all(buf[n:] == 0xAB)
    buf = np.zeros(64, np.uint8)
    with pytest.raises(B.CBError) as e:
        B.cb_file_read(str(tmp_path / "missing.bin"), 0, buf.ctypes.data, 64)
    assert e.value.status == 10 and "missing.bin" in str(e.value)
    with pytest.raises(B.CBError) as e:
        B.cb_file_read(str(path), len(data) - 10, buf.ctypes.data, 64)
    assert e.value.status == 10 and "end of file" in str(e.value)


def test_precheck_split_balances_load_and_recompute():
    """The pre-check split: loading X rows (host link, then re-positioning) takes as long as
    RMSNorm + Q for every row and K/V for the other rows, to within one 64-row step; a
    faster link loads more rows, a faster GEMM recomputes more; clamped to the cached rows."""
    from non_prefix_kv_gb300 import engine as E
    from non_prefix_kv_gb300 import synth
    shape = synth.WORKLOADS["llama7b_layer_4k"].shape
    N, nc = 4096, 3840
    d, qc, W = shape.d_model, shape.q_width, shape.kv_width

    def sides(x, link, tf, hbm):
        R, L, H = tf * 1e12, link * 1e9, hbm * 1e9
        comp = 2.0 * N * d * qc / R + 2.0 * N * d * 2 / H + (N - x) * 2.0 * d * 2 * W / R
        load = x * (2.0 * W * 2 / L + 4.0 * W * 2 / H)
        return comp, load

    x = E.precheck_split_rows(shape, N, nc, 200.0, 1800.0, 6800.0)
    assert x % 64 == 0 and 0 < x < nc
    c0, l0 = sides(x, 200.0, 1800.0, 6800.0)
    c1, l1 = sides(x + 64, 200.0, 1800.0, 6800.0)
    assert l0 <= c0 and l1 > c1                # the largest 64-row multiple that still hides
    assert E.precheck_split_rows(shape, N, nc, 400.0, 1800.0, 6800.0) > x
    assert E.precheck_split_rows(shape, N, nc, 200.0, 3600.0, 6800.0) < x
    assert E.precheck_split_rows(shape, N, nc, 1e6, 1800.0, 6800.0) == nc
    # an 8-bit store moves one byte per element over the link and its decode reads the codes
    # and writes bf16: a row costs less to load, so more rows are loaded
    x8 = E.precheck_split_rows(shape, N, nc, 200.0, 1800.0, 6800.0, store_esz=1)
    R, L, H = 1800.0e12, 200.0e9, 6800.0e9
    comp8 = lambda x: 2.0 * N * d * qc / R + 2.0 * N * d * 2 / H + (N - x) * 2.0 * d * 2 * W / R  # noqa: E731
    load8 = lambda x: x * (2.0 * W * 1 / L + 2.0 * W * (1 + 2) / H)  # noqa: E731
    assert x8 > x and x8 % 64 == 0
    assert load8(x8) <= comp8(x8) and (x8 == nc or load8(x8 + 64) > comp8(x8 + 64))


def test_contiguous_pool_ranges():
    """The pool rows a partial pre-check load copies: runs of consecutive pool rows in the
    request's slot order (chunks may come from anywhere in the pool, in any order)."""
    from non_prefix_kv_gb300 import engine as E
    assert E.contiguous_ranges([]) == []
    assert E.contiguous_ranges([5]) == [(5, 1)]
    assert E.contiguous_ranges(range(10, 20)) == [(10, 10)]
    # chunk 2 (rows 1280..1919) then chunk 0 (0..639), a partial third chunk (640..703)
    rows = list(range(1280, 1920)) + list(range(0, 640)) + list(range(640, 704))
    assert E.contiguous_ranges(rows) == [(1280, 640), (0, 704)]
    # a repeated chunk is two runs
    assert E.contiguous_ranges(list(range(0, 4)) + list(range(0, 4))) == [(0, 4), (0, 4)]


def test_whole_step_roofline_floor():
    """bench.py's step floor: each launch at the longer of bytes / bandwidth and FLOPs / rate,
    attention from the step's FLOPs, averaged over the profiled steps."""
    import bench
    recs = [{"kind": "gemm", "bytes": 1e9, "flops": 2e12},        # 1.0 ms at 2 PFLOP/s (> 0.1 ms of bytes)
            {"kind": "rmsnorm", "bytes": 5e9, "flops": 1e9},       # 0.5 ms at 10 TB/s
            {"kind": "attention", "bytes": 1e9, "flops": 9e12},    # replaced by the step's FLOPs
            {"kind": "gemm", "bytes": 1e9, "flops": 2e12},         # the second profiled step
            {"kind": "rmsnorm", "bytes": 5e9, "flops": 1e9}]
    got = bench.whole_step_floor_ms(recs, 2, 1e12, 10000.0, 2000.0)
    assert abs(got - 2.0) < 1e-9                           # (1.0 + 0.5 + 1.0 + 0.5) / 2 + 0.5


def test_token_ids_are_checked_on_the_host():
    from non_prefix_kv_gb300 import engine as E
    np.testing.assert_array_equal(E.check_token_ids([0, 5, 1023], 1024), [0, 5, 1023])
    for bad in ([0, 1024], [-1, 3], [[1, 2]]):
        with pytest.raises(ValueError):
            E.check_token_ids(bad, 1024)


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference runs the oracle on the host cores and prints one JSON line
    with the contract's keys: ms_per_step is the measured step (the bounded sample), and the
    workload's throughput extrapolated from it is labelled as such."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["extrapolated"] is True and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # the measured step is the sample; the whole step's time is an estimate several times longer
    assert 0 < line["ms_per_step"] < line["ms_per_full_step_extrapolated"]
    assert abs(line["value"] - 4096 / (line["ms_per_full_step_extrapolated"] / 1e3)) < 1e-6 * line["value"]
