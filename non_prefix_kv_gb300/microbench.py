"""Per-entry-point microbenchmark: times one library call at a given shape with CUDA events
and prints achieved TFLOP/s or GB/s against the algorithmic work.  Also the small, single-
kernel command that ncu captures are taken on.

  python -m non_prefix_kv_gb300.microbench gemm --m 4096 --n 8192 --k 4096 [--epi swiglu]
  python -m non_prefix_kv_gb300.microbench attention --m 832 --n 4096 --heads 32 --kv-heads 32 --hd 128
  python -m non_prefix_kv_gb300.microbench rope_shift --rows 3840 --width 4096
  python -m non_prefix_kv_gb300.microbench deviation --cand 3840 --width 4096 --k 576
  python -m non_prefix_kv_gb300.microbench rope_shift_q8 --rows 3840 --width 4096
  python -m non_prefix_kv_gb300.microbench check_layer --rows 4096 --k 576
  python -m non_prefix_kv_gb300.microbench rmsnorm --rows 4096 --width 4096
  python -m non_prefix_kv_gb300.microbench gather --rows 4096 --width 4096 --n 32000
  python -m non_prefix_kv_gb300.microbench lmhead --width 4096 --n 32000
"""
from __future__ import annotations

import argparse
import json
import sys

import numpy as np
import torch

from . import binding as B
from . import build as nb
from . import engine as E
from .synth import ModelShape


def _time(fn, iters: int, warmup: int):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def run(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("what", choices=["gemm", "o_proj_ffn", "attention", "rope_shift", "rope_shift_q8", "deviation",
                                    "check_layer",
                                    "rmsnorm", "gather", "lmhead"])
    p.add_argument("--m", type=int, default=4096)
    p.add_argument("--n", type=int, default=8192)
    p.add_argument("--k", type=int, default=4096)
    p.add_argument("--epi", choices=["store", "swiglu"], default="store")
    p.add_argument("--unit-gains", action="store_true",
                   help="swiglu: NULL norm gains, as the bf16 step runs it (the FFN norm folded into the "
                        "gate/up GEMM, the O-projection leaving its rows' sums of squares)")
    p.add_argument("--host-src", action="store_true", help="rope_shift: sources in pinned host memory")
    p.add_argument("--heads", type=int, default=32)
    p.add_argument("--kv-heads", type=int, default=32)
    p.add_argument("--hd", type=int, default=128)
    p.add_argument("--pos-const", type=int, default=None,
                   help="attention: every query at this position (each query tile visits the same key tiles)")
    p.add_argument("--rows", type=int, default=3840)
    p.add_argument("--width", type=int, default=4096)
    p.add_argument("--cand", type=int, default=3840)
    p.add_argument("--iters", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    a = p.parse_args(argv)
    nb.build()
    B.lib()
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    bf = torch.bfloat16
    out = {"what": a.what}
    if a.what == "gemm":
        if a.epi == "store":
            x = torch.randn(a.m, a.k, device="cuda", generator=g).to(bf)
            w = (torch.randn(a.n, a.k, device="cuda", generator=g) * 0.02).to(bf)
            y = torch.empty(a.m, a.n, device="cuda", dtype=bf)
            ms = _time(lambda: B.cb_linear(x, w, y, a.m, a.n, a.k, B.CB_BF16), a.iters, a.warmup)
            fl = 2.0 * a.m * a.n * a.k
        else:
            # gate/up GEMM with the fused SwiGLU epilogue, inside the O-proj + FFN call
            shape = ModelShape(1, a.k, 1, 1, 128, a.n, 64, dtype="bf16")
            dims = E.make_dims(shape)
            lw = {"attn_norm": torch.ones(a.k, device="cuda", dtype=bf),
                  "wqkv": torch.zeros(384, a.k, device="cuda", dtype=bf),
                  "wo": (torch.randn(a.k, 128, device="cuda", generator=g) * 0.02).to(bf),
                  "ffn_norm": torch.ones(a.k, device="cuda", dtype=bf),
                  "w_gate_up": (torch.randn(2 * a.n, a.k, device="cuda", generator=g) * 0.02).to(bf),
                  "w_down": (torch.randn(a.k, a.n, device="cuda", generator=g) * 0.02).to(bf)}
            cw = B.cb_layer_w(*(0 if a.unit_gains and k.endswith("_norm") else lw[k].data_ptr()
                                for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate_up", "w_down")))
            attn = torch.randn(a.m, 128, device="cuda", generator=g).to(bf)
            x = torch.randn(a.m, a.k, device="cuda", generator=g).to(bf)
            y = torch.empty_like(x)
            ws = torch.empty(B.cb_workspace_bytes(dims, a.m, a.m), dtype=torch.uint8, device="cuda")
            ms = _time(lambda: B.cb_o_proj_ffn(attn, x, a.m, dims, cw, y, ws), a.iters, a.warmup)
            fl = 2.0 * a.m * a.k * (128 + 3 * a.n)
        out.update(ms=ms, tflops=fl / (ms / 1e3) / 1e12, m=a.m, n=a.n, k=a.k, epi=a.epi, unit_gains=a.unit_gains)
    elif a.what == "o_proj_ffn":
        # the O-projection + residual and the SwiGLU FFN of --m rows, d = --k, --heads heads of 128,
        # F = --n, unit norm gains (the FFN norm folded into the gate/up GEMM, as in the bf16 step);
        # per-launch times from the library's launch profile
        shape = ModelShape(1, a.k, a.heads, a.heads, 128, a.n, 64, dtype="bf16")
        dims = E.make_dims(shape)
        qc = a.heads * 128

        def rnd(*sz, std=0.02):
            return (torch.randn(*sz, device="cuda", generator=g) * std).to(bf)
        lw = {"wqkv": rnd(3 * qc, a.k), "wo": rnd(a.k, qc), "w_gate_up": rnd(2 * a.n, a.k), "w_down": rnd(a.k, a.n)}
        cw = B.cb_layer_w(0, lw["wqkv"].data_ptr(), lw["wo"].data_ptr(), 0, lw["w_gate_up"].data_ptr(),
                          lw["w_down"].data_ptr())
        attn = rnd(a.m, qc, std=1.0)
        x = rnd(a.m, a.k, std=1.0)
        y = torch.empty_like(x)
        ws = torch.empty(B.cb_workspace_bytes(dims, a.m, a.m), dtype=torch.uint8, device="cuda")
        call = lambda: B.cb_o_proj_ffn(attn, x, a.m, dims, cw, y, ws)   # noqa: E731
        ms = _time(call, a.iters, a.warmup)
        B.cb_profile_begin(64 * a.iters)
        for _ in range(a.iters):
            call()
        torch.cuda.synchronize()
        recs = B.cb_profile_end(64 * a.iters)
        per = {}
        for r in recs:
            key = "%dx%dx%d" % (r["m"], r["n"], r["k"])
            t = per.setdefault(key, [0, 0.0, r["flops"]])
            t[0] += 1
            t[1] += r["ms"]
        launches = {k: {"us": 1e3 * v[1] / v[0], "tflops": v[2] / (v[1] / v[0] / 1e3) / 1e12} for k, v in per.items()}
        fl = 2.0 * a.m * a.k * (qc + 3 * a.n)
        out.update(ms=ms, tflops=fl / (ms / 1e3) / 1e12, m=a.m, d=a.k, heads=a.heads, f=a.n, launches=launches)
    elif a.what == "attention":
        shape = ModelShape(1, 256, a.heads, a.kv_heads, a.hd, 256, 64, dtype="bf16")
        dims = E.make_dims(shape)
        n = a.n
        K = torch.randn(n, a.kv_heads * a.hd, device="cuda", generator=g).to(bf)
        V = torch.randn(n, a.kv_heads * a.hd, device="cuda", generator=g).to(bf)
        q = torch.randn(a.m, a.heads * a.hd, device="cuda", generator=g).to(bf)
        rng = np.random.default_rng(0)
        if a.pos_const is not None:
            pos = np.full(a.m, min(max(a.pos_const, 0), n - 1), dtype=np.int64)
        else:
            pos = np.sort(rng.choice(n, a.m, replace=False)) if a.m < n else np.arange(n)[:a.m]
            pos[-1] = n - 1
        q_pos = torch.from_numpy(pos.astype(np.int32)).cuda()
        o = torch.empty_like(q)
        ms = _time(lambda: B.cb_partial_attention(q, q_pos, a.m, K, V, n, dims, o), a.iters, a.warmup)
        fl = 4.0 * a.heads * a.hd * float(np.sum(pos + 1))
        out.update(ms=ms, tflops=fl / (ms / 1e3) / 1e12, m=a.m, n=n)
    elif a.what == "rope_shift":
        hd = a.hd
        shape = ModelShape(1, 256, a.width // hd, a.width // hd, hd, 256, 64, dtype="bf16")
        dims = E.make_dims(shape)
        tab = torch.empty(16384 * hd, device="cuda")
        B.cb_rope_table(tab, 16384, hd, 1e4)
        ks = torch.randn(a.rows, a.width, device="cuda", generator=g).to(bf)
        vs = torch.randn(a.rows, a.width, device="cuda", generator=g).to(bf)
        if a.host_src:
            ks, vs = ks.cpu().pin_memory(), vs.cpu().pin_memory()
        kd, vd = torch.empty_like(ks), torch.empty_like(vs)
        delta = torch.full((a.rows,), 1280, dtype=torch.int32, device="cuda")
        ms = _time(lambda: B.cb_rope_shift(kd, vd, ks, vs, None, delta, a.rows, dims, tab, 16384), a.iters,
                   a.warmup)
        by = 4.0 * a.rows * a.width * 2
        out.update(ms=ms, gbs=by / (ms / 1e3) / 1e9, rows=a.rows, width=a.width, host_src=a.host_src)
    elif a.what == "rope_shift_q8":
        # decode + re-rotation of an 8-bit store of 6 chunks into rows of the blended cache
        hd = a.hd
        shape = ModelShape(1, 256, a.width // hd, a.width // hd, hd, 256, 64, dtype="bf16")
        dims = E.make_dims(shape)
        tab = torch.empty(16384 * hd, device="cuda")
        B.cb_rope_table(tab, 16384, hd, 1e4)
        kq = torch.randint(0, 256, (a.rows, a.width), device="cuda", generator=g, dtype=torch.uint8)
        vq = torch.randint(0, 256, (a.rows, a.width), device="cuda", generator=g, dtype=torch.uint8)
        tabs = [torch.rand(6, a.width, device="cuda", generator=g) * 0.01 for _ in range(4)]
        qrow = (torch.arange(a.rows, device="cuda", dtype=torch.int32) * 6) // a.rows
        delta = qrow * 640
        kd = torch.empty(a.rows, a.width, device="cuda", dtype=bf)
        vd = torch.empty_like(kd)
        ms = _time(lambda: B.cb_rope_shift_q8(kd, vd, kq, vq, tabs[0], tabs[1], tabs[2], tabs[3], None, a.rows,
                                              qrow, 6, delta, a.rows, dims, tab, 16384), a.iters, a.warmup)
        by = 2.0 * a.rows * a.width * (1 + 2)
        out.update(ms=ms, gbs=by / (ms / 1e3) / 1e9, rows=a.rows, width=a.width)
    elif a.what == "rmsnorm":
        x = torch.randn(a.rows, a.width, device="cuda", generator=g).to(bf)
        gain = torch.ones(a.width, device="cuda", dtype=bf)
        y = torch.empty_like(x)
        ms = _time(lambda: B.cb_rmsnorm(y, x, None, a.rows, a.width, gain, 1e-5, B.CB_BF16, B.CB_BF16), a.iters,
                   a.warmup)
        by = 4.0 * a.rows * a.width
        out.update(ms=ms, gbs=by / (ms / 1e3) / 1e9, rows=a.rows, width=a.width)
    elif a.what == "gather":
        # embedding gather: rows of a [n, width] table at uniform random token ids
        table = torch.randn(a.n, a.width, device="cuda", generator=g).to(bf)
        ids = torch.randint(0, a.n, (a.rows,), device="cuda", generator=g, dtype=torch.int32)
        y = torch.empty(a.rows, a.width, device="cuda", dtype=bf)
        ms = _time(lambda: B.cb_gather_rows(y, table, ids, a.rows, a.width * 2), a.iters, a.warmup)
        by = 4.0 * a.rows * a.width
        out.update(ms=ms, gbs=by / (ms / 1e3) / 1e9, rows=a.rows, width=a.width, table_rows=a.n)
    elif a.what == "lmhead":
        # final RMSNorm of one row, [n, width] lm_head GEMV and argmax
        shape = ModelShape(1, a.width, a.width // 128, a.width // 128, 128, 256, a.n, dtype="bf16")
        dims = E.make_dims(shape)
        h = torch.randn(a.width, device="cuda", generator=g).to(bf)
        fn = torch.ones(a.width, device="cuda", dtype=bf)
        w = (torch.randn(a.n, a.width, device="cuda", generator=g) * 0.02).to(bf)
        tok = torch.empty(1, dtype=torch.int32, device="cuda")
        ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
        ms = _time(lambda: B.cb_lmhead_argmax(h, fn, w, dims, None, tok, ws), a.iters, a.warmup)
        by = 2.0 * a.n * a.width
        out.update(ms=ms, gbs=by / (ms / 1e3) / 1e9, vocab=a.n, width=a.width)
    elif a.what == "check_layer":
        # the check layer at the 7B shape: K/V GEMM over every row with the deviation in its
        # epilogue, top-k, KV expansion, Q of the selection, attention, O-proj + FFN
        shape = ModelShape(2, 4096, 32, 32, 128, 11008, 32000, dtype="bf16")
        dims = E.make_dims(shape)
        N, n_cached, k = a.rows, a.rows - 256, a.k

        def rnd(*sz, std=0.02):
            return (torch.randn(*sz, device="cuda", generator=g) * std).to(bf)
        lw = {"attn_norm": torch.ones(4096, device="cuda", dtype=bf), "wqkv": rnd(12288, 4096),
              "wo": rnd(4096, 4096), "ffn_norm": torch.ones(4096, device="cuda", dtype=bf),
              "w_gate_up": rnd(22016, 4096), "w_down": rnd(4096, 11008)}
        cw = B.cb_layer_w(*(lw[n].data_ptr() for n in ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate_up",
                                                       "w_down")))
        x = rnd(N, 4096, std=1.0)
        kc, vc = rnd(N, 4096, std=0.5), rnd(N, 4096, std=0.5)
        tab = torch.empty(N * 128, device="cuda")
        B.cb_rope_table(tab, N, 128, 1e4)
        xo = torch.empty_like(x)
        so = torch.empty(N, dtype=torch.int32, device="cuda")
        ws = torch.empty(B.cb_workspace_bytes(dims, N, N), dtype=torch.uint8, device="cuda")
        ms = _time(lambda: B.cb_blend_layer(dims, cw, B.CB_LAYER_CHECK, x, None, N, N, n_cached, kc, vc, tab, N, k,
                                            B.CB_DEV_KV, None, xo, so, None, ws), a.iters, a.warmup)
        out.update(ms=ms, rows=N, k=k)
    else:
        hd = a.hd
        shape = ModelShape(1, 256, a.width // hd, a.width // hd, hd, 256, 64, dtype="bf16")
        dims = E.make_dims(shape)
        tens = [torch.randn(a.cand, a.width, device="cuda", generator=g).to(bf) for _ in range(4)]
        sc = torch.empty(a.cand, device="cuda")
        sel = torch.empty(max(a.k, 1), dtype=torch.int32, device="cuda")
        ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
        ms = _time(lambda: B.cb_kv_deviation_topk(tens[0], tens[1], tens[2], tens[3], None, None, a.cand, a.k, 0,
                                                  dims, sc, sel, ws), a.iters, a.warmup)
        by = 4.0 * a.cand * a.width * 2
        out.update(ms=ms, gbs=by / (ms / 1e3) / 1e9, cand=a.cand, width=a.width, k=a.k)
    B.cb_sync(None)
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(run())
