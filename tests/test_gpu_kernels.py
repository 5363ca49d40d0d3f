"""Per-entry-point parity of the CUDA path against the CPU oracle on seeded inputs.
Index and copy results are compared bit-exactly; floats by relative Frobenius error."""
import numpy as np
import pytest

import oracle.cacheblend_oracle as O
from non_prefix_kv_gb300 import synth
from tests.gpu_util import TOL, dev, dev_i32, ensure_lib, host, rel, tdt, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    torch_mod()
    ensure_lib()
    from non_prefix_kv_gb300 import binding
    return binding


def dims_for(B, shape):
    from non_prefix_kv_gb300 import engine as E
    return E.make_dims(shape)


SHAPE_F32 = synth.ModelShape(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, d_ff=688,
                             vocab=1024, dtype="f32", w_std=0.05)
SHAPE_BF16 = synth.ModelShape(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=64, d_ff=1024,
                              vocab=2048, dtype="bf16", w_std=0.04)
# a mid-size GQA layer: at 640 rows every GEMM spans several tiles in M, N and K
SHAPE_BF16_MID = synth.ModelShape(n_layers=2, d_model=2048, n_heads=16, n_kv_heads=4, head_dim=128, d_ff=2048,
                                  vocab=2048, dtype="bf16", w_std=0.02)


def rope_tab(B, max_pos, hd, base):
    torch = torch_mod()
    t = torch.empty(max_pos * hd, dtype=torch.float32, device="cuda")
    B.cb_rope_table(t, max_pos, hd, base)
    return t


# ------------------------------------------------------------------------------ RoPE
@pytest.mark.parametrize("base", [1e4, 5e6])
def test_rope_table(B, base):
    hd, P = 128, 16384
    t = host(rope_tab(B, P, hd, base)).reshape(P, hd // 2, 2)
    pos = np.arange(P)[:, None]
    ang = pos * O.rope_theta(hd, base)
    assert np.max(np.abs(t[..., 0] - np.cos(ang))) < 2e-7
    assert np.max(np.abs(t[..., 1] - np.sin(ang))) < 2e-7


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_shift_gather_and_negative_offsets(B, dtype):
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, 6, 3, 64, 256, 64, dtype=dtype)
    dims = dims_for(B, shape)
    W = shape.kv_width
    n_src, n = 500, 333
    g = synth.rng(11, synth.P_NOISE)
    ks = synth.test_tensor((n_src, W), 12, dtype=dtype)
    vs = synth.test_tensor((n_src, W), 13, dtype=dtype)
    src_row = g.integers(0, n_src, n).astype(np.int32)
    delta = g.integers(-5000, 16383, n).astype(np.int32)
    delta[:3] = [0, 16383, -16383]
    tab = rope_tab(B, 16384, shape.head_dim, shape.rope_base)
    kd = torch.empty(n, W, dtype=tdt(dtype), device="cuda")
    vd = torch.empty_like(kd)
    B.cb_rope_shift(kd, vd, dev(ks, dtype), dev(vs, dtype), dev_i32(src_row), dev_i32(delta), n, dims, tab, 16384)
    B.cb_sync(None)
    want = O.rope_shift(ks[src_row].reshape(n, 3, 64), delta, shape.rope_base).reshape(n, W)
    assert rel(host(kd), want) < (2e-6 if dtype == "f32" else 4e-3)
    np.testing.assert_array_equal(host(vd), vs[src_row])


def test_rope_shift_in_place_keys_only(B):
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, 2, 2, 128, 256, 64, dtype="bf16")
    dims = dims_for(B, shape)
    k0 = synth.test_tensor((640, 256), 14, dtype="bf16")
    k = dev(k0, "bf16")
    delta = np.full(640, 1280, np.int32)
    tab = rope_tab(B, 4096, 128, 1e4)
    B.cb_rope_shift(k, None, k, None, None, dev_i32(delta), 640, dims, tab, 4096)
    B.cb_sync(None)
    want = O.rope_shift(k0.reshape(640, 2, 128), 1280, 1e4).reshape(640, 256)
    assert rel(host(k), want) < 4e-3


# ------------------------------------------------------------------------------ selection
def _topk_case(g, n, kind):
    if kind == "random":
        s = g.random(n).astype(np.float32) * 100
    elif kind == "ties":
        s = g.integers(0, 4, n).astype(np.float32)
    elif kind == "equal":
        s = np.full(n, 2.5, np.float32)
    else:  # zeros of both signs and subnormals among ordinary values
        s = g.random(n).astype(np.float32)
        s[::3] = 0.0
        s[1::7] = -0.0
        s[2::11] = np.float32(1e-40)
    return s


@pytest.mark.parametrize("n", [1, 5, 1000, 3840, 15360, 16391])
@pytest.mark.parametrize("kind", ["random", "ties", "equal", "zeros"])
def test_topk_from_scores_bit_exact(B, n, kind):
    torch = torch_mod()
    g = synth.rng(n + len(kind), synth.P_NOISE)
    s = _topk_case(g, n, kind)
    cand = np.sort(g.choice(4 * n, size=n, replace=False)).astype(np.int32)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    sel = torch.empty(n, dtype=torch.int32, device="cuda")
    for k in sorted({0, 1, n // 7, n // 2, max(n - 1, 0), n}):
        for use_cand in (False, True):
            B.cb_topk_from_scores(dev(s), dev_i32(cand) if use_cand else None, n, k, sel, ws)
            B.cb_sync(None)
            got = sel[:k].cpu().numpy()
            want = O.topk_rows(s, cand if use_cand else np.arange(n), k)
            np.testing.assert_array_equal(got, want)


def test_topk_flags_nonfinite(B):
    torch = torch_mod()
    s = np.ones(100, np.float32)
    s[17] = np.nan
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    sel = torch.empty(100, dtype=torch.int32, device="cuda")
    B.cb_topk_from_scores(dev(s), None, 100, 10, sel, ws)
    with pytest.raises(B.CBError) as e:
        B.cb_sync(None)
    assert e.value.status == 5
    B.cb_sync(None)      # the error word was cleared


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dev_mode", [0, 1])
def test_kv_deviation_topk(B, dtype, dev_mode):
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, 8, 2, 128, 256, 64, dtype=dtype)
    dims = dims_for(B, shape)
    W = shape.kv_width
    n_ref, n_new, n_cand, k = 3000, 2000, 1500, 225
    g = synth.rng(21, synth.P_NOISE)
    kr = synth.test_tensor((n_ref, W), 22, dtype=dtype)
    vr = synth.test_tensor((n_ref, W), 23, dtype=dtype)
    kn = synth.test_tensor((n_new, W), 24, dtype=dtype)
    vn = synth.test_tensor((n_new, W), 25, dtype=dtype)
    new_row = np.sort(g.choice(n_new, n_cand, replace=False)).astype(np.int32)
    ref_row = np.sort(g.choice(n_ref, n_cand, replace=False)).astype(np.int32)
    scores = torch.empty(n_cand, dtype=torch.float32, device="cuda")
    sel = torch.empty(k, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    B.cb_kv_deviation_topk(dev(kn, dtype), dev(vn, dtype), dev(kr, dtype), dev(vr, dtype), dev_i32(new_row),
                           dev_i32(ref_row), n_cand, k, dev_mode, dims, scores, sel, ws)
    B.cb_sync(None)
    if dev_mode == 0:
        want = O.kv_deviation(kn[new_row], kr[ref_row], vn[new_row], vr[ref_row])
    else:
        want = O.kv_deviation(kn[new_row], kr[ref_row])
    got = host(scores)
    assert np.max(np.abs(got - want) / want) < 1e-5
    # the selection is a valid top-k of the exact scores up to fp32 rounding of the sums
    chosen = sel.cpu().numpy()
    assert np.all(np.diff(chosen) > 0) and np.all(np.isin(chosen, ref_row))
    mask = np.isin(ref_row, chosen)
    assert mask.sum() == k
    assert want[mask].min() >= want[~mask].max() * (1 - 2e-5)
    ref_sel = O.topk_rows(want, ref_row, k)
    srt = np.sort(want)[::-1]
    if (srt[k - 1] - srt[k]) / srt[k - 1] > 2e-5:
        np.testing.assert_array_equal(chosen, ref_sel)


# ------------------------------------------------------------------------------ row copies
@pytest.mark.parametrize("row_bytes", [4 * 37, 16 * 64])
def test_gather_scatter_bitwise(B, row_bytes):
    torch = torch_mod()
    g = synth.rng(31, synth.P_NOISE)
    n_src, n = 700, 450
    src = g.integers(0, 2**31, (n_src, row_bytes // 4)).astype(np.int32)
    idx = g.integers(0, n_src, n).astype(np.int32)
    dst = torch.empty(n, row_bytes // 4, dtype=torch.int32, device="cuda")
    B.cb_gather_rows(dst, dev_i32(src), dev_i32(idx), n, row_bytes)
    B.cb_sync(None)
    np.testing.assert_array_equal(dst.cpu().numpy(), src[idx])
    # scatter of K/V rows (dims fix the row width): bf16 rows of W = 2 * 256
    shape = synth.ModelShape(1, 256, 2, 2, 128, 256, 64, dtype="bf16")
    dims = dims_for(B, shape)
    cache = synth.test_tensor((800, 256), 32, dtype="bf16")
    rows = synth.test_tensor((300, 256), 33, dtype="bf16")
    dst_idx = np.sort(g.choice(800, 300, replace=False)).astype(np.int32)
    src_idx = g.permutation(300).astype(np.int32)
    kc, vc = dev(cache, "bf16"), dev(cache, "bf16")
    B.cb_scatter_kv(kc, vc, dev(rows, "bf16"), dev(rows, "bf16"), dev_i32(dst_idx), dev_i32(src_idx), 300, dims)
    B.cb_sync(None)
    want = cache.copy()
    want[dst_idx] = rows[src_idx]
    np.testing.assert_array_equal(host(kc), want)
    np.testing.assert_array_equal(host(vc), want)


# ------------------------------------------------------------------------------ 8-bit chunk KV
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,W", [(1, 8), (5, 100), (640, 4096), (333, 264)])
def test_kv_quantize_codes_bit_exact(B, dtype, n, W):
    """Codes, scales and zeros equal the oracle's bit for bit (both decide in IEEE fp32)."""
    torch = torch_mod()
    x = synth.test_tensor((n, W), 70 + n, std=0.7, dtype=dtype)
    x[:, W // 2] = x[0, W // 2]                     # a constant channel
    codes = torch.empty(n, W, dtype=torch.uint8, device="cuda")
    sc = torch.empty(W, dtype=torch.float32, device="cuda")
    zp = torch.empty(W, dtype=torch.float32, device="cuda")
    B.cb_kv_quantize(dev(x, dtype), n, W, B.CB_BF16 if dtype == "bf16" else B.CB_F32, codes, sc, zp)
    B.cb_sync(None)
    q, s, z = O.kv_quantize(x)
    np.testing.assert_array_equal(codes.cpu().numpy(), q)
    np.testing.assert_array_equal(sc.cpu().numpy(), s)
    np.testing.assert_array_equal(zp.cpu().numpy(), z)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_shift_q8_decodes_and_rotates(B, dtype):
    """Rows gathered from an 8-bit store of three chunks, decoded with their chunk's tables
    and re-rotated by positive and negative offsets, against the oracle's decode + RoPE."""
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, 4, 2, 64, 256, 64, dtype=dtype)
    dims = dims_for(B, shape)
    W = shape.kv_width
    lens = [40, 7, 90]
    store = [synth.test_tensor((m, W), 80 + i, std=0.5, dtype=dtype) for i, m in enumerate(lens)]
    qs = [O.kv_quantize(x) for x in store]
    vstore = [synth.test_tensor((m, W), 90 + i, std=0.5, dtype=dtype) for i, m in enumerate(lens)]
    vqs = [O.kv_quantize(x) for x in vstore]
    kq = dev(np.concatenate([q[0] for q in qs]).astype(np.float32), "f32").to(torch.uint8)
    vq = dev(np.concatenate([q[0] for q in vqs]).astype(np.float32), "f32").to(torch.uint8)
    ks, kz = dev(np.stack([q[1] for q in qs]), "f32"), dev(np.stack([q[2] for q in qs]), "f32")
    vs, vz = dev(np.stack([q[1] for q in vqs]), "f32"), dev(np.stack([q[2] for q in vqs]), "f32")
    offs = np.cumsum([0] + lens[:-1])
    g = synth.rng(95, synth.P_NOISE)
    n_rows = 150
    chunk = g.integers(0, 3, n_rows)
    local = np.array([g.integers(0, lens[c]) for c in chunk])
    src = (offs[chunk] + local).astype(np.int32)
    delta = g.integers(-2000, 2000, n_rows).astype(np.int32)
    tab = rope_tab(B, 2048, shape.head_dim, shape.rope_base)
    kd = torch.empty(n_rows, W, dtype=tdt(dtype), device="cuda")
    vd = torch.empty_like(kd)
    B.cb_rope_shift_q8(kd, vd, kq, vq, ks, kz, vs, vz, dev_i32(src), sum(lens), dev_i32(chunk.astype(np.int32)), 3,
                       dev_i32(delta), n_rows, dims, tab, 2048)
    B.cb_sync(None)
    dk = np.concatenate([O.kv_dequantize(*q) for q in qs])[src]
    dv = np.concatenate([O.kv_dequantize(*q) for q in vqs])[src]
    want_k = O.rope_shift(dk.reshape(n_rows, shape.n_kv_heads, shape.head_dim), delta,
                          shape.rope_base).reshape(n_rows, -1)
    if dtype == "f32":
        np.testing.assert_array_equal(host(vd), dv)        # the decode itself is bit-exact
        assert rel(host(kd), want_k) < 1e-6
    else:
        assert rel(host(vd), dv) < 4e-3 and rel(host(kd), want_k) < 4e-3


# ------------------------------------------------------------------------------ GEMM
# ragged M, N and K tails, single-wave and multi-wave tile counts, the 7B layer's shapes; the
# launches cover the 256-, 224- and 192-column tile widths (4096 x 8192 keeps 256, 4096 x 4096
# takes 224, 832 x 12288 takes 192)
@pytest.mark.parametrize("M,N,K", [(1, 16, 64), (7, 256, 72), (127, 272, 4096), (129, 512, 136),
                                   (300, 4096, 1024), (832, 1024, 4096), (1000, 768, 11008),
                                   (832, 4096, 4096), (4096, 4096, 1000), (256, 8192, 4096),
                                   (832, 12288, 4096), (4096, 4096, 11008), (4096, 8192, 512)])
def test_linear_bf16_tensor_cores(B, M, N, K):
    torch = torch_mod()
    x = synth.test_tensor((M, K), 40 + M, dtype="bf16")
    w = synth.test_tensor((N, K), 41 + N, std=0.02, dtype="bf16")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    B.cb_linear(dev(x, "bf16"), dev(w, "bf16"), y, M, N, K, B.CB_BF16)
    B.cb_sync(None)
    want = x.astype(np.float64) @ w.astype(np.float64).T
    assert rel(host(y), want) < 5e-3


@pytest.mark.parametrize("M,N,K", [(1, 4, 3), (65, 100, 129), (300, 688, 256)])
def test_linear_f32(B, M, N, K):
    torch = torch_mod()
    x = synth.test_tensor((M, K), 50, dtype="f32")
    w = synth.test_tensor((N, K), 51, dtype="f32")
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    B.cb_linear(dev(x), dev(w), y, M, N, K, B.CB_F32)
    B.cb_sync(None)
    assert rel(host(y), x.astype(np.float64) @ w.astype(np.float64).T) < 1e-6


# ------------------------------------------------------------------------------ layer pieces
def _layer(shape, seed=0):
    return synth.make_layer_weights(shape, synth.rng(seed, synth.P_WEIGHTS), gains="random")


def _layer_dev(B, shape, layer):
    t = {k: dev(v, shape.dtype) for k, v in layer.items()}
    w = B.cb_layer_w(*(t[k].data_ptr() for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate_up", "w_down")))
    return t, w


@pytest.mark.parametrize("shape,M", [(SHAPE_F32, 1), (SHAPE_F32, 7), (SHAPE_F32, 129), (SHAPE_BF16, 1),
                                     (SHAPE_BF16, 7), (SHAPE_BF16, 129), (SHAPE_BF16_MID, 640)],
                         ids=["f32-1", "f32-7", "f32-129", "bf16-1", "bf16-7", "bf16-129", "bf16_mid-640"])
def test_selective_qkv(B, shape, M):
    torch = torch_mod()
    dims = dims_for(B, shape)
    layer = _layer(shape)
    t, w = _layer_dev(B, shape, layer)
    n_x = max(300, M + 100)
    x = synth.test_tensor((n_x, shape.d_model), 60, dtype=shape.dtype)
    g = synth.rng(61, synth.P_NOISE)
    rows = np.sort(g.choice(n_x, M, replace=False)).astype(np.int32)
    pos = g.integers(0, 9000, M).astype(np.int32)
    tab = rope_tab(B, 9000, shape.head_dim, shape.rope_base)
    q = torch.empty(M, shape.q_width, dtype=tdt(shape.dtype), device="cuda")
    k = torch.empty(M, shape.kv_width, dtype=tdt(shape.dtype), device="cuda")
    v = torch.empty_like(k)
    ws = torch.empty(B.cb_workspace_bytes(dims, n_x, n_x), dtype=torch.uint8, device="cuda")
    B.cb_selective_qkv(dev(x, shape.dtype), dev_i32(rows), dev_i32(pos), M, dims, w, tab, 9000, q, k, v, ws)
    B.cb_sync(None)
    a = O.rmsnorm(x[rows], layer["attn_norm"], shape.rms_eps)
    p = O.project_qkv(layer, a, pos, shape)
    tol = TOL[shape.dtype]
    assert rel(host(q), p["q"].reshape(M, -1)) < tol
    assert rel(host(k), p["k"].reshape(M, -1)) < tol
    assert rel(host(v), p["v"].reshape(M, -1)) < tol


@pytest.mark.parametrize("shape", [SHAPE_F32, SHAPE_BF16], ids=["f32", "bf16_gqa"])
@pytest.mark.parametrize("M", [1, 7, 129])
def test_partial_attention(B, shape, M):
    torch = torch_mod()
    dims = dims_for(B, shape)
    N = 700
    H, Hkv, hd = shape.n_heads, shape.n_kv_heads, shape.head_dim
    g = synth.rng(70 + M, synth.P_NOISE)
    K = synth.test_tensor((N, Hkv * hd), 71, dtype=shape.dtype)
    V = synth.test_tensor((N, Hkv * hd), 72, dtype=shape.dtype)
    q = synth.test_tensor((M, H * hd), 73, std=0.3, dtype=shape.dtype)
    q_pos = np.sort(g.choice(N, M, replace=False)).astype(np.int32)
    q_pos[0] = 0 if M > 1 else q_pos[0]
    q_pos[-1] = N - 1
    out = torch.empty(M, H * hd, dtype=tdt(shape.dtype), device="cuda")
    B.cb_partial_attention(dev(q, shape.dtype), dev_i32(q_pos), M, dev(K, shape.dtype), dev(V, shape.dtype), N,
                           dims, out)
    B.cb_sync(None)
    want = O.attend(q.reshape(M, H, hd), q_pos, K.reshape(N, Hkv, hd), V.reshape(N, Hkv, hd))
    assert rel(host(out), want) < TOL[shape.dtype] / (10 if shape.dtype == "f32" else 2)


@pytest.mark.parametrize("H,Hkv,hd", [(4, 4, 128), (8, 2, 64), (7, 1, 128)])
@pytest.mark.parametrize("M,N,qstd,order", [(1, 1, 0.3, "asc"), (128, 300, 0.3, "asc"), (257, 2100, 3.0, "asc"),
                                            (300, 4096, 1.0, "shuffled"), (129, 129, 8.0, "asc")])
def test_partial_attention_bf16_tensor_cores(B, H, Hkv, hd, M, N, qstd, order):
    """Tile edges (M, N around 128), GQA groups of 1/4/7, softmax ranges wide enough to
    force the lazy rescale of O, and query positions in any order."""
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, H, Hkv, hd, 256, 64, dtype="bf16")
    dims = dims_for(B, shape)
    g = synth.rng(M * 7 + N, synth.P_NOISE)
    K = synth.test_tensor((N, Hkv * hd), 74, dtype="bf16")
    V = synth.test_tensor((N, Hkv * hd), 75, dtype="bf16")
    q = synth.test_tensor((M, H * hd), 76, std=qstd, dtype="bf16")
    q_pos = np.sort(g.choice(N, M, replace=False)).astype(np.int32)
    q_pos[-1] = N - 1
    if order == "shuffled":
        q_pos = g.permutation(q_pos).astype(np.int32)
    out = torch.empty(M, H * hd, dtype=torch.bfloat16, device="cuda")
    B.cb_partial_attention(dev(q, "bf16"), dev_i32(q_pos), M, dev(K, "bf16"), dev(V, "bf16"), N, dims, out)
    B.cb_sync(None)
    want = O.attend(q.reshape(M, H, hd), q_pos, K.reshape(N, Hkv, hd), V.reshape(N, Hkv, hd))
    assert rel(host(out), want) < 5e-3


@pytest.mark.parametrize("H,Hkv,hd,M,N", [(32, 8, 128, 1100, 3000), (40, 40, 64, 1000, 1000),
                                          (32, 32, 128, 4096, 4096), (32, 8, 128, 2200, 2200)])
def test_partial_attention_at_scale(B, H, Hkv, hd, M, N):
    """Grids of several waves over the SMs: dense causal prefill (every row attends) with GQA
    and a ragged last query tile, and selected rows in shuffled order over a longer sequence."""
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, H, Hkv, hd, 256, 64, dtype="bf16")
    dims = dims_for(B, shape)
    g = synth.rng(H + M, synth.P_NOISE)
    K = synth.test_tensor((N, Hkv * hd), 77, dtype="bf16")
    V = synth.test_tensor((N, Hkv * hd), 78, dtype="bf16")
    q = synth.test_tensor((M, H * hd), 79, std=1.0, dtype="bf16")
    q_pos = np.sort(g.choice(N, M, replace=False)).astype(np.int32) if M < N else np.arange(N, dtype=np.int32)
    if M == 1100:
        q_pos = g.permutation(q_pos).astype(np.int32)
    out = torch.empty(M, H * hd, dtype=torch.bfloat16, device="cuda")
    B.cb_partial_attention(dev(q, "bf16"), dev_i32(q_pos), M, dev(K, "bf16"), dev(V, "bf16"), N, dims, out)
    B.cb_sync(None)
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1]]))   # sampled rows of the oracle
    want = O.attend(q.reshape(M, H, hd)[rows], q_pos[rows], K.reshape(N, Hkv, hd), V.reshape(N, Hkv, hd))
    assert rel(host(out)[rows], want) < 5e-3


@pytest.mark.parametrize("shape,M", [(SHAPE_F32, 1), (SHAPE_F32, 130), (SHAPE_BF16, 1), (SHAPE_BF16, 130),
                                     (SHAPE_BF16_MID, 640)], ids=["f32-1", "f32-130", "bf16-1", "bf16-130",
                                                                  "bf16_mid-640"])
@pytest.mark.parametrize("unit_gains", [False, True], ids=["gains", "unit_gains"])
def test_o_proj_ffn(B, shape, M, unit_gains):
    """O-projection + residual, SwiGLU FFN + residual.  With unit FFN-norm gains passed as
    NULL, the bf16 path folds the norm into the GEMMs (the O-projection leaves the rows' sums
    of squares, the gate/up GEMM scales its rows by 1/rms); fp32 normalises with unit gains."""
    torch = torch_mod()
    dims = dims_for(B, shape)
    layer = _layer(shape, seed=3)
    if unit_gains:
        layer = dict(layer, ffn_norm=np.ones(shape.d_model, np.float32))
    t, w = _layer_dev(B, shape, layer)
    if unit_gains:
        w.ffn_norm = None
    attn = synth.test_tensor((M, shape.q_width), 80, dtype=shape.dtype)
    xr = synth.test_tensor((M, shape.d_model), 81, dtype=shape.dtype)
    out = torch.empty(M, shape.d_model, dtype=tdt(shape.dtype), device="cuda")
    ws = torch.empty(B.cb_workspace_bytes(dims, M, M), dtype=torch.uint8, device="cuda")
    B.cb_o_proj_ffn(dev(attn, shape.dtype), dev(xr, shape.dtype), M, dims, w, out, ws)
    B.cb_sync(None)
    want = O.out_ffn(layer, xr, attn, shape)
    assert rel(host(out), want) < TOL[shape.dtype]


@pytest.mark.parametrize("shape,dev_mode", [(SHAPE_BF16, 0), (SHAPE_BF16, 1), (SHAPE_BF16_MID, 0)],
                         ids=["bf16-kv", "bf16-k", "bf16_mid-kv"])
def test_check_layer_deviation_in_kv_gemm_epilogue(B, shape, dev_mode):
    """bf16 check layers take the KV deviation inside the K/V GEMM's epilogue.  The scores
    equal the standalone deviation of the same K/V rows (the selective Q/K/V call runs the
    same GEMM, so its rows are bitwise the layer's) up to fp32 summation order, the set is
    the top-k of those scores plus the forced rows, and the scores match the oracle's
    deviation of the exact K/V within bf16 error."""
    torch = torch_mod()
    dims = dims_for(B, shape)
    layer = _layer(shape, seed=5)
    t, w = _layer_dev(B, shape, layer)
    N, n_cand, k_budget = 700, 600, 90
    x = synth.test_tensor((N, shape.d_model), 90, dtype="bf16")
    kc = synth.test_tensor((N, shape.kv_width), 91, std=0.3, dtype="bf16")
    vc = synth.test_tensor((N, shape.kv_width), 92, std=0.3, dtype="bf16")
    tab = rope_tab(B, N, shape.head_dim, shape.rope_base)
    ws = torch.empty(B.cb_workspace_bytes(dims, N, N), dtype=torch.uint8, device="cuda")
    x_out = torch.empty(N, shape.d_model, dtype=torch.bfloat16, device="cuda")
    s_out = torch.empty(N, dtype=torch.int32, device="cuda")
    scores = torch.empty(N, dtype=torch.float32, device="cuda")
    m = B.cb_blend_layer(dims, w, B.CB_LAYER_CHECK, dev(x, "bf16"), None, N, N, n_cand, dev(kc, "bf16"),
                         dev(vc, "bf16"), tab, N, k_budget, dev_mode, None, x_out, s_out, scores, ws)
    B.cb_sync(None)
    assert m == k_budget + (N - n_cand)
    got = host(scores)[:n_cand].astype(np.float64)

    rows = dev_i32(np.arange(N, dtype=np.int32))
    q = torch.empty(N, shape.q_width, dtype=torch.bfloat16, device="cuda")
    kn = torch.empty(N, shape.kv_width, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    B.cb_selective_qkv(dev(x, "bf16"), rows, rows, N, dims, w, tab, N, q, kn, vn, ws)
    sc2 = torch.empty(n_cand, dtype=torch.float32, device="cuda")
    sel2 = torch.empty(k_budget, dtype=torch.int32, device="cuda")
    B.cb_kv_deviation_topk(kn, vn, dev(kc, "bf16"), dev(vc, "bf16"), None, None, n_cand, k_budget, dev_mode,
                           dims, sc2, sel2, ws)
    B.cb_sync(None)
    want = host(sc2).astype(np.float64)
    assert np.max(np.abs(got - want) / want) < 1e-5

    S = s_out[:m].cpu().numpy()
    np.testing.assert_array_equal(S[k_budget:], np.arange(n_cand, N))
    top = np.sort(np.lexsort((np.arange(n_cand), -got))[:k_budget])
    np.testing.assert_array_equal(S[:k_budget], top)

    a = O.rmsnorm(x, layer["attn_norm"], shape.rms_eps)
    p = O.project_qkv(layer, a, np.arange(N), shape)
    k_ex, v_ex = p["k"].reshape(N, -1)[:n_cand], p["v"].reshape(N, -1)[:n_cand]
    ref = (O.kv_deviation(k_ex, kc[:n_cand], v_ex, vc[:n_cand]) if dev_mode == 0
           else O.kv_deviation(k_ex, kc[:n_cand]))
    assert rel(got, ref) < 2e-2


# d up to 4096 and up to 8192 take the register-resident bf16 kernels, wider rows and fp32
# input the generic one; a row list gathers, a ragged d covers a partial last vector pass.
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("n,d,gather", [(1, 8, False), (5, 1000, True), (300, 4096, False), (77, 4104, True),
                                        (64, 8192, True), (9, 8200, False)])
def test_rmsnorm(B, din, dout, n, d, gather):
    torch = torch_mod()
    n_x = n + 13
    x = synth.test_tensor((n_x, d), 70 + d, std=1.5, dtype=din)
    g = synth.test_tensor((d,), 71 + d, std=0.3, dtype=din) + 1.0
    g = synth.round_bf16(g) if din == "bf16" else g
    rows = (synth.rng(72, synth.P_NOISE).permutation(n_x)[:n] if gather else np.arange(n)).astype(np.int32)
    out = torch.empty((n, d), dtype=tdt(dout), device="cuda")
    code = {"f32": B.CB_F32, "bf16": B.CB_BF16}
    B.cb_rmsnorm(out, dev(x, din), dev_i32(rows) if gather else None, n, d, dev(g, din), 1e-5, code[din],
                 code[dout])
    B.cb_sync(None)
    want = O.rmsnorm(x[rows], g, 1e-5)
    assert rel(host(out), want) < TOL[dout if din == "f32" else "bf16"]
    assert np.max(np.abs(host(out) - want)) < (1e-4 if dout == "f32" and din == "f32" else 3e-2) * np.max(
        np.abs(want))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lmhead_argmax(B, dtype):
    torch = torch_mod()
    shape = synth.ModelShape(1, 512, 4, 4, 128, 512, 5000, dtype=dtype)
    dims = dims_for(B, shape)
    model = {"shape": shape, "final_norm": synth.test_tensor((512,), 90, std=0.2, dtype=dtype) + 1,
             "w_lm": synth.test_tensor((5000, 512), 91, std=0.02, dtype=dtype)}
    model["final_norm"] = synth.round_bf16(model["final_norm"]) if dtype == "bf16" else model["final_norm"]
    h = synth.test_tensor((512,), 92, dtype=dtype)
    logits = torch.empty(5000, dtype=torch.float32, device="cuda")
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    B.cb_lmhead_argmax(dev(h, dtype), dev(model["final_norm"], dtype), dev(model["w_lm"], dtype), dims, logits,
                       tok, ws)
    B.cb_sync(None)
    want_tok, want_logits = O.lm_head_argmax(model, h)
    got = host(logits)
    assert rel(got, want_logits) < 1e-5
    top2 = np.sort(want_logits)[-2:]
    if top2[1] - top2[0] > 1e-4 * abs(top2[1]):
        assert int(tok.item()) == want_tok
    # ties go to the lowest index
    w2 = np.zeros((5000, 512), np.float32)
    w2[[7, 3, 4000]] = 1.0
    B.cb_lmhead_argmax(dev(h, dtype), dev(np.ones(512, np.float32), dtype), dev(w2, dtype), dims, None, tok, ws)
    B.cb_sync(None)
    assert int(tok.item()) == (3 if np.sum(h, dtype=np.float64) > 0 else 0)


def test_full_prefill_f32_matches_oracle(B):
    torch = torch_mod()
    shape = synth.WORKLOADS["tiny_f32"].shape
    dims = dims_for(B, shape)
    model = synth.make_model(shape, seed=0)
    from non_prefix_kv_gb300 import engine as E
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, 416)
    toks = synth.rng(0, synth.P_TOKENS).integers(0, shape.vocab, 200).astype(np.int32)
    k_out = [torch.empty(200, shape.kv_width, device="cuda") for _ in range(2)]
    v_out = [torch.empty(200, shape.kv_width, device="cuda") for _ in range(2)]
    h = torch.empty(shape.d_model, device="cuda")
    x_all = torch.empty(200, shape.d_model, device="cuda")
    eng.full_prefill(dev_i32(toks), k_out, v_out, h, x_all, pos0=17)
    B.cb_sync(None)
    ref = O.full_prefill(model, toks, pos0=17)
    for l in range(2):
        assert rel(host(k_out[l]), ref["K"][l].reshape(200, -1)) < 1e-5
        assert rel(host(v_out[l]), ref["V"][l].reshape(200, -1)) < 1e-5
    assert rel(host(x_all), ref["x"][-1]) < 1e-5
    assert rel(host(h), ref["h_last"]) < 1e-5


# ------------------------------------------------------------------------------ failure paths
def test_bounded_device_wait_expires_and_context_survives(B):
    """A wait that nothing completes gives up after its bound, the error word reports it once,
    and the same context keeps working (no trap, no hang)."""
    torch = torch_mod()
    B.cb_sync(None)
    B.cb_selftest_wait(1000, arrive=False)
    with pytest.raises(B.CBError) as e:
        B.cb_sync(None)
    assert e.value.status == 9 and "bounded wait" in str(e.value)
    B.cb_selftest_wait(1000, arrive=True)
    B.cb_sync(None)                       # completed wait: no error, the word was cleared
    x = torch.ones(64, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    B.cb_linear(x, x, y, 64, 64, 64, B.CB_BF16)
    B.cb_sync(None)
    assert torch.all(y.float() == 64.0)


def test_host_sync_limit_returns_timeout_then_completes(B):
    """cb_sync with a limit shorter than the queued work returns CB_ERR_TIMEOUT without
    cancelling anything; waiting again completes normally."""
    torch = torch_mod()
    n = 8192
    x = torch.full((n, n), 0.01, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(8):
            B.cb_linear(x, x, y, n, n, n, B.CB_BF16, stream=s)
    with pytest.raises(B.CBError) as e:
        B.cb_sync(s, timeout_s=1e-5)
    assert e.value.status == 7
    B.cb_sync(s, timeout_s=0.0)
    assert abs(float(y[0, 0]) - n * 1e-4) < 0.05 * n * 1e-4


# ------------------------------------------------------------------------------ index checks
def _expect_device_error(B):
    with pytest.raises(B.CBError) as e:
        B.cb_sync(None)
    assert e.value.status == 9 and "out-of-range index" in str(e.value)
    B.cb_sync(None)                       # the word was cleared; the context still works


def test_rope_shift_out_of_range_source_row_is_skipped_and_reported(B):
    """A source row at or past the pool's height is not read: that destination row stays as
    it was, every other row is re-positioned, and cb_sync reports CB_ERR_DEVICE."""
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, 2, 2, 128, 256, 64, dtype="bf16")
    dims = dims_for(B, shape)
    n_src, n = 300, 64
    ks = synth.test_tensor((n_src, 256), 41, dtype="bf16")
    vs = synth.test_tensor((n_src, 256), 42, dtype="bf16")
    src_row = np.arange(n, dtype=np.int32) * 3
    src_row[17] = n_src                   # one past the end
    delta = np.full(n, 640, np.int32)
    tab = rope_tab(B, 4096, 128, 1e4)
    kd = torch.full((n, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    vd = torch.full((n, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    B.cb_rope_shift(kd, vd, dev(ks, "bf16"), dev(vs, "bf16"), dev_i32(src_row), dev_i32(delta), n, dims, tab, 4096)
    _expect_device_error(B)
    ok = np.arange(n) != 17
    want = O.rope_shift(ks[src_row[ok]].reshape(-1, 2, 128), 640, 1e4).reshape(-1, 256)
    assert rel(host(kd)[ok], want) < 4e-3
    np.testing.assert_array_equal(host(vd)[ok], vs[src_row[ok]])
    assert np.all(host(kd)[17] == 7.0) and np.all(host(vd)[17] == 7.0)


def test_embedding_gather_out_of_range_token_is_skipped_and_reported(B):
    """A token id >= vocab is not looked up (the embedding table is bounded by its height)."""
    torch = torch_mod()
    vocab, d, n = 512, 256, 40
    table = synth.test_tensor((vocab, d), 43, dtype="bf16")
    ids = synth.rng(44, synth.P_TOKENS).integers(0, vocab, n).astype(np.int32)
    ids[5], ids[30] = vocab, -1
    out = torch.full((n, d), 3.0, dtype=torch.bfloat16, device="cuda")
    B.cb_gather_rows(out, dev(table, "bf16"), dev_i32(ids), n, d * 2)
    _expect_device_error(B)
    ok = (ids >= 0) & (ids < vocab)
    np.testing.assert_array_equal(host(out)[ok], table[ids[ok]])
    assert np.all(host(out)[~ok] == 3.0)


def test_scatter_out_of_range_cache_row_is_skipped_and_reported(B):
    torch = torch_mod()
    shape = synth.ModelShape(1, 256, 2, 2, 128, 256, 64, dtype="bf16")
    dims = dims_for(B, shape)
    cache = synth.test_tensor((100, 256), 45, dtype="bf16")
    rows = synth.test_tensor((10, 256), 46, dtype="bf16")
    dst_idx = np.arange(10, dtype=np.int32) * 9
    dst_idx[4] = 100                      # past the cache
    kc, vc = dev(cache, "bf16"), dev(cache, "bf16")
    B.cb_scatter_kv(kc, vc, dev(rows, "bf16"), dev(rows, "bf16"), dev_i32(dst_idx), None, 10, dims)
    _expect_device_error(B)
    want = cache.copy()
    ok = dst_idx < 100
    want[dst_idx[ok]] = rows[ok]
    np.testing.assert_array_equal(host(kc), want)
    np.testing.assert_array_equal(host(vc), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rmsnorm_and_deviation_out_of_range_rows_are_reported(B, dtype):
    torch = torch_mod()
    n_x, d = 50, 512
    x = synth.test_tensor((n_x, d), 47, dtype=dtype)
    gain = np.ones(d, np.float32)
    rows = np.array([3, 7, n_x, 1], np.int32)
    out = torch.full((4, d), 5.0, dtype=tdt(dtype), device="cuda")
    code = B.CB_BF16 if dtype == "bf16" else B.CB_F32
    B.cb_rmsnorm(out, dev(x, dtype), dev_i32(rows), 4, d, dev(gain, dtype), 1e-5, code, code)
    _expect_device_error(B)
    assert np.all(host(out)[2] == 5.0)
    want = O.rmsnorm(x[[3, 7, 1]], gain, 1e-5)
    assert rel(host(out)[[0, 1, 3]], want) < (1e-6 if dtype == "f32" else 1e-2)
    # deviation with one cached row past the cache
    shape = synth.ModelShape(1, 256, 2, 2, 128, 256, 64, dtype=dtype)
    dims = dims_for(B, shape)
    kn, vn = (dev(synth.test_tensor((20, 256), s, dtype=dtype), dtype) for s in (48, 49))
    kr, vr = (dev(synth.test_tensor((30, 256), s, dtype=dtype), dtype) for s in (50, 51))
    ref_row = np.arange(20, dtype=np.int32)
    ref_row[11] = 30
    sc = torch.full((20,), -1.0, device="cuda")
    sel = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    B.cb_kv_deviation_topk(kn, vn, kr, vr, None, dev_i32(ref_row), 20, 0, B.CB_DEV_KV, dims, sc, sel, ws)
    _expect_device_error(B)
    s = sc.cpu().numpy()
    assert s[11] == -1.0 and np.all(s[np.arange(20) != 11] > 0)


def test_steady_layer_with_a_row_past_the_cache_writes_nothing_there(B):
    """STEADY takes the caller's row set as the rows whose K/V it writes: a row at or past
    n_tok is not written (the error word reports it), the cache outside stays untouched."""
    torch = torch_mod()
    from non_prefix_kv_gb300 import engine as E
    shape = SHAPE_BF16
    model = synth.make_model(shape, seed=3)
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, 300)
    N = 256
    W = shape.kv_width
    # the caches live inside a larger buffer so that a stray write past row N would show
    big_k = torch.zeros(N + 64, W, dtype=torch.bfloat16, device="cuda")
    big_v = torch.zeros_like(big_k)
    s_in = np.array([10, 50, 100, 255, N + 3], np.int32)
    x = dev(synth.test_tensor((5, shape.d_model), 52, dtype="bf16"), "bf16")
    x_out = torch.empty_like(x)
    s_out = torch.empty(5, dtype=torch.int32, device="cuda")
    B.cb_blend_layer(dm.dims, dm.layers_c[0], B.CB_LAYER_STEADY, x, dev_i32(s_in), 5, N, N - 32, big_k[:N],
                     big_v[:N], eng.cos_sin, eng.max_pos, 0, 0, None, x_out, s_out, None, eng.ws)
    _expect_device_error(B)
    assert torch.count_nonzero(big_k[N:]) == 0 and torch.count_nonzero(big_v[N:]) == 0
    assert torch.count_nonzero(big_k[[10, 50, 100, 255]].float().abs().sum(1)) == 4


# ------------------------------------------------------------------------------ span profiling
def test_span_profiling_records_execution_windows(B):
    """Span mode: every tensor-core GEMM launch records its execution window from the GPU's
    global timer; a kernel without span support reports -1 and no launch gets events.  Launches
    on one stream run one after another (each waits for its predecessor), so their windows add
    up to no more than the event-timed duration of the whole chain."""
    torch = torch_mod()
    M, N, K, d = 832, 4096, 4096, 2048
    x = dev(synth.test_tensor((M, K), 90, dtype="bf16"), "bf16")
    w = dev(synth.test_tensor((N, K), 91, std=0.02, dtype="bf16"), "bf16")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    xn = dev(synth.test_tensor((64, d), 92, dtype="bf16"), "bf16")
    g = dev(synth.round_bf16(synth.test_tensor((d,), 93, std=0.1, dtype="bf16") + 1.0), "bf16")
    out = torch.empty((64, d), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def chain():
        for _ in range(4):
            B.cb_linear(x, w, y, M, N, K, B.CB_BF16, s)
        B.cb_rmsnorm(out, xn, None, 64, d, g, 1e-5, B.CB_BF16, B.CB_BF16, s)

    chain()
    s.synchronize()
    B.cb_profile_begin_spans(16)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    chain()
    e1.record(s)
    recs = B.cb_profile_end(16)
    total_ms = e0.elapsed_time(e1)
    gemm = [r for r in recs if r["kind"] == "gemm"]
    norm = [r for r in recs if r["kind"] == "rmsnorm"]
    assert len(gemm) == 4 and len(norm) == 1
    assert all(r["span_ms"] > 0 for r in gemm), gemm
    assert norm[0]["span_ms"] == -1
    assert all(r["ms"] == -1 for r in recs)
    assert sum(r["span_ms"] for r in gemm) <= total_ms * 1.01 + 0.002, (gemm, total_ms)
    # event mode again afterwards: events, no spans
    B.cb_profile_begin(16)
    chain()
    ev = B.cb_profile_end(16)
    assert len(ev) == 5 and all(r["ms"] > 0 and r["span_ms"] == -1 for r in ev)


def test_span_profiling_serves_one_thread_at_a_time(B):
    """The span slot buffer is the device's: while one host thread is in span mode another
    thread's request is refused, and it succeeds once the first thread has ended."""
    import threading
    out = {}

    def other(tag):
        try:
            B.cb_profile_begin_spans(4)
            out[tag] = "ok"
            B.cb_profile_end(4)
        except RuntimeError as e:
            out[tag] = str(e)

    B.cb_profile_begin_spans(4)
    t = threading.Thread(target=other, args=("while_held",))
    t.start()
    t.join()
    B.cb_profile_end(4)
    t = threading.Thread(target=other, args=("after_end",))
    t.start()
    t.join()
    assert out["while_held"] != "ok" and "another thread" in out["while_held"], out
    assert out["after_end"] == "ok", out
