"""Parity at the benchmark's full size: the 7B-shaped three-layer shared-weight stack over
4096 tokens (6 chunks x 640 + 256 query, r = 15 %), run by the same engine calls the
benchmark replays.  The oracle cannot run the whole blend at this size in seconds, so the
checks are (a) outputs it can compute one piece at a time and (b) properties that hold at
any size."""
import dataclasses

import numpy as np
import pytest

import oracle.cacheblend_oracle as O
from non_prefix_kv_gb300 import synth
from tests.gpu_util import ensure_lib, host, rel, torch_mod

pytestmark = pytest.mark.gpu


def _within(name, err, tol):
    """Asserts err < tol and prints the measured margin (shown with pytest -s)."""
    print(f"{name}: relative error {err:.2e} (bound {tol:.0e})")
    assert err < tol, (name, err)


@pytest.fixture(scope="module")
def setup():
    torch = torch_mod()
    ensure_lib()
    from non_prefix_kv_gb300 import binding as B
    from non_prefix_kv_gb300 import engine as E
    wl = synth.WORKLOADS["llama7b_layer_4k"]
    model = synth.make_model(wl.shape, seed=wl.seed)
    req_h = synth.make_requests(wl)[0]
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, wl.n_tokens)
    pool = eng.precompute_pool(req_h.chunk_tokens)
    ratios = O.ratio_schedule(wl.ratio, wl.shape.n_layers, wl.check_layer, wl.gradual)
    plan = E.layer_plan(wl.shape, wl.n_tokens, wl.n_cached, ratios)
    req = E.Request(eng, pool, req_h.order, req_h.tokens)
    E.run_blend(req, plan, keep_history=True)
    B.cb_sync(None)
    one_layer = dict(model, shape=dataclasses.replace(wl.shape, n_layers=1), layers=model["layers"][:1])
    return dict(torch=torch, B=B, E=E, wl=wl, model=model, one_layer=one_layer, req_h=req_h, dm=dm, eng=eng,
                pool=pool, plan=plan, req=req)


def test_chunk_precompute_matches_oracle(setup):
    """KV^pre of the first chunk through all three layers (the layers share weights)."""
    s = setup
    ref = O.full_prefill(s["model"], s["req_h"].chunk_tokens[0], 0)
    n = s["pool"].lens[0]
    for l in range(s["wl"].shape.n_layers):
        assert rel(host(s["pool"].k[l][:n]), ref["K"][l].reshape(n, -1)) < 1e-2
        assert rel(host(s["pool"].v[l][:n]), ref["V"][l].reshape(n, -1)) < 1e-2


def test_repositioned_chunk_keys_match_oracle(setup):
    """The second slot's cached keys are its chunk's local-position keys re-rotated by 640."""
    s = setup
    c = s["req_h"].order[1]
    ref = O.full_prefill(s["one_layer"], s["req_h"].chunk_tokens[c], 0)
    n = s["pool"].lens[c]
    want = O.rope_shift(ref["K"][0], 640, s["wl"].shape.rope_base).reshape(n, -1)
    got = host(s["req"].K[0][640:640 + n])
    assert rel(got, want) < 1e-2
    # values are copied untouched (layer 0 is never recomputed for cached rows)
    off = s["pool"].offsets[c]
    np.testing.assert_array_equal(host(s["req"].V[0][640:640 + n]), host(s["pool"].v[0][off:off + n]))


def test_precheck_layer_prefix_rows_match_oracle(setup):
    """Layer 0 runs every row; rows of the first chunk only see the first chunk, so their
    output equals a one-layer prefill of that chunk alone."""
    s = setup
    torch, B, E = s["torch"], s["B"], s["E"]
    req = s["req"]
    x0 = torch.empty_like(req.x[0])
    B.cb_gather_rows(x0, s["dm"].embed, req.tokens, req.N, s["wl"].shape.d_model * 2)
    x1 = torch.empty_like(req.x[0])
    s_out = torch.empty(req.N, dtype=torch.int32, device="cuda")
    Kc = [t.clone() for t in req.K]
    Vc = [t.clone() for t in req.V]
    m = B.cb_blend_layer(s["dm"].dims, s["dm"].layers_c[0], B.CB_LAYER_PRECHECK, x0, None, req.N, req.N,
                         req.n_cached, Kc[0], Vc[0], s["eng"].cos_sin, s["eng"].max_pos, 0, 0, None, x1, s_out,
                         None, s["eng"].ws)
    B.cb_sync(None)
    assert m == req.N
    ref = O.full_prefill(s["one_layer"], s["req_h"].chunk_tokens[s["req_h"].order[0]], 0)
    rows = [0, 1, 17, 128, 333, 639]
    assert rel(host(x1[rows]), ref["x"][1][rows]) < 1e-2


def test_selection_structure_and_true_prefix(setup):
    s = setup
    req, wl = s["req"], s["wl"]
    N, n_c = wl.n_tokens, wl.n_cached
    k = O.budget(n_c, wl.ratio, n_c)
    assert s["plan"][1][1] == k == 576
    for l in (1, 2):
        S = req.sel_hist[l].cpu().numpy()
        assert len(S) == k + (N - n_c) == 832
        assert np.all(np.diff(S) > 0)
        np.testing.assert_array_equal(S[-(N - n_c):], np.arange(n_c, N))
        # the first chunk is a true prefix: its KV matches the cache up to rounding (the
        # pre-check layer and the chunk precompute may run different attention kernels),
        # so it is never selected
        assert not np.any(S < 640)
    np.testing.assert_array_equal(req.sel_hist[1].cpu().numpy(), req.sel_hist[2].cpu().numpy())
    sc = req.scores[:n_c].cpu().numpy()
    assert np.all(sc[640:] > 0.0)
    assert sc[:640].max() < 1e-3 * np.median(sc[640:])
    # the top-k rows are exactly the k largest of the kernel's own scores, ties to the lower row
    want = np.sort(np.lexsort((np.arange(n_c), -sc.astype(np.float64)))[:k])
    np.testing.assert_array_equal(req.sel_hist[1].cpu().numpy()[:k], want)


def test_zero_ratio_keeps_the_rerotated_cache_bit_exact(setup):
    s = setup
    torch, B, E = s["torch"], s["B"], s["E"]
    req = E.Request(s["eng"], s["pool"], s["req_h"].order, s["req_h"].tokens)
    ratios0 = O.ratio_schedule(0.0, s["wl"].shape.n_layers, 1, False)
    plan0 = E.layer_plan(s["wl"].shape, req.N, req.n_cached, ratios0)
    E.run_blend(req, plan0)
    B.cb_sync(None)
    for l in range(s["wl"].shape.n_layers):
        kd = torch.empty(req.n_cached, s["wl"].shape.kv_width, dtype=torch.bfloat16, device="cuda")
        vd = torch.empty_like(kd)
        B.cb_rope_shift(kd, vd, s["pool"].k[l], s["pool"].v[l], req.src_row, req.delta, req.n_cached,
                        s["dm"].dims, s["eng"].cos_sin, s["eng"].max_pos)
        B.cb_sync(None)
        assert torch.equal(req.K[l][:req.n_cached], kd)
        assert torch.equal(req.V[l][:req.n_cached], vd)


@pytest.mark.parametrize("name", ["llama13b_40_8k", "yi34b_60_16k_b4"])
def test_full_width_layer_of_the_larger_workloads(name):
    """One layer at the 13B and Yi-34B widths (d 5120 / 7168, GQA 56/8 heads, FFN 13824 /
    20480, RoPE base 1e4 / 5e6) over a 640-token chunk, as the chunk precompute runs it:
    K, V and the layer's output rows against the oracle.  The vocabulary is cut to 4096 rows
    (only the embedding lookup sees it)."""
    torch = torch_mod()
    ensure_lib()
    from non_prefix_kv_gb300 import binding as B
    from non_prefix_kv_gb300 import engine as E
    wl = synth.WORKLOADS[name]
    shape = dataclasses.replace(wl.shape, n_layers=1, vocab=4096)
    model = synth.make_model(shape, seed=wl.seed)
    tokens = synth.rng(wl.seed, synth.P_TOKENS).integers(0, shape.vocab, 640).astype(np.int32)
    ref = O.full_prefill(model, tokens, 0)
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, len(tokens))
    dt = E.torch_dtype(shape)
    k = [torch.empty(len(tokens), shape.kv_width, dtype=dt, device="cuda")]
    v = [torch.empty_like(k[0])]
    x_all = torch.empty(len(tokens), shape.d_model, dtype=dt, device="cuda")
    tok = torch.from_numpy(tokens).cuda()
    eng.full_prefill(tok, k, v, None, x_all)
    B.cb_sync(None)
    n = len(tokens)
    assert rel(host(k[0]), ref["K"][0].reshape(n, -1)) < 1e-2
    assert rel(host(v[0]), ref["V"][0].reshape(n, -1)) < 1e-2
    assert rel(host(x_all), ref["x"][1]) < 1e-2


@pytest.fixture(scope="module")
def stepwise(setup):
    """The three layers of the benchmark's request run one call at a time on the GPU, each
    on freshly re-positioned chunk KV, with every layer's input and output kept: the
    pre-check layer over all 4096 rows, the check layer (K/V for every row, deviation, top-k
    576 + 256 forced rows) and the steady layer over the check layer's rows."""
    s = setup
    torch, B, E = s["torch"], s["B"], s["E"]
    req, dm, eng, wl = s["req"], s["dm"], s["eng"], s["wl"]
    N, n_c, W, d = wl.n_tokens, wl.n_cached, wl.shape.kv_width, wl.shape.d_model

    def cache(l):
        k = torch.zeros(N, W, dtype=torch.bfloat16, device="cuda")
        v = torch.zeros_like(k)
        B.cb_rope_shift(k[:n_c], v[:n_c], s["pool"].k[l], s["pool"].v[l], req.src_row, req.delta, n_c, dm.dims,
                        eng.cos_sin, eng.max_pos)
        return k, v

    x0 = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    B.cb_gather_rows(x0, dm.embed, req.tokens, N, d * 2)
    x1, x2, x3 = (torch.empty_like(x0) for _ in range(3))
    s1, s2, s3 = (torch.empty(N, dtype=torch.int32, device="cuda") for _ in range(3))
    K0, V0 = cache(0)
    B.cb_blend_layer(dm.dims, dm.layers_c[0], B.CB_LAYER_PRECHECK, x0, None, N, N, n_c, K0, V0, eng.cos_sin,
                     eng.max_pos, 0, 0, None, x1, s1, None, eng.ws)
    K1, V1 = cache(1)
    K1_pre, V1_pre = K1.clone(), V1.clone()
    scores = torch.empty(N, dtype=torch.float32, device="cuda")
    k = s["plan"][1][1]
    m2 = B.cb_blend_layer(dm.dims, dm.layers_c[1], B.CB_LAYER_CHECK, x1, None, N, N, n_c, K1, V1, eng.cos_sin,
                          eng.max_pos, k, B.CB_DEV_KV, None, x2, s2, scores, eng.ws)
    K2, V2 = cache(2)
    K2_pre, V2_pre = K2.clone(), V2.clone()
    m3 = B.cb_blend_layer(dm.dims, dm.layers_c[2], B.CB_LAYER_STEADY, x2[:m2], s2[:m2], m2, N, n_c, K2, V2,
                          eng.cos_sin, eng.max_pos, 0, 0, None, x3, s3, None, eng.ws)
    B.cb_sync(None)
    S = s2[:m2].cpu().numpy().astype(np.int64)
    return dict(k=k, S=S, m3=m3, x1=host(x1), x2=host(x2[:m2]), x3=host(x3[:m3]), s3=s3[:m3].cpu().numpy(),
                scores=scores[:n_c].cpu().numpy().astype(np.float64), K1_pre=host(K1_pre), V1_pre=host(V1_pre),
                K1=host(K1), V1=host(V1), K2_pre=host(K2_pre), V2_pre=host(V2_pre), K2=host(K2), V2=host(V2))


def _oracle_layer_rows(shape, layer, x_rows, rows, K, V, sample):
    """The oracle's selective recompute of one layer for the given rows (their hidden inputs
    x_rows, positions = rows): K/V of every row written into K, V (Step 3), then Q,
    attention over the whole cache and O-proj + FFN for the rows at `sample` (indices into
    rows).  Returns (K/V rows, the sampled output rows)."""
    a = O.rmsnorm(x_rows, layer["attn_norm"], shape.rms_eps)
    p = O.project_qkv(layer, a, rows, shape, want=("k", "v"))
    K[rows] = p["k"]
    V[rows] = p["v"]
    q = O.project_qkv(layer, a[sample], rows[sample], shape, want=("q",))["q"]
    o = O.attend(q, rows[sample], K, V)
    return p, O.out_ffn(layer, x_rows[sample], o, shape)


def test_check_layer_scores_selection_and_outputs_match_oracle(setup, stepwise):
    """The check layer at the 7B shape ([CB-A] §Selective recomputation Steps 1-4; §HKVD
    selection), the oracle fed the GPU's own layer input x1: the deviation scores of all 3840
    candidates (1e-2 relative), the chosen 576 rows a top-k of the oracle's fp64 scores up to
    the arithmetic's error, then (teacher-forced with the GPU's set) the recomputed K/V at S,
    the layer's output rows (a sample, always with the last row) at 1e-2."""
    s, t = setup, stepwise
    wl = s["wl"]
    shape, layer = wl.shape, s["model"]["layers"][1]
    N, n_c, Hkv, hd = wl.n_tokens, wl.n_cached, shape.n_kv_heads, shape.head_dim
    rows = np.arange(N)
    a = O.rmsnorm(t["x1"], layer["attn_norm"], shape.rms_eps)
    p = O.project_qkv(layer, a, rows, shape, want=("k", "v"))
    Kc = t["K1_pre"].reshape(N, Hkv, hd)
    Vc = t["V1_pre"].reshape(N, Hkv, hd)
    sc = O.kv_deviation(p["k"][:n_c], Kc[:n_c], p["v"][:n_c], Vc[:n_c])
    _within("check layer, deviation scores", rel(t["scores"], sc), 1e-2)
    # the selection: k cached rows + the 256 query rows, ascending
    k, S = t["k"], t["S"]
    T = S[S < n_c]
    assert len(T) == k and np.array_equal(S[k:], np.arange(n_c, N)) and np.all(np.diff(S) > 0)
    kth = np.sort(sc)[::-1][k - 1]
    tol = 2e-2 * kth
    assert sc[T].min() >= kth - tol
    assert np.delete(sc, T).max() <= kth + tol
    jacc = len(set(T) & set(O.topk_rows(sc, np.arange(n_c), k))) / len(set(T) | set(O.topk_rows(sc, np.arange(n_c), k)))
    print(f"check layer: HKVD set Jaccard overlap with the oracle's fp64 top-k {jacc:.3f}")
    # teacher-forced with the GPU's set: K/V at S, then the sampled output rows
    K = Kc.copy()
    V = Vc.copy()
    sample = np.unique(np.concatenate([np.linspace(0, len(S) - 1, 48).astype(int), [len(S) - 1]]))
    pk, y = _oracle_layer_rows(shape, layer, t["x1"][S], S, K, V, sample)
    _within("check layer, K at S", rel(t["K1"][S], pk["k"].reshape(len(S), -1)), 1e-2)
    _within("check layer, V at S", rel(t["V1"][S], pk["v"].reshape(len(S), -1)), 1e-2)
    keep = np.setdiff1d(rows, S)
    np.testing.assert_array_equal(t["K1"][keep], t["K1_pre"][keep])      # rows outside S keep the cache
    _within("check layer, sampled output rows", rel(t["x2"][sample], y), 1e-2)


def test_steady_layer_outputs_and_last_hidden_row_match_oracle(setup, stepwise):
    """The steady layer at the 7B shape (fixed mode: S_2 = S_1, [CB-A] §Selective
    recomputation), the oracle fed the GPU's x2 rows: K/V written at S, the sampled output
    rows and the last hidden row h_last (row N-1, the one the first token comes from) at 1e-2."""
    s, t = setup, stepwise
    wl = s["wl"]
    shape, layer = wl.shape, s["model"]["layers"][2]
    N, Hkv, hd = wl.n_tokens, shape.n_kv_heads, shape.head_dim
    S = t["S"]
    assert t["m3"] == len(S) and np.array_equal(t["s3"], S)
    K = t["K2_pre"].reshape(N, Hkv, hd).copy()
    V = t["V2_pre"].reshape(N, Hkv, hd).copy()
    sample = np.unique(np.concatenate([np.linspace(0, len(S) - 1, 48).astype(int), [len(S) - 1]]))
    pk, y = _oracle_layer_rows(shape, layer, t["x2"], S, K, V, sample)
    _within("steady layer, K at S", rel(t["K2"][S], pk["k"].reshape(len(S), -1)), 1e-2)
    _within("steady layer, V at S", rel(t["V2"][S], pk["v"].reshape(len(S), -1)), 1e-2)
    _within("steady layer, sampled output rows", rel(t["x3"][sample], y), 1e-2)
    _within("steady layer, h_last", rel(t["x3"][-1], y[-1]), 1e-2)
