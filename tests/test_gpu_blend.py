"""End-to-end blended prefill on the GPU against the CPU oracle: chunk precompute, KV
re-positioning, pre-check / check / steady / gradual layers, lm_head.

The HKVD row sets are compared exactly; where the GPU's fp32/bf16 scores order a near-tie
differently from the fp64 oracle (gap below the arithmetic's error), the run is repeated
with the oracle's sets passed in (teacher forcing) and the floats are compared then."""
from dataclasses import replace

import numpy as np
import pytest

import oracle.cacheblend_oracle as O
from non_prefix_kv_gb300 import synth
from tests.gpu_util import TOL, ensure_lib, host, rel, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    torch_mod()
    ensure_lib()
    from non_prefix_kv_gb300 import engine
    return engine


def _near_tie(ref, l, got_set, tol):
    """True when the GPU set differs from the oracle's only among candidates whose oracle
    scores lie within tol (relative) of the k-th largest score."""
    sc, cand = ref["scores"][l], ref["cand"][l]
    k = len(ref["S"][l]) - len(ref["forced"])
    if k == 0 or k == len(cand):
        return False
    kth = np.sort(sc)[::-1][k - 1]
    diff = set(ref["S"][l].tolist()) ^ set(got_set.tolist())
    idx = {int(c): i for i, c in enumerate(cand)}
    return all(abs(sc[idx[r]] - kth) <= tol * kth for r in diff if r in idx)


def _score_gap(ref, l, got_scores):
    """Largest |GPU score - oracle score| over layer l's candidates, and the oracle's largest
    score (the GPU's scores come back in the same candidate order)."""
    sc = np.asarray(ref["scores"][l], dtype=np.float64)
    g = got_scores[:len(sc)].astype(np.float64)
    return float(np.max(np.abs(g - sc))) if len(sc) else 0.0, float(np.max(sc)) if len(sc) else 0.0


def _within_score_gap(ref, l, got_set, delta):
    """True when every row that the GPU set and the oracle's set do not share has an oracle
    score within 2 delta of the oracle's k-th largest score: with the scores perturbed by at
    most delta, an exact top-k can swap only such rows."""
    sc, cand = ref["scores"][l], ref["cand"][l]
    k = len(ref["S"][l]) - len(ref["forced"])
    if k == 0 or k == len(cand):
        return False
    kth = np.sort(sc)[::-1][k - 1]
    diff = set(ref["S"][l].tolist()) ^ set(got_set.tolist())
    idx = {int(c): i for i, c in enumerate(cand)}
    return all(abs(sc[idx[r]] - kth) <= 2.0 * delta * (1 + 1e-6) for r in diff if r in idx)


# bf16 deviation scores against the oracle's, relative to the layer's largest score.  A score
# is a sum of squared differences K_new - K_cached (and V); the differences carry the bf16
# rounding of the rows they come from, about 2^-8 relative, so a large score moves by about
# 2 x 2^-8 of itself.  Measured on GB300: at most 3.2e-3.
BF16_SCORE_TOL = 1e-2


def q8_pool_from_codes(E, pool, chunk_kv, dims):
    """An 8-bit device pool holding the oracle's codes of the oracle's chunk KV, so the GPU
    decodes exactly the values the oracle blends with (the quantizer itself is checked bit
    for bit in the kernel tests)."""
    torch = torch_mod()
    q = E.ChunkPoolQ8.from_pool(pool, dims)
    for c, (off, n) in enumerate(zip(pool.offsets, pool.lens)):
        for l in range(len(pool.k)):
            for key, codes, sc, zp in (("K", q.kq, q.ks, q.kz), ("V", q.vq, q.vs, q.vz)):
                cq, cs, cz = O.kv_quantize(chunk_kv[c][key][l])
                codes[l][off:off + n] = torch.from_numpy(cq).cuda()
                sc[l][c] = torch.from_numpy(cs).cuda()
                zp[l][c] = torch.from_numpy(cz).cuda()
    return q


def with_text_segments(req_h, vocab, seed=11):
    """A system prompt, separators between the chunks and the query: uncached spans spread
    through the request (chunk order as in req_h)."""
    g = synth.rng(seed, synth.P_TOKENS)
    sys_p, sep = g.integers(0, vocab, 7).astype(np.int32), g.integers(0, vocab, 2).astype(np.int32)
    q = g.integers(0, vocab, 20).astype(np.int32)
    segs = [sys_p]
    for i, c in enumerate(req_h.order):
        segs += ([sep] if i else []) + [int(c)]
    segs.append(q)
    toks = np.concatenate([req_h.chunk_tokens[x] if isinstance(x, int) else x for x in segs]).astype(np.int32)
    return segs, toks


def loaded_source(E, pool, load, tmp_path):
    """Layer-ahead loading of the chunk KV: from pinned host memory ("host") or from a file
    read layer by layer into pinned memory ("file").  The device pool is cleared first (and
    for the file tier the pinned copy too), so every cached value the blend uses must have
    travelled through that tier."""
    hp = E.HostPool(pool)
    for ts in hp.dev:
        for t in ts:
            t.zero_()
    if load == "host":
        return {"host_pool": hp}
    fs = E.FileStore(str(tmp_path / "chunk_store.bin"), hp)
    for ts in hp.host:
        for t in ts:
            t.zero_()
    return {"file_store": fs}


def run_case(E, wl, r, gradual, tol, check_sets=True, q8=False, segments=False, recompute=False, split=None,
             load=None, tmp_path=None):
    torch = torch_mod()
    shape = wl.shape
    model = synth.make_model(shape, seed=wl.seed)
    req_h = synth.make_requests(wl)[0]
    tokens = req_h.tokens
    segs = None
    if segments:
        segs, tokens = with_text_segments(req_h, shape.vocab)
    ratios = O.ratio_schedule(r, shape.n_layers, 1, gradual)
    chunk_kv = O.precompute_chunks(model, req_h.chunk_tokens)
    blend_kv = O.quantize_chunks(chunk_kv) if q8 else chunk_kv
    ref = O.blend(model, blend_kv, req_h.order, tokens, ratios, gradual=gradual, segments=segs)

    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, len(tokens))
    pool = eng.precompute_pool(req_h.chunk_tokens)
    # the chunk precompute itself (KV^pre) against the oracle
    for c, off in enumerate(pool.offsets):
        n = pool.lens[c]
        for l in range(shape.n_layers):
            assert rel(host(pool.k[l][off:off + n]), chunk_kv[c]["K"][l].reshape(n, -1)) < tol
            assert rel(host(pool.v[l][off:off + n]), chunk_kv[c]["V"][l].reshape(n, -1)) < tol
    if q8:
        pool = q8_pool_from_codes(E, pool, chunk_kv, dm.dims)
    req = E.Request(eng, pool, req_h.order, tokens, segments=segs)
    plan = req.plan(ratios, gradual=gradual)
    src = loaded_source(E, pool, load, tmp_path) if load else {}
    m = E.run_blend(req, plan, keep_history=True, recompute_precheck_kv=recompute, precheck_load_rows=split, **src)
    from non_prefix_kv_gb300 import binding as B
    B.cb_sync(None)
    forced_teacher = False
    diverged = False   # a set differed at an earlier layer: later layers see other inputs
    for l in range(shape.n_layers):
        got = req.sel_hist[l].cpu().numpy()
        assert len(got) == len(ref["S"][l]), (l, len(got), len(ref["S"][l]))
        assert np.all(np.diff(got) > 0) and set(ref["forced"].tolist()) <= set(got.tolist())
        if not check_sets and not diverged and ref["scores"][l] is not None:
            # bf16: the layer's scores against the oracle's, and the set against the scores
            delta, smax = _score_gap(ref, l, host(req.score_hist[l]))
            print(f"layer {l}: bf16 deviation scores, max gap {delta / max(smax, 1e-30):.2e} of the largest")
            assert delta <= BF16_SCORE_TOL * smax, (l, delta, smax)
            if not np.array_equal(got, ref["S"][l]):
                assert _within_score_gap(ref, l, got, delta), f"layer {l}: set differs beyond the score gap"
        if not np.array_equal(got, ref["S"][l]):
            a, b = set(got.tolist()), set(ref["S"][l].tolist())
            jacc = len(a & b) / len(a | b)
            print(f"layer {l}: HKVD set Jaccard overlap with the oracle {jacc:.3f}")
            if check_sets:
                assert _near_tie(ref, l, got, 1e-4), f"layer {l} set differs"
            diverged = True
            forced_teacher = True
    if forced_teacher or not check_sets:
        override = {}
        for l, (mode, k) in enumerate(plan):
            if mode in (B.CB_LAYER_CHECK, B.CB_LAYER_GRADUAL) and k > 0:
                T = np.setdiff1d(ref["S"][l], ref["forced"]).astype(np.int32)
                override[l] = torch.from_numpy(T).cuda()
        m = E.run_blend(req, plan, sel_override=override, keep_history=True, recompute_precheck_kv=recompute,
                        precheck_load_rows=split, **src)
        B.cb_sync(None)
        for l in range(shape.n_layers):
            np.testing.assert_array_equal(req.sel_hist[l].cpu().numpy(), ref["S"][l])
            if not check_sets and ref["scores"][l] is not None:
                # teacher-forced: every check and gradual layer sees the oracle's sets
                delta, smax = _score_gap(ref, l, host(req.score_hist[l]))
                print(f"layer {l} (teacher-forced): bf16 deviation scores, max gap "
                      f"{delta / max(smax, 1e-30):.2e} of the largest")
                assert delta <= BF16_SCORE_TOL * smax, (l, delta, smax)
    assert m == len(ref["S"][-1])
    for l in range(shape.n_layers):
        assert rel(host(req.K[l]), ref["K"][l].reshape(req.N, -1)) < tol, l
        assert rel(host(req.V[l]), ref["V"][l].reshape(req.N, -1)) < tol, l
    assert rel(host(req.x_last[:m]), ref["x"][-1]) < tol
    assert rel(host(req.x_last[m - 1]), ref["h_last"]) < tol
    lg = np.sort(ref["logits"])[-2:]
    if lg[1] - lg[0] > 1e-2 * abs(lg[1]):
        assert int(req.token.item()) == ref["token"]
    return req, ref


@pytest.mark.parametrize("r", [0.0, 0.15, 1.0])
def test_blend_tiny_f32(E, r):
    run_case(E, synth.WORKLOADS["tiny_f32"], r, False, TOL["f32"])


@pytest.mark.parametrize("r", [0.1, 0.5])
def test_blend_tiny_f32_gradual_3_layers(E, r):
    wl = synth.WORKLOADS["tiny_f32"]
    wl = replace(wl, shape=replace(wl.shape, n_layers=3))
    run_case(E, wl, r, True, TOL["f32"])


@pytest.mark.parametrize("how", ["all", "split"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_blend_with_precheck_kv_recomputed(E, dtype, how):
    """The pre-check layer computing K/V for every row (or for every row from a split on,
    reading the chunk caches below it) instead of reusing the chunk caches (they agree
    there up to rounding) matches the oracle's blend."""
    kw = dict(recompute=True) if how == "all" else {}
    if dtype == "f32":
        wl = synth.WORKLOADS["tiny_f32"]
        wl = replace(wl, shape=replace(wl.shape, n_layers=3))
        run_case(E, wl, 0.15, False, TOL["f32"], split=None if how == "all" else 200, **kw)
    else:
        wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                            ratio=0.15)
        run_case(E, wl, 0.15, True, TOL["bf16"], check_sets=False, split=None if how == "all" else 160, **kw)


@pytest.mark.parametrize("r", [0.0, 0.15])
def test_blend_tiny_f32_from_8bit_chunk_store(E, r):
    """The chunk store kept as 8-bit per-channel codes, decoded while re-positioning: the
    blend matches the oracle's blend over the decoded store."""
    run_case(E, synth.WORKLOADS["tiny_f32"], r, False, TOL["f32"], q8=True)


@pytest.mark.parametrize("r,gradual", [(0.15, False), (0.3, True), (1.0, False)])
def test_blend_with_uncached_spans_f32(E, r, gradual):
    """System prompt, separators and query as uncached spans between the chunks (a forced-row
    mask): sets, blended K/V and outputs against the oracle's segment blend."""
    wl = synth.WORKLOADS["tiny_f32"]
    wl = replace(wl, shape=replace(wl.shape, n_layers=3))
    run_case(E, wl, r, gradual, TOL["f32"], segments=True)


def test_blend_with_uncached_spans_bf16(E):
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15)
    run_case(E, wl, 0.15, True, TOL["bf16"], check_sets=False, segments=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefix_caching_baseline_equals_full_prefill(E, dtype):
    """The comparison workload that reuses only a true prefix (the first chunk) and
    recomputes everything after it at every layer reproduces the full prefill."""
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    if dtype == "f32":
        wl, tol = replace(synth.WORKLOADS["tiny_f32"], shape=replace(synth.WORKLOADS["tiny_f32"].shape, n_layers=3)), \
            TOL["f32"]
    else:
        wl, tol = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3),
                                 n_query=32, ratio=0.15), TOL["bf16"]
    shape = wl.shape
    model = synth.make_model(shape, seed=wl.seed)
    req_h = synth.make_requests(wl)[0]
    first = req_h.order[0]
    n0 = len(req_h.chunk_tokens[first])
    full = O.full_prefill(model, req_h.tokens, 0)
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, len(req_h.tokens))
    pool = eng.precompute_pool(req_h.chunk_tokens)
    req = E.Request(eng, pool, None, req_h.tokens, segments=[int(first), req_h.tokens[n0:]])
    m = E.run_blend(req, req.prefix_cache_plan(), keep_history=True)
    B.cb_sync(None)
    assert m == len(req_h.tokens) - n0
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(req.sel_hist[l].cpu().numpy(), np.arange(n0, len(req_h.tokens)))
        assert rel(host(req.K[l]), full["K"][l].reshape(req.N, -1)) < tol
        assert rel(host(req.V[l]), full["V"][l].reshape(req.N, -1)) < tol
    assert rel(host(req.x_last[m - 1]), full["x"][-1][-1]) < tol


def test_blend_ragged_chunks_no_query_f32(E):
    # chunks of odd lengths and no uncached suffix: the only forced row is the last one
    shape = replace(synth.WORKLOADS["tiny_f32"].shape, n_layers=3)
    wl = synth.Workload("ragged", shape, chunk_len=77, n_distinct=3, order=(2, 0, 1, 0), n_query=0, ratio=0.2)
    run_case(E, wl, 0.2, False, TOL["f32"])


BF16_SMALL = synth.ModelShape(n_layers=3, d_model=512, n_heads=4, n_kv_heads=4, head_dim=128, d_ff=1024,
                              vocab=2048, dtype="bf16", w_std=0.03)


@pytest.mark.parametrize("gradual", [False, True])
def test_blend_bf16_small(E, gradual):
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15)
    run_case(E, wl, 0.15, gradual, TOL["bf16"], check_sets=False)


def test_blend_bf16_gqa(E):
    shape = replace(BF16_SMALL, n_heads=8, n_kv_heads=2, head_dim=64)
    wl = synth.Workload("bf16_gqa", shape, chunk_len=160, n_distinct=3, order=(0, 1, 2, 1), n_query=48,
                        ratio=0.2)
    run_case(E, wl, 0.2, True, TOL["bf16"], check_sets=False)


@pytest.mark.parametrize("q8,from_file,recompute", [(False, False, False), (True, False, False), (False, True, False),
                                                     (True, True, False), (False, False, True), (False, True, True),
                                                     (False, False, 160), (False, True, 200), (True, False, 160),
                                                     (True, True, 200)],
                         ids=["bf16_pool", "8bit_pool", "bf16_file", "8bit_file", "bf16_pool_recompute",
                              "bf16_file_recompute", "bf16_pool_split", "bf16_file_split", "8bit_pool_split",
                              "8bit_file_split"])
def test_layer_ahead_loading_matches_resident_pool(E, q8, from_file, recompute, tmp_path):
    """Loading every layer's chunk KV (bf16, or 8-bit codes with their tables) from pinned
    host memory on a side stream, one event per layer, or from a file read layer by layer
    by a loader thread, gives bit-identical results to the device-resident pool; so does
    loading only the first rows of the pre-check layer (an int: the split) and recomputing
    the rest."""
    split = None if isinstance(recompute, bool) else recompute
    recompute = recompute is True
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15)
    model = synth.make_model(wl.shape, seed=1)
    req_h = synth.make_requests(wl)[0]
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, wl.n_tokens)
    pool = eng.precompute_pool(req_h.chunk_tokens)
    if q8:
        pool = E.ChunkPoolQ8.from_pool(pool, dm.dims)
    hp = E.HostPool(pool)
    plan = E.layer_plan(wl.shape, wl.n_tokens, wl.n_cached, [None, 0.15, 0.15])
    a = E.Request(eng, pool, req_h.order, req_h.tokens)
    E.run_blend(a, plan, recompute_precheck_kv=recompute, precheck_load_rows=split)
    B.cb_sync(None)
    ka = [t.clone() for t in a.K]
    xa = a.x_last[:a.m_last].clone()
    ta = int(a.token.item())
    for ts in hp.dev:                # the streamed run must reload the whole pool
        for t in ts:
            t.zero_()
    if from_file:
        fs = E.FileStore(str(tmp_path / "chunk_store.bin"), hp)
        for ts in hp.host:           # the pinned tier must be refilled from the file
            for t in ts:
                t.zero_()
    b = E.Request(eng, pool, req_h.order, req_h.tokens)
    if from_file:
        E.run_blend(b, plan, file_store=fs, recompute_precheck_kv=recompute, precheck_load_rows=split)
    else:
        E.run_blend(b, plan, host_pool=hp, recompute_precheck_kv=recompute, precheck_load_rows=split)
    B.cb_sync(None)
    for l in range(wl.shape.n_layers):
        assert torch.equal(ka[l], b.K[l])
    assert torch.equal(xa, b.x_last[:b.m_last]) and ta == int(b.token.item())


@pytest.mark.parametrize("load,q8,gradual,extra", [
    ("host", False, False, {}), ("file", False, True, {}), ("host", True, False, {}), ("file", True, False, {}),
    ("host", False, False, {"split": 200}), ("file", False, False, {"recompute": True})],
    ids=["host", "file_gradual", "host_8bit", "file_8bit", "host_split", "file_precheck_recomputed"])
def test_blend_loaded_layer_by_layer_matches_oracle_f32(E, load, q8, gradual, extra, tmp_path):
    """The pages' pipeline (CacheBlend explainer §Pipelining and load controller): each layer's
    chunk KV is loaded one layer ahead, from pinned host memory or from a file, while the
    previous layer recomputes.  The blend built from the loaded KV (bf16/fp32, or 8-bit codes
    decoded while re-positioning) matches the oracle's blend over the same store."""
    wl = synth.WORKLOADS["tiny_f32"]
    wl = replace(wl, shape=replace(wl.shape, n_layers=3))
    run_case(E, wl, 0.15, gradual, TOL["f32"], q8=q8, load=load, tmp_path=tmp_path, **extra)


@pytest.mark.parametrize("load,extra", [("host", {"split": 160}), ("file", {}), ("host", {"q8": True})],
                         ids=["host_split", "file", "host_8bit"])
def test_blend_loaded_layer_by_layer_matches_oracle_bf16(E, load, extra, tmp_path):
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15)
    run_case(E, wl, 0.15, True, TOL["bf16"], check_sets=False, load=load, tmp_path=tmp_path, **extra)


def test_short_request_is_prefilled_in_full(E):
    """Below the blending threshold (256 tokens) the engine runs a full prefill of the
    request: every layer's K/V and the output equal the oracle's full prefill."""
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    wl = replace(synth.WORKLOADS["tiny_f32"], chunk_len=64, n_query=24)
    shape = wl.shape
    model = synth.make_model(shape, seed=wl.seed)
    req_h = synth.make_requests(wl)[0]
    assert len(req_h.tokens) < 256
    full = O.full_prefill(model, req_h.tokens, 0)
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, len(req_h.tokens))
    pool = eng.precompute_pool(req_h.chunk_tokens)
    req = E.Request(eng, pool, req_h.order, req_h.tokens)
    ratios = O.ratio_schedule(0.15, shape.n_layers, 1, False)
    m = E.run_blend(req, req.plan(ratios))
    B.cb_sync(None)
    assert m == req.N
    for l in range(shape.n_layers):
        assert rel(host(req.K[l]), full["K"][l].reshape(req.N, -1)) < TOL["f32"]
    assert rel(host(req.x_last[m - 1]), full["x"][-1][-1]) < TOL["f32"]
    tok, logits = O.lm_head_argmax(model, full["x"][-1][-1])
    top2 = np.sort(logits)[-2:]
    if top2[1] - top2[0] > 1e-2 * abs(top2[1]):
        assert int(req.token.item()) == tok


def test_request_graph_replays_match_eager_runs(E):
    """A request captured once (token upload, layer-ahead loading from pinned host memory,
    layers, read-back) and replayed gives bit-identical results to eager runs, also after
    the host swaps in another query."""
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15)
    model = synth.make_model(wl.shape, seed=1)
    req_h = synth.make_requests(wl)[0]
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, wl.n_tokens)
    pool = eng.precompute_pool(req_h.chunk_tokens)
    plan = E.layer_plan(wl.shape, wl.n_tokens, wl.n_cached, [None, 0.15, 0.15])
    toks2 = req_h.tokens.copy()
    toks2[-wl.n_query:] = synth.rng(99, synth.P_TOKENS).integers(0, wl.shape.vocab, wl.n_query)
    eager = []
    for t in (req_h.tokens, toks2):
        a = E.Request(eng, pool, req_h.order, t)
        E.run_blend(a, plan)
        B.cb_sync(None)
        eager.append(([k.clone() for k in a.K], a.x_last[:a.m_last].clone(), int(a.token.item())))
    hp = E.HostPool(pool)
    b = E.Request(eng, pool, req_h.order, req_h.tokens)
    rg = E.RequestGraph(b, plan, host_pool=hp)
    for t, (ks, xs, tok) in zip((req_h.tokens, toks2), eager):
        assert rg.run(t) == tok
        for l in range(wl.shape.n_layers):
            assert torch.equal(ks[l], b.K[l])
        assert torch.equal(xs, b.x_last[:b.m_last])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_batched_steady_layers_match_per_request_blends(E, dtype):
    """Three requests over one chunk pool (chunk orders shuffled per request, as in the Yi
    workload's batch): the pre-check and check layers per request, then every steady layer
    once for all requests' selected rows.  Sets, every layer's blended K/V, the last layer's
    rows and the first token match the requests blended one at a time."""
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    if dtype == "f32":
        shape = replace(synth.WORKLOADS["tiny_f32"].shape, n_layers=4)
        tol = TOL["f32"]
    else:
        shape = replace(BF16_SMALL, n_layers=4, n_heads=8, n_kv_heads=2, head_dim=64)
        tol = 1e-3
    wl = synth.Workload("batch", shape, chunk_len=96, n_distinct=6, order=(0, 1, 2), n_query=40, ratio=0.15,
                        n_requests=3)
    model = synth.make_model(shape, seed=5)
    reqs_h = synth.make_requests(wl)
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, wl.n_tokens)
    pool = eng.precompute_pool(reqs_h[0].chunk_tokens)
    ratios = O.ratio_schedule(wl.ratio, shape.n_layers, 1, False)
    plan = E.layer_plan(shape, wl.n_tokens, wl.n_cached, ratios)
    single = []
    for rh in reqs_h:
        a = E.Request(eng, pool, rh.order, rh.tokens)
        # the batch normalises with the norm pass; so do these references
        E.run_blend(a, plan, keep_history=True, fold_norms=False)
        B.cb_sync(None)
        single.append(a)
    batch = E.RequestBatch(eng, pool, [rh.order for rh in reqs_h], [rh.tokens for rh in reqs_h])
    ms = E.run_blend_batch(batch, plan)
    B.cb_sync(None)
    for r, (a, b) in enumerate(zip(single, batch.reqs)):
        assert ms[r] == a.m_last
        np.testing.assert_array_equal(batch.S[sum(ms[:r]):sum(ms[:r + 1])].cpu().numpy(),
                                      a.sel_hist[1].cpu().numpy())
        for l in range(shape.n_layers):
            assert rel(host(b.K[l]), host(a.K[l])) <= tol and rel(host(b.V[l]), host(a.V[l])) <= tol, (r, l)
        assert rel(host(b.x_last[:ms[r]]), host(a.x_last[:a.m_last])) <= tol
        assert int(b.token.item()) == int(a.token.item())


def test_precheck_reads_embedding_rows_in_place(E):
    """The pre-check layer given the embedding table and the token ids as its input rows gives
    the same K/V and output rows, bit for bit, as the layer given the gathered rows; a token
    id past the vocabulary is reported (CB_ERR_DEVICE), not followed."""
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15)
    model = synth.make_model(wl.shape, seed=2)
    req_h = synth.make_requests(wl)[0]
    dm = E.DeviceModel.from_host(model)
    eng = E.BlendEngine(dm, wl.n_tokens)
    pool = eng.precompute_pool(req_h.chunk_tokens)
    req = E.Request(eng, pool, req_h.order, req_h.tokens)
    N, d, W = wl.n_tokens, wl.shape.d_model, wl.shape.kv_width
    outs = []
    for in_place in (False, True):
        K = torch.zeros(N, W, dtype=torch.bfloat16, device="cuda")
        V = torch.zeros_like(K)
        B.cb_rope_shift(K[:req.n_cached], V[:req.n_cached], pool.k[0], pool.v[0], req.src_row, req.delta,
                        req.n_cached, dm.dims, eng.cos_sin, eng.max_pos)
        x1 = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
        s1 = torch.empty(N, dtype=torch.int32, device="cuda")
        if in_place:
            B.cb_blend_layer(dm.dims, dm.layers_c[0], B.CB_LAYER_PRECHECK, dm.embed, None, N, N, req.n_cached, K, V,
                             eng.cos_sin, eng.max_pos, 0, 0, None, x1, s1, None, eng.ws, x_rows=req.tokens,
                             n_x_rows=wl.shape.vocab)
        else:
            x0 = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
            B.cb_gather_rows(x0, dm.embed, req.tokens, N, d * 2)
            B.cb_blend_layer(dm.dims, dm.layers_c[0], B.CB_LAYER_PRECHECK, x0, None, N, N, req.n_cached, K, V,
                             eng.cos_sin, eng.max_pos, 0, 0, None, x1, s1, None, eng.ws)
        B.cb_sync(None)
        outs.append((K, V, x1))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    bad = req.tokens.clone()
    bad[7] = wl.shape.vocab
    x1 = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    s1 = torch.empty(N, dtype=torch.int32, device="cuda")
    B.cb_blend_layer(dm.dims, dm.layers_c[0], B.CB_LAYER_PRECHECK, dm.embed, None, N, N, req.n_cached,
                     outs[1][0].clone(), outs[1][1].clone(), eng.cos_sin, eng.max_pos, 0, 0, None, x1, s1, None,
                     eng.ws, x_rows=bad, n_x_rows=wl.shape.vocab)
    with pytest.raises(B.CBError) as e:
        B.cb_sync(None)
    assert e.value.status == 9
    B.cb_sync(None)


def test_shutdown_then_fresh_calls_and_concurrent_host_threads(E):
    """cb_shutdown between two blends leaves the library usable: the second blend (which
    rebuilds every per-device cache) gives bit-identical results.  Two host threads then blend
    two requests at once on their own streams and engines (the per-device caches are shared
    and guarded): each result equals its request's blend run alone."""
    import threading
    torch = torch_mod()
    from non_prefix_kv_gb300 import binding as B
    wl = synth.Workload("bf16_small", BF16_SMALL, chunk_len=96, n_distinct=4, order=(0, 1, 2, 3), n_query=32,
                        ratio=0.15, n_requests=2)
    model = synth.make_model(wl.shape, seed=4)
    reqs_h = synth.make_requests(wl)
    dm = E.DeviceModel.from_host(model)
    plan = E.layer_plan(wl.shape, wl.n_tokens, wl.n_cached, [None, 0.15, 0.15])
    engines = [E.BlendEngine(dm, wl.n_tokens) for _ in range(2)]
    pool = engines[0].precompute_pool(reqs_h[0].chunk_tokens)
    alone = []
    for i, rh in enumerate(reqs_h):
        a = E.Request(engines[i], pool, rh.order, rh.tokens)
        E.run_blend(a, plan)
        B.cb_sync(None)
        alone.append(([k.clone() for k in a.K], a.x_last[:a.m_last].clone(), int(a.token.item())))
    B.cb_shutdown()
    again = E.Request(engines[0], pool, reqs_h[0].order, reqs_h[0].tokens)
    E.run_blend(again, plan)
    B.cb_sync(None)
    assert all(torch.equal(x, y) for x, y in zip(alone[0][0], again.K))
    assert torch.equal(alone[0][1], again.x_last[:again.m_last])
    B.cb_shutdown()
    streams = [torch.cuda.Stream() for _ in range(2)]
    reqs = [E.Request(engines[i], pool, rh.order, rh.tokens) for i, rh in enumerate(reqs_h)]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            with torch.cuda.stream(streams[i]):
                for _ in range(3):
                    E.run_blend(reqs[i], plan, stream=streams[i])
            streams[i].synchronize()
        except BaseException as e:   # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    B.cb_sync(None)
    for i in range(2):
        assert all(torch.equal(x, y) for x, y in zip(alone[i][0], reqs[i].K))
        assert torch.equal(alone[i][1], reqs[i].x_last[:reqs[i].m_last])
        assert alone[i][2] == int(reqs[i].token.item())
