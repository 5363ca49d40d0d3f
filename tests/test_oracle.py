"""Pins for the CPU oracle: each test checks it against something other than itself
(closed forms, the pages' printed formulas and numbers, brute force, invariants the
method implies).  CPU only."""
import itertools
import math
from dataclasses import replace

import numpy as np
import pytest

import oracle.cacheblend_oracle as O
from non_prefix_kv_gb300 import synth
from tests.conftest import read_golden

MICRO = synth.ModelShape(n_layers=3, d_model=32, n_heads=2, n_kv_heads=2, head_dim=16,
                         d_ff=48, vocab=64, dtype="f32", w_std=0.25)
MICRO_GQA = replace(MICRO, n_heads=4, n_kv_heads=1, head_dim=8)


def micro_setup(shape=MICRO, lens=(5, 9, 7), n_query=4, seed=0, order=None):
    model = synth.make_model(shape, seed=seed, gains="random")
    g = synth.rng(seed, synth.P_TOKENS)
    pool = [g.integers(0, shape.vocab, size=n).astype(np.int32) for n in lens]
    order = list(range(len(lens))) if order is None else order
    q = g.integers(0, shape.vocab, size=n_query).astype(np.int32)
    tokens = np.concatenate([pool[i] for i in order] + [q])
    chunk_kv = O.precompute_chunks(model, pool)
    return model, pool, order, tokens, chunk_kv


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------------------- RoPE
def test_rope_golden_points():
    for row in read_golden("rope_points.txt"):
        base, hd, pos = float(row[0]), int(row[1]), int(row[2])
        x = np.array([float(v) for v in row[3:3 + hd]])
        y = np.array([float(v) for v in row[3 + hd:3 + 2 * hd]])
        got = O.rope_rotate(x[None, :], pos, base)[0]
        np.testing.assert_allclose(got, y, atol=2e-10)


def test_rope_composition_and_orthogonality():
    x = synth.test_tensor((7, 3, 16), seed=1).astype(np.float64)
    for a, b in [(5, 11), (-3, 100), (16000, 383)]:
        two = O.rope_rotate(O.rope_rotate(x, a, 1e4), b, 1e4)
        one = O.rope_rotate(x, a + b, 1e4)
        assert rel(two, one) < 1e-13
    # R(p)^T R(p) = I: norms preserved, inverse by -p
    y = O.rope_rotate(x, 1234, 5e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert rel(O.rope_rotate(y, -1234, 5e6), x) < 1e-13


def test_rope_shift_equals_rotation_from_scratch():
    """Delta-rotating a key precomputed at p' equals rotating the raw key at p = p'+delta
    (Prompt Cache explainer, RoPE position adjustment)."""
    raw = synth.test_tensor((9, 2, 16), seed=2).astype(np.float64)
    p_prime = np.arange(9)
    delta = np.array([0, 1, 7, 640, 3839, 16383, 5, 2, 9000])
    k_pre = O.rope_rotate(raw, p_prime, 1e4)
    got = O.rope_shift(k_pre, delta, 1e4)
    want = O.rope_rotate(raw, p_prime + delta, 1e4)
    assert rel(got, want) < 1e-12


def test_rope_relative_score_closed_form():
    """q_{m+l} . k_m depends on l only; per pair it equals
    (q0 k0 + q1 k1) cos(l theta) + (q0 k1 - q1 k0) sin(l theta).  The CacheBlend page
    prints the symmetric (cos) part; the antisymmetric part vanishes when each q pair is
    parallel to its k pair, which the second check uses."""
    hd, base = 16, 1e4
    q = synth.test_tensor((hd,), seed=3).astype(np.float64)
    k = synth.test_tensor((hd,), seed=4).astype(np.float64)
    th = O.rope_theta(hd, base)
    for l in [0, 1, 5, 77]:
        vals = [O.rope_rotate(q[None], m + l, base)[0] @ O.rope_rotate(k[None], m, base)[0]
                for m in [0, 3, 100, 4000]]
        q0, q1, k0, k1 = q[0::2], q[1::2], k[0::2], k[1::2]
        closed = np.sum((q0 * k0 + q1 * k1) * np.cos(l * th) + (q0 * k1 - q1 * k0) * np.sin(l * th))
        np.testing.assert_allclose(vals, closed, rtol=1e-11, atol=1e-11)
    kp = np.repeat(q[0::2] * 0.5, 2)
    kp[1::2] = q[1::2] * 0.5          # k pair = 0.5 * q pair (parallel)
    page = np.sum((q[0::2] * kp[0::2] + q[1::2] * kp[1::2]) * np.cos(9 * th))
    got = O.rope_rotate(q[None], 12, base)[0] @ O.rope_rotate(kp[None], 3, base)[0]
    assert abs(got - page) < 1e-12


# ---------------------------------------------------------------------------- layer pieces
def test_rmsnorm_closed_form():
    d = 8
    g = np.arange(1, d + 1, dtype=np.float64)
    for c in [1.0, -3.0, 0.001]:
        x = np.full((1, d), c)
        want = c / math.sqrt(c * c + 1e-5) * g
        np.testing.assert_allclose(O.rmsnorm(x, g, 1e-5)[0], want, rtol=1e-14)
    x = synth.test_tensor((3, d), seed=5).astype(np.float64)
    # scale invariance with eps = 0
    np.testing.assert_allclose(O.rmsnorm(7 * x, g, 0.0), O.rmsnorm(x, g, 0.0), rtol=1e-13)


def test_linear_is_x_times_w_transposed():
    w = np.zeros((3, 5))
    w[2, 4] = 1.0          # output 2 reads input 4
    x = np.arange(5.0)[None]
    np.testing.assert_array_equal(O.linear(x, w)[0], [0, 0, 4.0])


def test_silu_special_values():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    z = np.linspace(-6, 6, 13)
    np.testing.assert_allclose(O.silu(-z), O.silu(z) - z, atol=1e-14)
    np.testing.assert_allclose(O.silu(np.array([1.0])), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)


def test_attention_special_cases():
    g = synth.rng(6, synth.P_NOISE)
    K = g.standard_normal((5, 1, 4))
    V = g.standard_normal((5, 1, 4))
    q = g.standard_normal((3, 2, 4))          # 2 query heads share 1 KV head (GQA)
    o = O.attend(q, [0, 2, 4], K, V).reshape(3, 2, 4)
    np.testing.assert_allclose(o[0, 0], V[0, 0], rtol=1e-14)   # one visible key
    np.testing.assert_allclose(o[0, 1], V[0, 0], rtol=1e-14)
    oz = O.attend(np.zeros((1, 2, 4)), [3], K, V).reshape(2, 4)
    np.testing.assert_allclose(oz[0], V[:4, 0].mean(axis=0), rtol=1e-13)


def test_attention_brute_force_masked_softmax():
    from scipy.special import softmax
    g = synth.rng(7, synth.P_NOISE)
    N, H, Hkv, hd = 11, 4, 2, 8
    K = g.standard_normal((N, Hkv, hd))
    V = g.standard_normal((N, Hkv, hd))
    qpos = [0, 3, 4, 10]
    q = g.standard_normal((len(qpos), H, hd))
    o = O.attend(q, qpos, K, V).reshape(len(qpos), H, hd)
    for i, p in enumerate(qpos):
        for h in range(H):
            kv = h // (H // Hkv)
            logits = np.array([q[i, h] @ K[t, kv] / math.sqrt(hd) if t <= p else -np.inf
                               for t in range(N)])
            np.testing.assert_allclose(o[i, h], softmax(logits) @ V[:, kv], rtol=1e-12)


# ---------------------------------------------------------------------------- selection
def test_budget_golden():
    for n, r, k in read_golden("budget_table.txt"):
        assert O.budget(int(n), float(r)) == int(k), (n, r)
    assert O.budget(3840, 0.15, n_candidates=100) == 100


@pytest.mark.parametrize("r", [0.0, 0.05, 0.15, 0.18, 0.5, 0.7, 1.0])
def test_ratio_schedule_follows_gradual_filtering(r):
    """CacheBlend explainer §Gradual filtering fixes the shape of the per-layer ratio: nothing
    before the check layer; the check layer's r1 is at least r (a little above it) and at most
    1; later layers never increase the ratio and approach r; fixed mode keeps r at every layer
    from the check layer on.  The nested selections need the budgets to be non-increasing."""
    L, c = 40, 1
    fixed = O.ratio_schedule(r, L, c, gradual=False)
    assert fixed[:c] == [None] * c and all(x == r for x in fixed[c:])
    grad = O.ratio_schedule(r, L, c, gradual=True)
    assert grad[:c] == [None] * c
    rs = np.array(grad[c:], dtype=np.float64)
    assert r <= rs[0] <= 1.0
    if 0.0 < r < 1.0:
        assert rs[0] > r                       # strictly above r at the check layer
    assert np.all(np.diff(rs) <= 0.0)          # non-increasing
    assert np.all(rs >= r)                     # never below the target
    assert rs[-1] - r < 1e-9 * max(r, 1.0)     # tends to r
    ks = [O.budget(3840, x) for x in rs]
    assert all(a >= b for a, b in zip(ks, ks[1:]))
    assert ks[-1] == O.budget(3840, r)
    # another check layer shifts the schedule without changing its values
    assert O.ratio_schedule(r, L, 3, gradual=True)[3:] == grad[1:L - 2]


def test_lm_head_argmax_hand_built():
    """First-token step on a hand-built case: one-hot lm_head rows, a non-unit final-norm gain,
    closed-form logits and a tie (lowest index wins, R8).  h = (3, -4, 0, 0) has
    mean(h^2) = 25/4, so RMSNorm(h) = h / sqrt(6.25 + eps)."""
    shape = synth.ModelShape(n_layers=1, d_model=4, n_heads=1, n_kv_heads=1, head_dim=4, d_ff=4, vocab=5)
    e = np.eye(4)
    w_lm = np.stack([e[0], e[1], 2.0 * e[2], -e[1], e[0]])   # rows 0 and 4 are the same
    h = np.array([3.0, -4.0, 0.0, 0.0])
    rms = math.sqrt(6.25 + shape.rms_eps)
    for gain, want_tok in (([2.0, 0.5, 1.0, 1.0], 0), ([0.5, 2.0, 1.0, 1.0], 3)):
        model = {"shape": shape, "final_norm": np.array(gain), "w_lm": w_lm}
        tok, logits = O.lm_head_argmax(model, h)
        b0, b1 = 3.0 * gain[0] / rms, -4.0 * gain[1] / rms
        np.testing.assert_allclose(logits, [b0, b1, 0.0, -b1, b0], rtol=1e-14, atol=1e-15)
        assert tok == want_tok
    # every logit equal: the lowest index
    flat = {"shape": shape, "final_norm": np.ones(4), "w_lm": np.zeros((5, 4))}
    assert O.lm_head_argmax(flat, h)[0] == 0


def test_kv_deviation_closed_form():
    g = synth.rng(8, synth.P_NOISE)
    k = g.standard_normal((6, 2, 4))
    v = g.standard_normal((6, 2, 4))
    c = np.arange(6)[:, None, None] * 0.5
    s = O.kv_deviation(k + c, k, v - 2 * c, v)
    np.testing.assert_allclose(s, (0.25 + 1.0) * 8 * np.arange(6) ** 2, rtol=1e-12)
    assert np.all(O.kv_deviation(k, k) == 0)


def _brute_topk(scores, cand, k):
    """Unique subset T of size k such that every member beats every non-member under
    (score desc, row asc)."""
    found = []
    idx = range(len(cand))
    for T in itertools.combinations(idx, k):
        Ts = set(T)
        ok = all((scores[t] > scores[u]) or (scores[t] == scores[u] and cand[t] < cand[u])
                 for t in Ts for u in idx if u not in Ts)
        if ok:
            found.append(sorted(cand[t] for t in T))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(seed):
    g = synth.rng(seed, synth.P_NOISE)
    n = int(g.integers(1, 11))
    scores = g.integers(0, 4, size=n).astype(np.float32)      # many ties
    if seed == 0:
        scores[:] = 1.0                                        # all equal
    cand = np.sort(g.choice(40, size=n, replace=False))        # strict subset of rows
    for k in range(0, n + 1):
        got = O.topk_rows(scores, cand, k).tolist()
        want = _brute_topk(scores, cand, k) if k else []
        assert got == want


def test_topk_rejects_nonfinite():
    with pytest.raises(ValueError):
        O.topk_rows(np.array([1.0, np.nan]), [0, 1], 1)


# ---------------------------------------------------------------------------- prefill invariants
def test_true_prefix_kv_unchanged():
    """The first chunk is a true prefix: its K/V inside the whole-input prefill equal its
    isolated precompute (CacheBlend explainer: prefix caching reuses exactly these)."""
    model, pool, order, tokens, chunk_kv = micro_setup()
    full = O.full_prefill(model, tokens)
    n0 = len(pool[order[0]])
    for l in range(MICRO.n_layers):
        assert rel(full["K"][l][:n0], chunk_kv[order[0]]["K"][l]) < 1e-12
        assert rel(full["V"][l][:n0], chunk_kv[order[0]]["V"][l]) < 1e-12


def test_causality():
    model, pool, order, tokens, _ = micro_setup()
    a = O.full_prefill(model, tokens)
    t2 = tokens.copy()
    j = 10
    t2[j + 1:] = (t2[j + 1:] + 7) % MICRO.vocab
    b = O.full_prefill(model, t2)
    for l in range(MICRO.n_layers + 1):
        np.testing.assert_allclose(a["x"][l][:j + 1], b["x"][l][:j + 1], rtol=1e-12, atol=1e-14)
    assert rel(a["x"][-1][j + 1:], b["x"][-1][j + 1:]) > 1e-3


@pytest.mark.parametrize("shape", [MICRO, MICRO_GQA], ids=["mha", "gqa"])
def test_chunk_prefill_is_shift_equivariant(shape):
    """A chunk prefilled alone at start s has, at every layer, keys equal to its
    position-0 precompute re-rotated by s (RoPE scores depend on relative position
    only), and identical values: the basis of re-positioning cached chunks."""
    model, pool, order, tokens, chunk_kv = micro_setup(shape)
    for s in [1, 13, 999]:
        at_s = O.full_prefill(model, pool[1], pos0=s)
        for l in range(shape.n_layers):
            assert rel(at_s["K"][l], O.rope_shift(chunk_kv[1]["K"][l], s, shape.rope_base)) < 1e-10
            assert rel(at_s["V"][l], chunk_kv[1]["V"][l]) < 1e-10


# ---------------------------------------------------------------------------- blend invariants
@pytest.mark.parametrize("gradual", [False, True])
@pytest.mark.parametrize("shape", [MICRO, MICRO_GQA], ids=["mha", "gqa"])
def test_blend_r1_equals_full_prefill(shape, gradual):
    model, pool, order, tokens, chunk_kv = micro_setup(shape)
    ratios = O.ratio_schedule(1.0, shape.n_layers, 1, gradual)
    b = O.blend(model, chunk_kv, order, tokens, ratios, gradual=gradual)
    full = O.full_prefill(model, tokens)
    for l in range(shape.n_layers):
        assert rel(b["K"][l], full["K"][l]) < 1e-10, l
        assert rel(b["V"][l], full["V"][l]) < 1e-10, l
    assert rel(b["h_last"], full["h_last"]) < 1e-10
    assert b["token"] == O.lm_head_argmax(model, full["h_last"])[0]


def _suffix_prefill_over_past(model, past_K, past_V, suffix_tokens, start):
    """Independent restatement of "full KV reuse": the suffix is prefilled over a fixed
    past KV (the re-rotated concatenation), nothing of the past recomputed."""
    shape = model["shape"]
    H, Hkv, hd, F = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.d_ff
    x = model["embed"][suffix_tokens].astype(np.float64)
    n = len(suffix_tokens)
    pos = start + np.arange(n)
    outK, outV = [], []
    for l, W in enumerate(model["layers"]):
        a = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + shape.rms_eps) * W["attn_norm"]
        qkv = a @ W["wqkv"].astype(np.float64).T
        th = shape.rope_base ** (-np.arange(0, hd, 2) / hd)

        def rot(t, heads):
            t = t.reshape(n, heads, hd // 2, 2)
            c = np.cos(pos[:, None, None] * th)
            s = np.sin(pos[:, None, None] * th)
            return np.stack([t[..., 0] * c - t[..., 1] * s, t[..., 0] * s + t[..., 1] * c], -1).reshape(n, heads, hd)

        q = rot(qkv[:, :H * hd], H)
        k = rot(qkv[:, H * hd:(H + Hkv) * hd], Hkv)
        v = qkv[:, (H + Hkv) * hd:].reshape(n, Hkv, hd)
        Kall = np.concatenate([past_K[l], k])
        Vall = np.concatenate([past_V[l], v])
        o = np.zeros((n, H, hd))
        for i in range(n):
            for h in range(H):
                kv = h * Hkv // H
                sc = Kall[:start + i + 1, kv] @ q[i, h] / math.sqrt(hd)
                w = np.exp(sc - sc.max())
                o[i, h] = (w / w.sum()) @ Vall[:start + i + 1, kv]
        hh = x + o.reshape(n, -1) @ W["wo"].astype(np.float64).T
        b = hh / np.sqrt(np.mean(hh * hh, axis=1, keepdims=True) + shape.rms_eps) * W["ffn_norm"]
        gu = b @ W["w_gate_up"].astype(np.float64).T
        x = hh + ((gu[:, :F] / (1 + np.exp(-gu[:, :F]))) * gu[:, F:]) @ W["w_down"].astype(np.float64).T
        outK.append(k)
        outV.append(v)
    return outK, outV, x


@pytest.mark.parametrize("shape", [MICRO, MICRO_GQA], ids=["mha", "gqa"])
def test_blend_r0_equals_full_kv_reuse(shape):
    model, pool, order, tokens, chunk_kv = micro_setup(shape)
    ratios = O.ratio_schedule(0.0, shape.n_layers, 1, False)
    b = O.blend(model, chunk_kv, order, tokens, ratios)
    n_c = b["n_cached"]
    # cached rows: exactly the re-rotated concatenation, every layer
    start = 0
    for c in order:
        n = len(pool[c])
        for l in range(shape.n_layers):
            want = O.rope_shift(chunk_kv[c]["K"][l], start, shape.rope_base)
            np.testing.assert_array_equal(b["K"][l][start:start + n], want)
            np.testing.assert_array_equal(b["V"][l][start:start + n], chunk_kv[c]["V"][l])
        start += n
    pastK = [b["K"][l][:n_c] for l in range(shape.n_layers)]
    pastV = [b["V"][l][:n_c] for l in range(shape.n_layers)]
    k, v, x = _suffix_prefill_over_past(model, pastK, pastV, tokens[n_c:], n_c)
    for l in range(shape.n_layers):
        assert rel(b["K"][l][n_c:], k[l]) < 1e-12
        assert rel(b["V"][l][n_c:], v[l]) < 1e-12
    assert rel(b["h_last"], x[-1]) < 1e-12
    assert all(len(S) == len(tokens) - n_c for S in b["S"][1:])


def test_layer0_deviation_is_zero_and_first_chunk_unselected():
    model, pool, order, tokens, chunk_kv = micro_setup()
    # deviation measured at layer 0 (embedding input, context-free) is rounding only
    b0 = O.blend(model, chunk_kv, order, tokens, O.ratio_schedule(0.3, 3, 0, False), check_layer=0)
    assert np.max(b0["scores"][0]) < 1e-20
    # at layer 1 the first chunk (a true prefix) still has ~0 deviation; later chunks do not
    b1 = O.blend(model, chunk_kv, order, tokens, O.ratio_schedule(0.3, 3, 1, False))
    sc, cand = b1["scores"][1], b1["cand"][1]
    n0 = len(pool[order[0]])
    first = sc[cand < n0]
    rest = sc[cand >= n0]
    assert np.max(first) < 1e-20 and np.min(rest) > 1e-10
    assert not np.any(b1["S"][1] < n0)


def test_duplicated_chunk_rows_differ_by_rotation():
    model, pool, order, tokens, chunk_kv = micro_setup(order=[0, 1, 0])
    b = O.blend(model, chunk_kv, [0, 1, 0], tokens, O.ratio_schedule(0.0, 3, 1, False))
    n0, n1 = len(pool[0]), len(pool[1])
    s2 = n0 + n1
    for l in range(MICRO.n_layers):
        np.testing.assert_allclose(b["K"][l][s2:s2 + n0],
                                   O.rope_shift(b["K"][l][:n0], s2, MICRO.rope_base), rtol=1e-12, atol=1e-13)
        np.testing.assert_array_equal(b["V"][l][s2:s2 + n0], b["V"][l][:n0])


def test_blend_selection_shapes_and_forced_rows():
    model, pool, order, tokens, chunk_kv = micro_setup()
    N = len(tokens)
    for gradual in [False, True]:
        ratios = O.ratio_schedule(0.3, 3, 1, gradual)
        b = O.blend(model, chunk_kv, order, tokens, ratios, gradual=gradual)
        n_c = b["n_cached"]
        prev = None
        for l in range(1, 3):
            S = b["S"][l]
            assert np.all(np.diff(S) > 0)
            assert set(range(n_c, N)) <= set(S.tolist())
            k = O.budget(n_c, ratios[l], len(b["cand"][l]) if b["cand"][l] is not None else None)
            if b["cand"][l] is not None:
                assert len(S) == k + (N - n_c)
            if gradual and prev is not None:
                assert set(S.tolist()) <= set(prev.tolist())
            # only the rows of S_l were overwritten: every other cached row keeps the
            # re-rotated chunk cache
            start = 0
            keep = np.ones(N, bool)
            keep[S] = False
            for c in order:
                n = len(pool[c])
                want = O.rope_shift(chunk_kv[c]["K"][l], start, MICRO.rope_base)
                rows = np.nonzero(keep[start:start + n])[0]
                np.testing.assert_array_equal(b["K"][l][start + rows], want[rows])
                np.testing.assert_array_equal(b["V"][l][start + rows], chunk_kv[c]["V"][l][rows])
                start += n
            prev = S


def test_cost_pins():
    for row in read_golden("cost_pins.txt"):
        if row[0] == "kv_bytes":
            L, S, H, dh, b, want = map(int, row[1:7])
            assert O.kv_bytes(L, S, H, dh, b) == want
        elif row[0] == "kv_gb_approx":
            L, S, H, dh, b = map(int, row[1:6])
            assert abs(O.kv_bytes(L, S, H, dh, b) / 1e9 - float(row[6])) / float(row[6]) < float(row[7])
        elif row[0] == "t_load_ms":
            per_tok, n, thr, want, tol = float(row[1]), int(row[2]), float(row[3]), float(row[4]), float(row[5])
            assert abs(O.t_load(per_tok, n, thr) * 1e3 - want) / want < tol
    assert O.optimal_ratio(0.15, 0.016, 0.020) == 0.8
    assert O.optimal_ratio(0.15, 0.001, 0.020) == 0.15


# ------------------------------------------------------------------ 8-bit chunk KV
def test_kv_quantize_integer_channels_and_half_to_even():
    """Channel 0 spans 0..255 (scale 1: codes are the values); channel 1 spans 0..510
    (scale 2: odd values land on .5 and round to the even code, as the page's round
    does)."""
    x = np.zeros((6, 2), np.float32)
    x[:, 0] = [0, 1, 2, 7, 128, 255]
    x[:, 1] = [0, 3, 5, 7, 101, 510]
    q, s, z = O.kv_quantize(x)
    assert s.tolist() == [1.0, 2.0] and z.tolist() == [0.0, 0.0]
    assert q[:, 0].tolist() == [0, 1, 2, 7, 128, 255]
    assert q[:, 1].tolist() == [0, 2, 2, 4, 50, 255]     # 1.5->2, 2.5->2, 3.5->4, 50.5->50
    np.testing.assert_array_equal(O.kv_dequantize(q, s, z)[:, 0], x[:, 0])


def test_kv_quantize_range_and_roundtrip_bound():
    g = np.random.default_rng(5)
    x = (g.standard_normal((300, 64)) * g.uniform(0.01, 5.0, 64) + g.uniform(-3, 3, 64)).astype(np.float32)
    q, s, z = O.kv_quantize(x)
    assert q.dtype == np.uint8
    np.testing.assert_array_equal(q[np.argmin(x, axis=0), np.arange(64)], 0)
    np.testing.assert_array_equal(q[np.argmax(x, axis=0), np.arange(64)], 255)
    np.testing.assert_allclose(s, (x.max(0).astype(np.float64) - x.min(0)) / 255, rtol=1e-6)
    err = np.abs(O.kv_dequantize(q, s, z).astype(np.float64) - x)
    assert np.all(err <= s * 0.5 + 4 * np.abs(x) * 2.0 ** -24 + 1e-7)
    # each code is a nearest level of (x - z) / s
    t = (x.astype(np.float64) - z) / s
    assert np.all(np.abs(q - t) <= 0.5 + 1e-4)


def test_kv_quantize_constant_channel():
    x = np.full((5, 3), 1.25, np.float32)
    x[:, 2] = [-1, 0, 1, 2, 3]
    q, s, z = O.kv_quantize(x)
    assert np.all(q[:, :2] == 0) and s[0] == np.float32(1e-8)
    np.testing.assert_array_equal(O.kv_dequantize(q, s, z)[:, :2], x[:, :2])


def test_quantized_chunks_blend_stays_close():
    """The decoded 8-bit chunk store changes each cached K/V entry by at most half a step,
    and a blend over it keeps the selection structure."""
    model, pool, order, tokens, chunk_kv = micro_setup()
    q = O.quantize_chunks(chunk_kv)
    for a, b in zip(chunk_kv, q):
        for key in ("K", "V"):
            for t, u in zip(a[key], b[key]):
                span = t.reshape(len(t), -1).max(0) - t.reshape(len(t), -1).min(0)
                assert np.all(np.abs(u - t).reshape(len(t), -1) <= span / 255 * 0.5 + 1e-6)
    ratios = O.ratio_schedule(0.3, MICRO.n_layers, 1, False)
    ref = O.blend(model, q, order, tokens, ratios)
    assert len(ref["S"][1]) == O.budget(ref["n_cached"], 0.3, ref["n_cached"]) + len(ref["forced"])


# ------------------------------------------------------------------ uncached segments
def test_segments_in_chunk_then_query_order_equal_the_plain_blend():
    model, pool, order, tokens, chunk_kv = micro_setup()
    q = tokens[sum(len(pool[i]) for i in order):]
    ratios = O.ratio_schedule(0.4, MICRO.n_layers, 1, True)
    a = O.blend(model, chunk_kv, order, tokens, ratios, gradual=True)
    b = O.blend(model, chunk_kv, order, tokens, ratios, gradual=True, segments=list(order) + [q])
    for l in range(MICRO.n_layers):
        np.testing.assert_array_equal(a["S"][l], b["S"][l])
        np.testing.assert_array_equal(a["K"][l], b["K"][l])
    np.testing.assert_array_equal(a["h_last"], b["h_last"])


def test_segments_r1_equal_full_prefill_and_text_rows_always_forced():
    """A system prompt, separators between chunks and a query: at r = 1 the blend is the
    full prefill (I1); at any r every uncached row is in every layer's set."""
    model, pool, order, tokens, chunk_kv = micro_setup()
    g = synth.rng(7, synth.P_TOKENS)
    sys_p, sep, q = (g.integers(0, MICRO.vocab, n).astype(np.int32) for n in (3, 1, 4))
    segs = [sys_p, 0, sep, 2, sep, 1, q]
    toks = np.concatenate([s if not isinstance(s, int) else pool[s] for s in segs])
    full = O.full_prefill(model, toks, 0)
    ref = O.blend(model, chunk_kv, None, toks, O.ratio_schedule(1.0, MICRO.n_layers, 1, False), segments=segs)
    for l in range(MICRO.n_layers):
        np.testing.assert_allclose(ref["K"][l], full["K"][l], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(ref["h_last"], full["x"][-1][-1], rtol=1e-9, atol=1e-10)
    ref = O.blend(model, chunk_kv, None, toks, O.ratio_schedule(0.25, MICRO.n_layers, 1, True), gradual=True,
                  segments=segs)
    _, _, cached = O.assemble_segments(model, chunk_kv, segs)
    text_rows = set(np.nonzero(~cached)[0].tolist()) | {len(toks) - 1}
    for S in ref["S"][1:]:
        assert text_rows <= set(S.tolist())
    assert len(ref["S"][1]) == O.budget(int(cached.sum()), O.ratio_schedule(0.25, MICRO.n_layers, 1, True)[1],
                                        int(cached.sum())) + len(text_rows)


def test_prefix_caching_baseline_is_exact():
    """Reusing only a true prefix (the first chunk) and recomputing every later row at every
    layer reproduces the full prefill: the prefix-caching comparison workload."""
    model, pool, order, tokens, chunk_kv = micro_setup()
    rest = tokens[len(pool[order[0]]):]
    full = O.full_prefill(model, tokens, 0)
    ref = O.blend(model, chunk_kv, None, tokens, O.ratio_schedule(0.0, MICRO.n_layers, 1, False),
                  segments=[order[0], rest])
    for l in range(MICRO.n_layers):
        np.testing.assert_allclose(ref["K"][l], full["K"][l], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(ref["h_last"], full["x"][-1][-1], rtol=1e-9, atol=1e-10)
