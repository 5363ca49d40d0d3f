"""The allocation-free deviation/top-k entry point gives the same scores and the same
selected rows as the workspace entry point, on two calls in a row.

It exists for callers that cannot give the library device memory (a plugin inside a host
program that owns all device memory, or a caller that must not call cudaMalloc).  Its
scratch is one fixed array in the library, shared by every call, so the second call here
runs on scratch that still holds the first call's contents.  This file is collected last
so that a run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

from non_prefix_kv_gb300 import synth
from tests.gpu_util import dev, dev_i32, ensure_lib, host, torch_mod

pytestmark = pytest.mark.gpu


def _case(B, seed, n_ref, n_new, n_cand, k, dtype, dev_mode):
    torch = torch_mod()
    from non_prefix_kv_gb300 import engine as E
    shape = synth.ModelShape(1, 256, 8, 2, 128, 256, 64, dtype=dtype)
    dims = E.make_dims(shape)
    W = shape.kv_width
    g = synth.rng(seed, synth.P_NOISE)
    kr = dev(synth.test_tensor((n_ref, W), seed + 1, dtype=dtype), dtype)
    vr = dev(synth.test_tensor((n_ref, W), seed + 2, dtype=dtype), dtype)
    kn = dev(synth.test_tensor((n_new, W), seed + 3, dtype=dtype), dtype)
    vn = dev(synth.test_tensor((n_new, W), seed + 4, dtype=dtype), dtype)
    new_row = dev_i32(np.sort(g.choice(n_new, n_cand, replace=False)))
    ref_row = dev_i32(np.sort(g.choice(n_ref, n_cand, replace=False)))
    # workspace entry point: the expected result
    sc_ref = torch.empty(n_cand, dtype=torch.float32, device="cuda")
    sel_ref = torch.full((max(k, 1),), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    B.cb_kv_deviation_topk(kn, vn, kr, vr, new_row, ref_row, n_cand, k, dev_mode, dims, sc_ref, sel_ref, ws)
    # allocation-free entry point, once with caller-provided scores, once with scores kept
    # in the fixed scratch
    sc = torch.empty(n_cand, dtype=torch.float32, device="cuda")
    sel = torch.full((max(k, 1),), -1, dtype=torch.int32, device="cuda")
    B.cb_kv_deviation_topk_noalloc(kn, vn, kr, vr, new_row, ref_row, n_cand, k, dev_mode, dims, sc, sel)
    sel2 = torch.full((max(k, 1),), -1, dtype=torch.int32, device="cuda")
    B.cb_kv_deviation_topk_noalloc(kn, vn, kr, vr, new_row, ref_row, n_cand, k, dev_mode, dims, None, sel2)
    B.cb_sync(None)
    a, b = host(sc), host(sc_ref)
    assert np.max(np.abs(a - b) / b) < 1e-5
    np.testing.assert_array_equal(sel[:k].cpu().numpy(), sel_ref[:k].cpu().numpy())
    np.testing.assert_array_equal(sel2[:k].cpu().numpy(), sel_ref[:k].cpu().numpy())


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    torch_mod()
    ensure_lib()
    from non_prefix_kv_gb300 import binding as B
    # first call: larger problem; second call: smaller problem over the stale scratch
    _case(B, 100, n_ref=5000, n_new=4000, n_cand=3840, k=576, dtype="bf16", dev_mode=0)
    _case(B, 200, n_ref=900, n_new=800, n_cand=700, k=105, dtype="f32", dev_mode=1)


def test_noalloc_rejects_more_candidates_than_its_scratch():
    torch_mod()
    ensure_lib()
    from non_prefix_kv_gb300 import binding as B
    from non_prefix_kv_gb300 import engine as E
    dims = E.make_dims(synth.ModelShape(1, 256, 8, 2, 128, 256, 64, dtype="bf16"))
    fake = 0x10000      # never dereferenced: the size check fails before any launch
    st = B.lib().cb_kv_deviation_topk_noalloc(fake, fake, 65537, fake, fake, 65537, None, None, 65537, 10, 0,
                                              ctypes.byref(dims), None, fake, None)
    assert st == 8
    assert b"65536" in B.lib().cb_last_error_message()
