"""The tensor-core GEMM has two kernels: single-SM 128-row tiles and CTA-pair 256-row tiles
(tcgen05.mma.cta_group::2), chosen per launch.  The default choice sends the large-M layer
GEMMs to pairs and small or padding-heavy ones to single SMs; these tests run the GEMM and
layer parity tests once more with each kernel forced for every launch (CB_GEMM_PAIR, read
once per process, hence the child processes), so both kernels are checked at every shape
and epilogue: tiny and ragged M, N and K, the RoPE/KV-scatter, residual, SwiGLU and fused
deviation epilogues, and whole blended layers."""
import os
import subprocess
import sys

import pytest

from tests.gpu_util import ensure_lib, torch_mod

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("mode", ["0", "1"], ids=["single_sm", "cta_pair"])
def test_gemm_parity_with_each_kernel_forced(mode):
    torch_mod()
    ensure_lib()
    env = dict(os.environ, CB_GEMM_PAIR=mode)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_kernels.py", "tests/test_gpu_blend.py", "-m",
                        "gpu", "-x", "-q", "-p", "no:cacheprovider", "-k",
                        "linear or qkv or o_proj or check_layer or blend"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


@pytest.mark.parametrize("mode", ["0", "1"], ids=["one_query_tile", "two_query_tiles"])
def test_attention_parity_with_each_kernel_forced(mode):
    """The tensor-core attention has two kernels: one query tile per CTA (two softmax groups
    on alternate key tiles) and two query tiles per CTA (one group per query tile over every
    key tile), chosen by the query tiles per head.  The attention and blend parity tests run
    once more with each kernel forced for every launch (CB_ATTN_PAIR)."""
    torch_mod()
    ensure_lib()
    env = dict(os.environ, CB_ATTN_PAIR=mode)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_kernels.py", "tests/test_gpu_blend.py", "-m",
                        "gpu", "-x", "-q", "-p", "no:cacheprovider", "-k", "attention or attn or blend"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
