"""Helpers for the GPU parity tests: moving generator arrays to the device and back, and the
relative Frobenius error used as the float bar (1e-4 in fp32, 1e-2 in bf16)."""
import numpy as np
import pytest

TOL = {"f32": 1e-4, "bf16": 1e-2}


def torch_mod():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch


def ensure_lib():
    from non_prefix_kv_gb300 import build as nb
    nb.build()
    from non_prefix_kv_gb300 import binding as B
    return B.lib()


def dev(a, dtype="f32"):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def dev_i32(a):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host(t):
    return t.detach().double().cpu().numpy()


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def tdt(dtype):
    torch = torch_mod()
    return torch.bfloat16 if dtype == "bf16" else torch.float32
