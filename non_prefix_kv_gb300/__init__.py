"""GB300-native (sm_103a) selective KV recompute for blended prefill (CacheBlend).

Layout: csrc/ (CUDA kernels and the C ABI, built into libcacheblend.so), binding.py (ctypes
binding under the C names), engine.py (device weights, chunk pool, per-request layer loop),
synth.py (seeded synthetic inputs), build.py (nvcc build)."""
__all__ = ["binding", "engine", "synth", "build"]
