// GEMM epilogues shared by the SIMT and the tcgen05 GEMMs.  Each call receives NV
// consecutive accumulator columns [n, n+NV) of output row m (n % NV == 0, NV even).
//
// EPI_QKV implements the Q/K/V step of selective recompute (CacheBlend explainer,
// 0h-n0.github.io/posts/paper-2312-03052, §Selective recomputation Step 2) with RoPE
// (§RoPE: pairs (x[2i], x[2i+1]) rotated by pos * theta_i) and, when kv_row is given, the
// KV expansion of Step 3 fused in (rows written straight into the cache).
#pragma once
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

template <typename T, int NV>
__device__ __forceinline__ void st_vec(T* p, const float* v) {
  if constexpr (NV == 16 && sizeof(T) == 2) {
    if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
      st16_v8(p, v);
      return;
    }
  }
  if constexpr (NV % 8 == 0) {
#pragma unroll
    for (int i = 0; i < NV; i += 8) st8(p + i, v + i);
  } else {
#pragma unroll
    for (int i = 0; i < NV; i += 4) st4(p + i, v + i);
  }
}
template <typename T, int NV>
__device__ __forceinline__ void ld_vec(const T* p, float* v) {
  if constexpr (NV == 16 && sizeof(T) == 2) {
    if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
      ld16_v8(p, v);
      return;
    }
  }
  if constexpr (NV % 8 == 0) {
#pragma unroll
    for (int i = 0; i < NV; i += 8) ld8(p + i, v + i);
  } else {
#pragma unroll
    for (int i = 0; i < NV; i += 4) ld4(p + i, v + i);
  }
}

// Rotate NV/2 interleaved pairs starting at pair index i0 by position pos.
template <int NV>
__device__ __forceinline__ void rope_vec(float* v, const float* tab, int half, int pos, int i0) {
  const float2* t = reinterpret_cast<const float2*>(tab) + (int64_t)pos * half + i0;
#pragma unroll
  for (int q = 0; q < NV / 2; ++q) {
    const float2 cs = t[q];
    const float x0 = v[2 * q], x1 = v[2 * q + 1];
    v[2 * q] = x0 * cs.x - x1 * cs.y;
    v[2 * q + 1] = x0 * cs.y + x1 * cs.x;
  }
}

// Returns false (and does nothing) if an index is out of range; the caller records it.
template <typename T, int NV>
__device__ __forceinline__ bool epi_apply(const EpiParams& p, int m, int n, float* v) {
  switch (p.kind) {
    case EPI_STORE:
      st_vec<T, NV>((T*)p.out + (int64_t)m * p.ldo + n, v);
      return true;
    case EPI_RESID: {
      const int64_t rr = p.resid_row ? (int64_t)p.resid_row[m] : (int64_t)m;
      if (rr < 0 || (p.resid_rows >= 0 && rr >= p.resid_rows)) return false;
      float r[NV];
      ld_vec<T, NV>((const T*)p.resid + rr * p.ldr + n, r);
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] += r[i];
      st_vec<T, NV>((T*)p.out + (int64_t)m * p.ldo + n, v);
      return true;
    }
    case EPI_QKV: {
      const int g = p.col0 + n;
      const int half = p.hd >> 1;
      if (g < p.q_cols + p.kv_cols) {
        const int pos = p.pos[m];
        if (pos < 0 || pos >= p.max_pos) return false;
        const int seg = g < p.q_cols ? g : g - p.q_cols;
        rope_vec<NV>(v, p.rope, half, pos, (seg % p.hd) >> 1);
      }
      if (g < p.q_cols) {
        st_vec<T, NV>((T*)p.q + (int64_t)m * p.ldq + g, v);
        return true;
      }
      const int64_t kr = p.kv_row ? (int64_t)p.kv_row[m] : (int64_t)m;
      if (kr < 0 || (p.kv_bound >= 0 && kr >= p.kv_bound)) return false;
      if (g < p.q_cols + p.kv_cols)
        st_vec<T, NV>((T*)p.k + kr * p.ldkv + (g - p.q_cols), v);
      else
        st_vec<T, NV>((T*)p.v + kr * p.ldkv + (g - p.q_cols - p.kv_cols), v);
      return true;
    }
    default:
      return false;
  }
}

// Squared deviation of 16 new K/V values (rotated, rounded to bf16 as they are stored)
// from the 16 cached bf16 values in r: one chunk of the per-token KV deviation of HKVD
// selection (CacheBlend explainer, §Selective recomputation Step 1), taken where the new
// K/V are produced.
__device__ __forceinline__ float sq_dev16(const float* v, const uint4* r) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(r);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 c = __bfloat1622float2(h[i]);
    const float d0 = __bfloat162float(__float2bfloat16_rn(v[2 * i])) - c.x;
    const float d1 = __bfloat162float(__float2bfloat16_rn(v[2 * i + 1])) - c.y;
    s = fmaf(d0, d0, s);
    s = fmaf(d1, d1, s);
  }
  return s;
}

}  // namespace cb
