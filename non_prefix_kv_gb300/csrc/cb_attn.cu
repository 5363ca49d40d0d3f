// Attention of selected queries over the whole causal KV (CacheBlend explainer,
// 0h-n0.github.io/posts/paper-2312-03052, §Selective recomputation Step 4; abeam.tech
// CacheBlend explainer §技術の仕組み: the selected tokens attend over the entire input).
//
//   out[j, h] = sum_{t <= q_pos[j]} softmax_t(q[j,h] . K[t,g] / sqrt(hd)) V[t,g],
//   g = h / (H / Hkv)
//
// SIMT kernel (fp32 parity mode): one 128-thread block per (query row, head); each warp streams a contiguous
// quarter of the visible keys with an online softmax, lanes splitting the head dimension;
// the four partial states are merged at the end.  fp32 arithmetic throughout.
#include <math.h>

#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

static __device__ uint32_t g_err_attn;

uint32_t take_error_attn() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_attn, sizeof(v)) != cudaSuccess) return ERRBIT_INDEX;
  cudaMemcpyToSymbol(g_err_attn, &z, sizeof(z));
  return v;
}

template <typename T, int DPL>
__global__ void __launch_bounds__(128) k_attn_simt(const T* __restrict__ q, const int32_t* __restrict__ q_pos,
                                                   const T* __restrict__ kc, const T* __restrict__ vc,
                                                   int64_t n_kv, int H, int Hkv, T* __restrict__ out,
                                                   float scale) {
  pdl_wait();
  pdl_trigger();
  constexpr int HD = DPL * 32;
  __shared__ float s_m[4], s_l[4];
  __shared__ float s_o[4][HD];
  const int j = blockIdx.x, h = blockIdx.y;
  const int g = h / (H / Hkv);
  const int64_t W = (int64_t)Hkv * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t p = q_pos[j];
  if (p < 0 || p >= n_kv) {
    if (threadIdx.x == 0) atomicOr(&g_err_attn, ERRBIT_INDEX);
    p = p < 0 ? 0 : n_kv - 1;
  }
  float qv[DPL];
  const T* qr = q + (int64_t)j * H * HD + (int64_t)h * HD + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) qv[i] = to_f(qr[i]) * scale;
  const int64_t nk = p + 1;
  const int64_t per = (nk + 3) / 4;
  const int64_t t0 = warp * per;
  const int64_t t1 = t0 + per < nk ? t0 + per : nk;
  float mrun = -INFINITY, l = 0.f, acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
  for (int64_t t = t0; t < t1; ++t) {
    const T* kr = kc + t * W + (int64_t)g * HD + lane * DPL;
    float sc = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) sc = fmaf(qv[i], to_f(kr[i]), sc);
    sc = warp_sum(sc);
    const float mnew = fmaxf(mrun, sc);
    const float corr = expf(mrun - mnew);
    const float pr = expf(sc - mnew);
    l = l * corr + pr;
    const T* vr = vc + t * W + (int64_t)g * HD + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = fmaf(acc[i], corr, pr * to_f(vr[i]));
    mrun = mnew;
  }
  if (lane == 0) {
    s_m[warp] = mrun;
    s_l[warp] = l;
  }
#pragma unroll
  for (int i = 0; i < DPL; ++i) s_o[warp][lane * DPL + i] = acc[i];
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, s_m[w]);
    float f[4], L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      f[w] = s_l[w] > 0.f ? expf(s_m[w] - mx) : 0.f;
      L += s_l[w] * f[w];
    }
    const float inv = 1.0f / L;
    T* orow = out + (int64_t)j * H * HD + (int64_t)h * HD;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int d = lane * DPL + i;
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) o = fmaf(s_o[w][d], f[w], o);
      orow[d] = from_f<T>(o * inv);
    }
  }
}

size_t attention_ws_bytes(int, int64_t, int, int) { return 0; }

template <typename T>
static cudaError_t launch_simt(const void* q, const int32_t* q_pos, int M, const void* kc,
                               const void* vc, int64_t n_kv, int H, int Hkv, int hd, void* out,
                               cudaStream_t s) {
  dim3 grid(M, H);
  const float scale = 1.0f / sqrtf((float)hd);
#define CB_ATTN_CASE(DPL)                                                                               \
  case DPL * 32: {                                                                                      \
    const cudaError_t e_ = launch_k(k_attn_simt<T, DPL>, dim3(grid), dim3(128), 0, s, (const T*)q, q_pos, \
                                    (const T*)kc, (const T*)vc, n_kv, H, Hkv, (T*)out, scale);            \
    if (e_ != cudaSuccess) return e_;                                                                   \
  } break;
  switch (hd) {
    CB_ATTN_CASE(1)
    CB_ATTN_CASE(2)
    CB_ATTN_CASE(4)
    CB_ATTN_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef CB_ATTN_CASE
  return cudaGetLastError();
}

bool attention_tc_supported(int hd);
cudaError_t launch_attention_tc(const void* q, const int32_t* q_pos, int M, const void* kc, const void* vc,
                                int64_t n_kv, int H, int Hkv, int hd, void* out, cudaStream_t s);

// bf16 with head_dim 64/128 runs on the tcgen05 kernel (cb_attn_tc.cu); fp32 (the exact
// parity mode) and other head sizes on the SIMT kernel above.
cudaError_t launch_attention(int dt, const void* q, const int32_t* q_pos, int M, const void* kc,
                             const void* vc, int64_t n_kv, int H, int Hkv, int hd, void* out,
                             void* ws, size_t ws_bytes, cudaStream_t s) {
  (void)ws;
  (void)ws_bytes;
  if (M == 0) return cudaSuccess;
  if (dt == DT_BF16 && attention_tc_supported(hd))
    return launch_attention_tc(q, q_pos, M, kc, vc, n_kv, H, Hkv, hd, out, s);
  if (dt == DT_BF16) return launch_simt<bf16>(q, q_pos, M, kc, vc, n_kv, H, Hkv, hd, out, s);
  return launch_simt<float>(q, q_pos, M, kc, vc, n_kv, H, Hkv, hd, out, s);
}

}  // namespace cb
