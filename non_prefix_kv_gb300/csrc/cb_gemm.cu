// GEMM dispatch.  fp32 runs on a plain SIMT kernel (exact fp32 FMA, no TF32, so the fp32
// mode stays within 1e-4 of the fp64 oracle); bf16 runs on the tcgen05/TMEM kernel
// (cb_gemm_tc.cu).
#include "cb_common.cuh"
#include "cb_epilogue.cuh"
#include "cb_internal.h"

namespace cb {

static __device__ uint32_t g_err_gemm;

uint32_t take_error_gemm() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_gemm, sizeof(v)) != cudaSuccess) return ERRBIT_INDEX;
  cudaMemcpyToSymbol(g_err_gemm, &z, sizeof(z));
  return v;
}

// acc[m][n] = sum_k A[m][k] B[n][k]; 64x64 tile per 256-thread block, 4x4 per thread.
// EPI_SWIGLU: the 64 tile columns are 32 gate rows (j) and their 32 up partners
// (b_up_row + j) of B; the block then writes out[m][j] = silu(gate) * up for 32 j.
template <typename T>
__global__ void __launch_bounds__(256) k_gemm_simt(const GemmDesc g) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[16][64 + 1];
  __shared__ float Bs[16][64 + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool swiglu = g.epi.kind == EPI_SWIGLU;
  const int m0 = blockIdx.y * 64;
  const int n0 = swiglu ? blockIdx.x * 32 : blockIdx.x * 64;
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < g.K; k0 += 16) {
    for (int e = threadIdx.x; e < 1024; e += 256) {
      const int r = e >> 4, c = e & 15;
      const int gk = k0 + c;
      const int gm = m0 + r;
      int64_t brow;
      if (!swiglu) {
        brow = n0 + r < g.N ? n0 + r : -1;
      } else {
        const int j = n0 + (r & 31);
        brow = j < g.N ? (r < 32 ? (int64_t)j : g.b_up_row + j) : -1;
      }
      As[c][r] = (gm < g.M && gk < g.K) ? to_f(A[(int64_t)gm * g.lda + gk]) : 0.f;
      Bs[c][r] = (brow >= 0 && gk < g.K) ? to_f(B[brow * g.ldb + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (swiglu) {
    __shared__ float Cs[64][64 + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
    __syncthreads();
    if (tx >= 8) return;
    const int n = n0 + tx * 4;
    if (n >= g.N) return;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + ty * 4 + i;
      if (m >= g.M) continue;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = silu_f(Cs[ty * 4 + i][tx * 4 + j]) * Cs[ty * 4 + i][32 + tx * 4 + j];
      st4((T*)g.epi.out + (int64_t)m * g.epi.ldo + n, v);
    }
    return;
  }
  const int n = n0 + tx * 4;
  if (n >= g.N) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m < g.M) {
      if (!epi_apply<T, 4>(g.epi, m, n, acc[i])) atomicOr(&g_err_gemm, ERRBIT_INDEX);
    }
  }
}

template <typename T>
static cudaError_t launch_simt(const GemmDesc& g, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  const int cols = g.epi.kind == EPI_SWIGLU ? 32 : 64;
  dim3 grid((g.N + cols - 1) / cols, (g.M + 63) / 64);
  { const cudaError_t e_ = launch_k(k_gemm_simt<T>, dim3(grid), dim3(256), 0, s, g); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const GemmDesc& g, cudaStream_t s);  // cb_gemm_tc.cu

cudaError_t launch_gemm_tc_group(const GemmDesc* gs, int n, cudaStream_t s);

cudaError_t launch_gemm(int dt, const GemmDesc& g, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (dt == DT_BF16) return launch_gemm_tc(g, s);
  return launch_simt<float>(g, s);
}

// Two independent GEMMs: one tensor-core launch sharing its tile walk when both are
// non-empty bf16 problems, otherwise one after the other.
cudaError_t launch_gemm_pair(int dt, const GemmDesc& a, const GemmDesc& b, cudaStream_t s) {
  const bool ea = a.M == 0 || a.N == 0, eb = b.M == 0 || b.N == 0;
  if (dt == DT_BF16 && !ea && !eb) {
    const GemmDesc gs[2] = {a, b};
    return launch_gemm_tc_group(gs, 2, s);
  }
  cudaError_t e = launch_gemm(dt, a, s);
  if (e != cudaSuccess) return e;
  return launch_gemm(dt, b, s);
}

}  // namespace cb
