// Bandwidth- and latency-bound kernels of the blend path: RoPE table and re-rotation (also
// from 8-bit per-channel codes, and the 8-bit quantization itself), row gathers/scatters and
// the batched row copies after a selection (also in small blocks that run beside a GEMM),
// RMSNorm, KV deviation, exact top-k, selection bookkeeping, lm_head GEMV + argmax.
//
// Sources: CacheBlend explainer (0h-n0.github.io/posts/paper-2312-03052) — §KV deviation,
// §HKVD selection, §Selective recomputation Steps 1 and 3, §RoPE; Prompt Cache explainer
// (0h-n0.github.io/posts/paper-2402-01008) — §RoPE position adjustment.
#include <mutex>

#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

static __device__ uint32_t g_err_mem;

// Host-side caches of this file, per device: SM count, resident blocks per kernel, the
// top-k kernel's shared-memory attribute, the allocation-free scratch address.  One mutex
// guards them (calls may come from several host threads); reset_mem_caches() empties them.
namespace {
std::mutex g_mem_mu;
int g_sms[64];
struct ResidentEnt {
  const void* k;
  int dev, threads, n;
};
ResidentEnt g_resident[64];
int g_resident_used = 0;
bool g_topk_attr[64];
void* g_noalloc_addr[64];
}  // namespace

void reset_mem_caches() {
  std::lock_guard<std::mutex> g(g_mem_mu);
  for (int i = 0; i < 64; ++i) {
    g_sms[i] = 0;
    g_topk_attr[i] = false;
    g_noalloc_addr[i] = nullptr;
  }
  g_resident_used = 0;
}

static int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  {
    std::lock_guard<std::mutex> g(g_mem_mu);
    if (g_sms[dev]) return g_sms[dev];
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();   // clears the error of the call just made (nothing is cached)
    return 148;
  }
  if (n <= 0) return 148;
  std::lock_guard<std::mutex> g(g_mem_mu);
  g_sms[dev] = n;
  return n;
}

// Blocks of `threads` threads of this kernel resident per SM at once (registers, shared
// memory), once per kernel, block size and device.  A failed query is not cached.
static int resident_blocks(const void* kernel, int threads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  {
    std::lock_guard<std::mutex> g(g_mem_mu);
    for (int i = 0; i < g_resident_used; ++i)
      if (g_resident[i].k == kernel && g_resident[i].dev == dev && g_resident[i].threads == threads)
        return g_resident[i].n;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess) {
    cudaGetLastError();   // clears the error of the call just made
    return 1;
  }
  if (n < 1) n = 1;
  std::lock_guard<std::mutex> g(g_mem_mu);
  if (g_resident_used < 64) g_resident[g_resident_used++] = ResidentEnt{kernel, dev, threads, n};
  return n;
}

// grid for a grid-stride loop: enough blocks for the work, at most as many as are resident
// at once (a block beyond that would run in a partial second round, after the others)
template <typename K>
static unsigned grid_for(K* kernel, int64_t work_items, int threads) {
  int64_t b = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void*>(kernel), threads);
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (unsigned)b;
}

uint32_t take_error_mem() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mem, sizeof(v)) != cudaSuccess) return ERRBIT_INDEX;
  cudaMemcpyToSymbol(g_err_mem, &z, sizeof(z));
  return v;
}

// ------------------------------------------------------------------------ RoPE table
// tab[p][i] = (cos(p theta_i), sin(p theta_i)), theta_i = base^(-2i/hd); angle in fp64.
__global__ void k_rope_table(float2* tab, int max_pos, int half, int hd, double base) {
  pdl_wait();
  pdl_trigger();
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)max_pos * half) return;
  int p = (int)(t / half), i = (int)(t % half);
  double theta = pow(base, -2.0 * (double)i / (double)hd);
  double s, c;
  sincos((double)p * theta, &s, &c);
  tab[t] = make_float2((float)c, (float)s);
}

cudaError_t launch_rope_table(float* tab, int max_pos, int hd, double base, cudaStream_t s) {
  int half = hd / 2;
  int64_t n = (int64_t)max_pos * half;
  if (n == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_rope_table, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, reinterpret_cast<float2*>(tab),
                                                           max_pos, half, hd, base); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ RoPE shift
// k_dst[r] = R(delta[r]) k_src[src_row[r]]; v_dst[r] = v_src[src_row[r]].
// One thread per 8 consecutive elements (4 rotation pairs, never crossing a head since
// hd % 8 == 0).  The negative-offset rotation negates the sine.  A source row outside
// [0, n_src) or an offset outside the table records ERRBIT_INDEX and the row is skipped.
template <typename T>
__global__ void __launch_bounds__(256) k_rope_shift(T* __restrict__ kd, T* __restrict__ vd,
                                                    const T* ks, const T* __restrict__ vs,
                                                    const int32_t* __restrict__ src_row,
                                                    const int32_t* __restrict__ delta,
                                                    int64_t n_rows, int64_t n_src, int W, int hd,
                                                    const float2* __restrict__ tab, int max_pos,
                                                    unsigned long long* span) {
  pdl_wait();
  pdl_trigger();
  span_begin(span);
  const int per_row = W >> 3;
  const int half = hd >> 1;
  const int64_t total = n_rows * per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / per_row;
    const int c0 = (int)(t - r * per_row) << 3;
    const int64_t sr = src_row ? (int64_t)src_row[r] : r;
    const int dl = delta[r];
    const int ad = dl < 0 ? -dl : dl;
    if (ad >= max_pos || sr < 0 || sr >= n_src) {
      atomicOr(&g_err_mem, ERRBIT_INDEX);
      continue;
    }
    const float sg = dl < 0 ? -1.0f : 1.0f;
    float x[8], y[8];
    ld8(ks + sr * W + c0, x);
    const float2* tb = tab + (int64_t)ad * half + ((c0 % hd) >> 1);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 cs = tb[q];
      const float c = cs.x, sn = cs.y * sg;
      y[2 * q] = x[2 * q] * c - x[2 * q + 1] * sn;
      y[2 * q + 1] = x[2 * q] * sn + x[2 * q + 1] * c;
    }
    st8(kd + r * W + c0, y);
    if (vd) {
      float v[8];
      ld8(vs + sr * W + c0, v);
      st8(vd + r * W + c0, v);
    }
  }
  if (span) {   // uniform; every thread of the block reaches this point
    __syncthreads();
    span_end(span);
  }
}

cudaError_t launch_rope_shift(int dt, void* kd, void* vd, const void* ks, const void* vs,
                              const int32_t* src_row, int64_t n_src, const int32_t* delta,
                              int64_t n_rows, int W, int hd, const float* tab, int max_pos,
                              cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t work = n_rows * (W / 8);
  const unsigned grid = dt == DT_BF16 ? grid_for(k_rope_shift<bf16>, work, 256) : grid_for(k_rope_shift<float>, work, 256);
  const float2* t2 = reinterpret_cast<const float2*>(tab);
  if (dt == DT_BF16)
    { const cudaError_t e_ = launch_k(k_rope_shift<bf16>, dim3(grid), dim3(256), 0, s, (bf16*)kd, (bf16*)vd, (const bf16*)ks,
                                            (const bf16*)vs, src_row, delta, n_rows, n_src, W, hd, t2,
                                            max_pos, prof_span_slot()); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_rope_shift<float>, dim3(grid), dim3(256), 0, s, (float*)kd, (float*)vd, (const float*)ks,
                                             (const float*)vs, src_row, delta, n_rows, n_src, W, hd, t2,
                                             max_pos, prof_span_slot()); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ 8-bit chunk KV
// Per-channel asymmetric quantization of one [n, W] block (CacheGen explainer, §Step 1
// per-channel quantization): zero = min over the rows, scale = max((max - min) / 255,
// 1e-8), code = rint((x - zero) / scale) clipped to [0, 255]; every step is one IEEE fp32
// operation so the code decision is reproducible.  A block owns 32 channels (a warp reads
// 32 consecutive channels of a row); its 8 warps stride the rows, then combine.
template <typename T>
__global__ void __launch_bounds__(256) k_kv_quantize(const T* __restrict__ x, int64_t n, int W,
                                                     uint8_t* __restrict__ q, float* __restrict__ scale,
                                                     float* __restrict__ zero) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_lo[8][32], s_hi[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float lo = INFINITY, hi = -INFINITY;
  bool bad = false;
  if (c < W) {
    for (int64_t t = w; t < n; t += 8) {
      const float v = to_f(x[t * W + c]);
      bad |= !isfinite(v);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
  }
  s_lo[w][lane] = lo;
  s_hi[w][lane] = hi;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo = fminf(lo, s_lo[i][lane]);
    hi = fmaxf(hi, s_hi[i][lane]);
  }
  if (bad) atomicOr(&g_err_mem, ERRBIT_NONFINITE);
  if (c >= W) return;
  const float sc = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), 255.0f), 1e-8f);
  if (w == 0) {
    scale[c] = sc;
    zero[c] = lo;
  }
  for (int64_t t = w; t < n; t += 8) {
    const float v = to_f(x[t * W + c]);
    const float r = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v, lo), sc)), 0.0f), 255.0f);
    q[t * W + c] = static_cast<uint8_t>(r);
  }
}

cudaError_t launch_kv_quantize(int dt, const void* x, int64_t n, int W, uint8_t* q, float* scale,
                               float* zero, cudaStream_t s) {
  if (n == 0 || W == 0) return cudaSuccess;
  const dim3 grid((unsigned)((W + 31) / 32));
  if (dt == DT_BF16)
    { const cudaError_t e_ = launch_k(k_kv_quantize<bf16>, grid, dim3(256), 0, s, (const bf16*)x, n, W, q, scale, zero); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_kv_quantize<float>, grid, dim3(256), 0, s, (const float*)x, n, W, q, scale, zero); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// x = code * s + z (product rounded, then the sum: no fused multiply-add) for 8 channels
__device__ __forceinline__ void dequant8(uint2 u, const float* sv, const float* zv, float* x) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t word = i < 4 ? u.x : u.y;
    const float code = static_cast<float>((word >> (8 * (i & 3))) & 0xffu);
    x[i] = __fadd_rn(__fmul_rn(code, sv[i]), zv[i]);
  }
}
__device__ __forceinline__ void load_tab8(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

constexpr int kQ8Rows = 8;   // rows per thread: a chunk's scale/zero stay in registers across them

// k_dst[r] = R(delta[r]) dequant(k_codes[src_row[r]]), v_dst[r] = dequant(v_codes[src_row[r]])
// with the scale/zero row qrow[r] of the per-chunk tables: loading 8-bit chunk KV and
// re-positioning it in one pass.  A thread owns 8 channels of kQ8Rows consecutive rows
// (consecutive threads: consecutive channel groups of the same rows) and reloads the
// channels' scale/zero only when the row's chunk changes.
template <typename T>
__global__ void __launch_bounds__(256) k_rope_shift_q8(T* __restrict__ kd, T* __restrict__ vd,
                                                       const uint8_t* __restrict__ kq,
                                                       const uint8_t* __restrict__ vq,
                                                       const float* __restrict__ ks, const float* __restrict__ kz,
                                                       const float* __restrict__ vs, const float* __restrict__ vz,
                                                       const int32_t* __restrict__ src_row, int64_t n_src,
                                                       const int32_t* __restrict__ qrow, int n_q,
                                                       const int32_t* __restrict__ delta, int64_t n_rows, int W,
                                                       int hd, const float2* __restrict__ tab, int max_pos) {
  pdl_wait();
  pdl_trigger();
  const int per_row = W >> 3;
  const int half = hd >> 1;
  const int64_t n_blocks = (n_rows + kQ8Rows - 1) / kQ8Rows;
  const int64_t total = n_blocks * per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rb = t / per_row;
    const int c0 = (int)(t - rb * per_row) << 3;
    const int pair0 = (c0 % hd) >> 1;
    // every row's indices and codes are loaded before any arithmetic (loads in flight)
    int64_t rr[kQ8Rows];
    int qv[kQ8Rows], dv[kQ8Rows];
    uint2 uk[kQ8Rows], uv[kQ8Rows];
#pragma unroll
    for (int j = 0; j < kQ8Rows; ++j) {
      const int64_t r = rb * kQ8Rows + j;
      rr[j] = -1;
      uk[j] = uv[j] = make_uint2(0, 0);
      if (r >= n_rows) continue;
      const int64_t sr = src_row ? (int64_t)src_row[r] : r;
      const int qi = qrow[r];
      const int dl = delta[r];
      const int ad = dl < 0 ? -dl : dl;
      if (ad >= max_pos || sr < 0 || sr >= n_src || qi < 0 || qi >= n_q) {
        atomicOr(&g_err_mem, ERRBIT_INDEX);
        continue;
      }
      rr[j] = r;
      qv[j] = qi;
      dv[j] = dl;
      uk[j] = *reinterpret_cast<const uint2*>(kq + sr * W + c0);
      if (vd) uv[j] = *reinterpret_cast<const uint2*>(vq + sr * W + c0);
    }
    int cur = -1;
    float ksv[8], kzv[8], vsv[8], vzv[8];
#pragma unroll
    for (int j = 0; j < kQ8Rows; ++j) {
      if (rr[j] < 0) continue;
      const int64_t r = rr[j];
      if (qv[j] != cur) {
        cur = qv[j];
        load_tab8(ks + (int64_t)cur * W + c0, ksv);
        load_tab8(kz + (int64_t)cur * W + c0, kzv);
        if (vd) {
          load_tab8(vs + (int64_t)cur * W + c0, vsv);
          load_tab8(vz + (int64_t)cur * W + c0, vzv);
        }
      }
      const int dl = dv[j];
      const int ad = dl < 0 ? -dl : dl;
      const float sg = dl < 0 ? -1.0f : 1.0f;
      float x[8], y[8];
      dequant8(uk[j], ksv, kzv, x);
      const float2* tb = tab + (int64_t)ad * half + pair0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 cs = tb[q];
        const float c = cs.x, sn = cs.y * sg;
        y[2 * q] = x[2 * q] * c - x[2 * q + 1] * sn;
        y[2 * q + 1] = x[2 * q] * sn + x[2 * q + 1] * c;
      }
      st8(kd + r * W + c0, y);
      if (vd) {
        float v[8];
        dequant8(uv[j], vsv, vzv, v);
        st8(vd + r * W + c0, v);
      }
    }
  }
}

cudaError_t launch_rope_shift_q8(int dt, void* kd, void* vd, const uint8_t* kq, const uint8_t* vq,
                                 const float* ks, const float* kz, const float* vs, const float* vz,
                                 const int32_t* src_row, int64_t n_src, const int32_t* qrow, int n_q,
                                 const int32_t* delta, int64_t n_rows, int W, int hd, const float* tab,
                                 int max_pos, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t work = (n_rows + kQ8Rows - 1) / kQ8Rows * (W / 8);
  const unsigned grid = dt == DT_BF16 ? grid_for(k_rope_shift_q8<bf16>, work, 256) : grid_for(k_rope_shift_q8<float>, work, 256);
  const float2* t2 = reinterpret_cast<const float2*>(tab);
  if (dt == DT_BF16)
    { const cudaError_t e_ = launch_k(k_rope_shift_q8<bf16>, dim3(grid), dim3(256), 0, s, (bf16*)kd, (bf16*)vd, kq, vq, ks, kz, vs, vz, src_row, n_src, qrow, n_q, delta, n_rows, W, hd, t2, max_pos); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_rope_shift_q8<float>, dim3(grid), dim3(256), 0, s, (float*)kd, (float*)vd, kq, vq, ks, kz, vs, vz, src_row, n_src, qrow, n_q, delta, n_rows, W, hd, t2, max_pos); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ row copies
// dst[dst_idx[r]] = src[src_idx[r]] for rows of rv vector words.  Index checks against the
// known buffer heights (bound < 0: unknown) record ERRBIT_INDEX and skip the row.  Each
// thread loads U words (a grid stride apart) before it stores any, so every SM keeps
// enough bytes in flight to stream from HBM.
template <typename V>
__global__ void __launch_bounds__(256) k_copy_rows(V* __restrict__ dst, const int32_t* __restrict__ di,
                                                   const V* __restrict__ src,
                                                   const int32_t* __restrict__ si, int64_t n,
                                                   int64_t rv, int64_t dbound, int64_t sbound) {
  pdl_wait();
  pdl_trigger();
  constexpr int U = 4;
  const int64_t total = n * rv;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t0 < total; t0 += U * stride) {
    V val[U];
    int64_t at[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      at[k] = -1;
      const int64_t t = t0 + k * stride;
      if (t >= total) continue;
      const int64_t r = t / rv, c = t - r * rv;
      const int64_t d = di ? (int64_t)di[r] : r;
      const int64_t sr = si ? (int64_t)si[r] : r;
      if (d < 0 || sr < 0 || (dbound >= 0 && d >= dbound) || (sbound >= 0 && sr >= sbound)) {
        atomicOr(&g_err_mem, ERRBIT_INDEX);
        continue;
      }
      val[k] = src[sr * rv + c];
      at[k] = d * rv + c;
    }
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (at[k] >= 0) dst[at[k]] = val[k];
  }
}

cudaError_t launch_copy_rows(void* dst, const int32_t* dst_idx, const void* src,
                             const int32_t* src_idx, int64_t n, int64_t row_bytes,
                             int64_t dst_bound, int64_t src_bound, cudaStream_t s) {
  if (n == 0 || row_bytes == 0) return cudaSuccess;
  const bool v16 = (row_bytes % 16 == 0) && ((uintptr_t)dst % 16 == 0) && ((uintptr_t)src % 16 == 0);
  if (v16) {
    const int64_t rv = row_bytes / 16;
    { const cudaError_t e_ = launch_k(k_copy_rows<uint4>, dim3(grid_for(k_copy_rows<uint4>, n * rv, 256)), dim3(256), 0, s, (uint4*)dst, dst_idx, (const uint4*)src,
                                                           src_idx, n, rv, dst_bound, src_bound); if (e_ != cudaSuccess) return e_; }
  } else {
    const int64_t rv = row_bytes / 4;
    { const cudaError_t e_ = launch_k(k_copy_rows<uint32_t>, dim3(grid_for(k_copy_rows<uint32_t>, n * rv, 256)), dim3(256), 0, s, (uint32_t*)dst, dst_idx,
                                                              (const uint32_t*)src, src_idx, n, rv,
                                                              dst_bound, src_bound); if (e_ != cudaSuccess) return e_; }
  }
  return cudaGetLastError();
}

// Up to kMaxCopyJobs independent row copies in one launch (the KV expansion and the row
// gathers that follow a selection share their indices and their moment).  One warp per row:
// the job, the indices and their checks are looked up once per row, and each lane issues
// all its 16-byte loads of the row (up to kCopyVec per pass) before it stores any.  Row r
// of all jobs together belongs to job j when row_end[j-1] <= r < row_end[j].
constexpr int kCopyVec = 16;
template <int VEC>
__device__ __forceinline__ void copy_rows_body(const CopyJobs& J) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t total = J.row_end[J.n - 1];
  for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < total; row += nwarps) {
    int j = 0;
    while (row >= J.row_end[j]) ++j;
    const int64_t r = row - (j ? J.row_end[j - 1] : 0);
    const int64_t d = J.di[j] ? (int64_t)J.di[j][r] : r;
    const int64_t sr = J.si[j] ? (int64_t)J.si[j][r] : r;
    if (d < 0 || sr < 0 || (J.dbound[j] >= 0 && d >= J.dbound[j]) || (J.sbound[j] >= 0 && sr >= J.sbound[j])) {
      if (lane == 0) atomicOr(&g_err_mem, ERRBIT_INDEX);   // warp-uniform: the whole row is skipped
      continue;
    }
    const int64_t rv = J.rv[j];
    const uint4* src = static_cast<const uint4*>(J.src[j]) + sr * rv;
    uint4* dst = static_cast<uint4*>(J.dst[j]) + d * rv;
    for (int64_t c0 = 0; c0 < rv; c0 += 32 * VEC) {
      uint4 v[VEC];
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        const int64_t c = c0 + k * 32 + lane;
        if (c < rv) v[k] = src[c];
      }
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        const int64_t c = c0 + k * 32 + lane;
        if (c < rv) dst[c] = v[k];
      }
    }
  }
}

__global__ void __launch_bounds__(256) k_copy_rows_multi(const CopyJobs J, unsigned long long* span) {
  pdl_wait();
  pdl_trigger();
  span_begin(span);
  copy_rows_body<kCopyVec>(J);
  if (span) {   // uniform; every thread of the block reaches this point
    __syncthreads();
    span_end(span);
  }
}

// The same copies in small blocks with few registers (four loads in flight per lane), for a
// launch that runs beside a tensor-core GEMM on another stream: a block fits in the registers
// and shared memory a GEMM CTA leaves free on its SM, so the copy proceeds on every SM instead
// of waiting for the GEMM's SMs to empty.
__global__ void __launch_bounds__(128) k_copy_rows_beside(const CopyJobs J, unsigned long long* span) {
  pdl_wait();
  pdl_trigger();
  span_begin(span);
  copy_rows_body<4>(J);
  if (span) {   // uniform; every thread of the block reaches this point
    __syncthreads();
    span_end(span);
  }
}

cudaError_t launch_copy_rows_multi(const CopyJobs& J, cudaStream_t s, bool beside) {
  if (J.n < 1 || J.n > kMaxCopyJobs) return cudaErrorInvalidValue;
  const int64_t rows = J.row_end[J.n - 1];
  if (rows == 0) return cudaSuccess;
  if (beside) {
    const cudaError_t e_ = launch_k(k_copy_rows_beside, dim3(grid_for(k_copy_rows_beside, rows * 32, 128)), dim3(128),
                                    0, s, J, prof_span_slot());
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_k(k_copy_rows_multi, dim3(grid_for(k_copy_rows_multi, rows * 32, 256)), dim3(256),
                                    0, s, J, prof_span_slot());
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ RMSNorm
// out[r] = x[rows[r]] / sqrt(mean(x^2) + eps) * g.  One block per row.  A row index outside
// [0, n_src) (n_src < 0: unchecked) records ERRBIT_INDEX and the output row is not written.
template <typename Ti, typename To>
__global__ void __launch_bounds__(256) k_rmsnorm(To* __restrict__ out, const Ti* __restrict__ x,
                                                 const int32_t* __restrict__ rows, int64_t n_src,
                                                 const Ti* __restrict__ g, int d, float eps) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  const int64_t r = blockIdx.x;
  const int64_t src = rows ? (int64_t)rows[r] : r;
  if (src < 0 || (n_src >= 0 && src >= n_src)) {   // uniform over the block
    if (threadIdx.x == 0) atomicOr(&g_err_mem, ERRBIT_INDEX);
    return;
  }
  const Ti* xr = x + src * d;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float v[8];
    ld8(xr + c, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  ss = warp_sum(ss);
  if (lane == 0) red[w] = ss;
  __syncthreads();
  if (w == 0) {
    float t = lane < nw ? red[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)d + eps);
  To* orow = out + r * d;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float v[8], gg[8], y[8];
    ld8(xr + c, v);
    if (g) {
      ld8(g + c, gg);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) gg[i] = 1.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = v[i] * inv * gg[i];
    st8(orow + c, y);
  }
}

// bf16 -> bf16 rows of up to 128*8*VPT elements: 128 threads per row, each holding its
// VPT 16-byte vectors in registers between the sum and the scaling (the row is read once).
template <int VPT>
__global__ void __launch_bounds__(128) k_rmsnorm_reg(bf16* __restrict__ out, const bf16* __restrict__ x,
                                                     const int32_t* __restrict__ rows, int64_t n_src,
                                                     const bf16* __restrict__ g, int d, float eps) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[4];
  const int64_t r = blockIdx.x;
  const int64_t src = rows ? (int64_t)rows[r] : r;
  if (src < 0 || (n_src >= 0 && src >= n_src)) {   // uniform over the block
    if (threadIdx.x == 0) atomicOr(&g_err_mem, ERRBIT_INDEX);
    return;
  }
  const uint4* xr = reinterpret_cast<const uint4*>(x + src * d);
  const int nv = d >> 3;
  uint4 v[VPT];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + 128 * i;
    v[i] = c < nv ? xr[c] : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      ss = fmaf(f.x, f.x, ss);
      ss = fmaf(f.y, f.y, ss);
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float inv = rsqrtf(((red[0] + red[1]) + (red[2] + red[3])) / (float)d + eps);
  uint4* orow = reinterpret_cast<uint4*>(out + r * d);
  const uint4* gv = reinterpret_cast<const uint4*>(g);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + 128 * i;
    if (c < nv) {
      const uint4 gw = gv ? gv[c] : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);   // bf16 ones
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
      const __nv_bfloat162* hg = reinterpret_cast<const __nv_bfloat162*>(&gw);
      uint4 o;
      __nv_bfloat162* ho = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]), fg = __bfloat1622float2(hg[q]);
        ho[q] = __floats2bfloat162_rn(f.x * inv * fg.x, f.y * inv * fg.y);
      }
      orow[c] = o;
    }
  }
}

cudaError_t launch_rmsnorm(int dt_in, int dt_out, void* out, const void* x, const int32_t* rows,
                           int64_t n_src, const void* g, int64_t n, int d, float eps, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (dt_in == DT_BF16 && dt_out == DT_BF16 && d % 8 == 0 && d <= 128 * 8 * 8) {
    if (d <= 128 * 8 * 4)
      { const cudaError_t e_ = launch_k(k_rmsnorm_reg<4>, dim3((unsigned)n), dim3(128), 0, s, (bf16*)out, (const bf16*)x, rows, n_src, (const bf16*)g, d, eps); if (e_ != cudaSuccess) return e_; }
    else
      { const cudaError_t e_ = launch_k(k_rmsnorm_reg<8>, dim3((unsigned)n), dim3(128), 0, s, (bf16*)out, (const bf16*)x, rows, n_src, (const bf16*)g, d, eps); if (e_ != cudaSuccess) return e_; }
    return cudaGetLastError();
  }
  const int threads = d >= 2048 ? 256 : (d >= 512 ? 64 : 32);
  if (dt_in == DT_BF16 && dt_out == DT_BF16)
    { const cudaError_t e_ = launch_k(k_rmsnorm<bf16, bf16>, dim3((unsigned)n), dim3(threads), 0, s, (bf16*)out, (const bf16*)x, rows,
                                                          n_src, (const bf16*)g, d, eps); if (e_ != cudaSuccess) return e_; }
  else if (dt_in == DT_BF16)
    { const cudaError_t e_ = launch_k(k_rmsnorm<bf16, float>, dim3((unsigned)n), dim3(threads), 0, s, (float*)out, (const bf16*)x, rows,
                                                           n_src, (const bf16*)g, d, eps); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_rmsnorm<float, float>, dim3((unsigned)n), dim3(threads), 0, s, (float*)out, (const float*)x, rows,
                                                            n_src, (const float*)g, d, eps); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ KV deviation
// scores[c] = sum (kn[new_row[c]] - kr[ref_row[c]])^2 (+ V).  One warp per candidate;
// each lane reads 16-byte vectors, partial sums reduced by shuffles (fixed order).  A row
// outside [0, n_new) or [0, n_ref) (bound < 0: unchecked) records ERRBIT_INDEX and the
// candidate's score is not written.
template <typename T>
__global__ void __launch_bounds__(256) k_deviation(const T* __restrict__ kn, const T* __restrict__ vn,
                                                   const T* __restrict__ kr, const T* __restrict__ vr,
                                                   const int32_t* __restrict__ new_row,
                                                   const int32_t* __restrict__ ref_row, int n_cand,
                                                   int64_t n_new, int64_t n_ref, int W, int use_v,
                                                   float* __restrict__ scores) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps_total = (gridDim.x * blockDim.x) >> 5;
  for (int c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < n_cand; c += warps_total) {
    const int64_t rn = new_row ? (int64_t)new_row[c] : c;
    const int64_t rr = ref_row ? (int64_t)ref_row[c] : c;
    if (rn < 0 || rr < 0 || (n_new >= 0 && rn >= n_new) || (n_ref >= 0 && rr >= n_ref)) {   // warp-uniform
      if (lane == 0) atomicOr(&g_err_mem, ERRBIT_INDEX);
      continue;
    }
    float acc = 0.f, accv = 0.f;
    const T* a = kn + rn * W;
    const T* b = kr + rr * W;
    const T* av = vn + rn * W;
    const T* bv = vr + rr * W;
    for (int e = lane * 8; e < W; e += 256) {
      float x[8], y[8], xv[8], yv[8];
      ld8(a + e, x);
      ld8(b + e, y);
      if (use_v) {
        ld8(av + e, xv);
        ld8(bv + e, yv);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float d = x[i] - y[i];
        acc = fmaf(d, d, acc);
      }
      if (use_v) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float d = xv[i] - yv[i];
          accv = fmaf(d, d, accv);
        }
      }
    }
    acc = warp_sum(acc) + warp_sum(accv);
    if (lane == 0) {
      scores[c] = acc;
      if (!isfinite(acc)) atomicOr(&g_err_mem, ERRBIT_NONFINITE);
    }
  }
}

// scores[c] = sum over column tiles t of part[t][c], the per-tile partials the Q/K/V GEMM
// epilogue leaves when it computes the deviation in place.  A block owns 32 candidates: warp
// w sums the partials t = part_lo + w, part_lo + w + 8, ... of its lane's candidate (every
// load coalesced over the 32 candidates, eight warps' loads in flight together), then the
// eight warp sums are added in warp order, so the result does not depend on the launch.
__global__ void __launch_bounds__(256) k_dev_reduce(const float* __restrict__ part, int part_lo, int n_parts,
                                                    int64_t ld, int n_cand, const int32_t* __restrict__ cand_pos,
                                                    float* __restrict__ scores) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float acc = 0.f;
  if (c < n_cand) {
    const int64_t row = cand_pos ? (int64_t)cand_pos[c] : c;
#pragma unroll 4
    for (int t = part_lo + w; t < n_parts; t += 8) acc += part[t * ld + row];
  }
  red[w][lane] = acc;
  __syncthreads();
  if (w == 0 && c < n_cand) {
    float sum = red[0][lane];
#pragma unroll
    for (int j = 1; j < 8; ++j) sum += red[j][lane];
    scores[c] = sum;
    if (!isfinite(sum)) atomicOr(&g_err_mem, ERRBIT_NONFINITE);
  }
}

cudaError_t launch_dev_reduce(const float* part, int part_lo, int n_parts, int64_t ld, int n_cand,
                              const int32_t* cand_pos, float* scores, cudaStream_t s) {
  if (n_cand == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_dev_reduce, dim3((n_cand + 31) / 32), dim3(256), 0, s, part, part_lo, n_parts, ld, n_cand, cand_pos, scores); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// bf16 rows whose width is a multiple of 1024: each lane issues the 16-byte loads of four
// column blocks of all four matrices (16 loads in flight) before the arithmetic.  The sum
// order is fixed (per lane: K then V of each block; then the warp reduction).
__global__ void __launch_bounds__(256) k_deviation_wide(const bf16* __restrict__ kn, const bf16* __restrict__ vn,
                                                        const bf16* __restrict__ kr, const bf16* __restrict__ vr,
                                                        const int32_t* __restrict__ new_row,
                                                        const int32_t* __restrict__ ref_row, int n_cand,
                                                        int64_t n_new, int64_t n_ref, int W, int use_v,
                                                        float* __restrict__ scores) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps_total = (gridDim.x * blockDim.x) >> 5;
  for (int c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < n_cand; c += warps_total) {
    const int64_t rn = new_row ? (int64_t)new_row[c] : c;
    const int64_t rr = ref_row ? (int64_t)ref_row[c] : c;
    if (rn < 0 || rr < 0 || (n_new >= 0 && rn >= n_new) || (n_ref >= 0 && rr >= n_ref)) {   // warp-uniform
      if (lane == 0) atomicOr(&g_err_mem, ERRBIT_INDEX);
      continue;
    }
    const uint4* a = reinterpret_cast<const uint4*>(kn + rn * W);
    const uint4* b = reinterpret_cast<const uint4*>(kr + rr * W);
    const uint4* av = reinterpret_cast<const uint4*>(vn + rn * W);
    const uint4* bv = reinterpret_cast<const uint4*>(vr + rr * W);
    float acc = 0.f, accv = 0.f;
    for (int e = lane; e < (W >> 3); e += 128) {
      uint4 x[4], y[4], xv[4], yv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x[u] = __ldcs(a + e + 32 * u);
        y[u] = __ldcs(b + e + 32 * u);
        if (use_v) {
          xv[u] = __ldcs(av + e + 32 * u);
          yv[u] = __ldcs(bv + e + 32 * u);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&x[u]);
        const __nv_bfloat162* hy = reinterpret_cast<const __nv_bfloat162*>(&y[u]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 fx = __bfloat1622float2(hx[q]), fy = __bfloat1622float2(hy[q]);
          const float d0 = fx.x - fy.x, d1 = fx.y - fy.y;
          acc = fmaf(d0, d0, acc);
          acc = fmaf(d1, d1, acc);
        }
        if (use_v) {
          const __nv_bfloat162* hxv = reinterpret_cast<const __nv_bfloat162*>(&xv[u]);
          const __nv_bfloat162* hyv = reinterpret_cast<const __nv_bfloat162*>(&yv[u]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 fx = __bfloat1622float2(hxv[q]), fy = __bfloat1622float2(hyv[q]);
            const float d0 = fx.x - fy.x, d1 = fx.y - fy.y;
            accv = fmaf(d0, d0, accv);
            accv = fmaf(d1, d1, accv);
          }
        }
      }
    }
    acc = warp_sum(acc) + warp_sum(accv);
    if (lane == 0) {
      scores[c] = acc;
      if (!isfinite(acc)) atomicOr(&g_err_mem, ERRBIT_NONFINITE);
    }
  }
}

cudaError_t launch_deviation(int dt, const void* kn, const void* vn, const void* kr,
                             const void* vr, const int32_t* new_row, const int32_t* ref_row,
                             int n_cand, int64_t n_new, int64_t n_ref, int W, int use_v, float* scores,
                             cudaStream_t s) {
  if (n_cand == 0) return cudaSuccess;
  if (dt == DT_BF16 && W % 1024 == 0) {
    { const cudaError_t e_ = launch_k(k_deviation_wide, dim3(grid_for(k_deviation_wide, (int64_t)n_cand * 32, 256)), dim3(256), 0, s, (const bf16*)kn, (const bf16*)vn, (const bf16*)kr, (const bf16*)vr, new_row, ref_row, n_cand, n_new, n_ref, W, use_v, scores); if (e_ != cudaSuccess) return e_; }
    return cudaGetLastError();
  }
  const unsigned grid = dt == DT_BF16 ? grid_for(k_deviation<bf16>, (int64_t)n_cand * 32, 256)
                                      : grid_for(k_deviation<float>, (int64_t)n_cand * 32, 256);
  if (dt == DT_BF16)
    { const cudaError_t e_ = launch_k(k_deviation<bf16>, dim3(grid), dim3(256), 0, s, (const bf16*)kn, (const bf16*)vn, (const bf16*)kr,
                                           (const bf16*)vr, new_row, ref_row, n_cand, n_new, n_ref, W, use_v,
                                           scores); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_deviation<float>, dim3(grid), dim3(256), 0, s, (const float*)kn, (const float*)vn, (const float*)kr,
                                            (const float*)vr, new_row, ref_row, n_cand, n_new, n_ref, W, use_v,
                                            scores); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ exact top-k
// Scores are finite and >= 0, so their IEEE bit patterns (with -0 folded to +0) order
// them as unsigned integers.  A 4-pass radix select (8 bits per pass) finds the k-th
// largest key T and how many keys equal to T must be taken; a block-wide scan in index
// order then takes every key > T and the lowest-index keys == T, writing the selected
// ordinals in ascending order.  One block of 1024 threads per problem.
__device__ __forceinline__ uint32_t score_key(float s) {
  return s == 0.0f ? 0u : __float_as_uint(s);
}

// exclusive block scan of v (blockDim.x <= 1024); *total receives the block sum
__device__ __forceinline__ int block_excl_scan(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    sh[lane] = t;
  }
  __syncthreads();
  const int base = w ? sh[w - 1] : 0;
  *total = sh[nw - 1];
  __syncthreads();
  return base + x - v;
}

// Up to this many keys are staged in shared memory (64 KB) and every pass reads them there.
constexpr int kTopkSmemKeys = 16384;

// Optional fused selection output (the default row layout): instead of the ordinals, write
// S = (candidate rows of the top-k ordinals, ascending) ++ (forced rows forced_row0 + f) and
// each row's position in the layer's input set (keep: the ordinal, or forced_pos0 + f).
struct SelOut {
  const int32_t* cand_row;   // null: the ordinal is the row
  int32_t forced_row0, forced_pos0;
  int n_forced;
  int32_t* s_out;            // null: plain ordinals to `out`
  int32_t* keep;
};

template <bool SMEM>
__global__ void __launch_bounds__(1024) k_topk(const float* __restrict__ scores, int n, int k,
                                               int32_t* __restrict__ out, const SelOut so) {
  pdl_wait();
  pdl_trigger();
  // the ordinal i taken at position pos of the selection
  auto emit = [&](int pos, int i) {
    if (so.s_out) {
      so.s_out[pos] = so.cand_row ? so.cand_row[i] : i;
      if (so.keep) so.keep[pos] = i;
    } else {
      out[pos] = i;
    }
  };
  if (so.s_out) {
    const int kk = k < n ? k : n;
    for (int f = threadIdx.x; f < so.n_forced; f += blockDim.x) {
      so.s_out[kk + f] = so.forced_row0 + f;
      if (so.keep) so.keep[kk + f] = so.forced_pos0 + f;
    }
  }
  extern __shared__ uint32_t skey[];
  __shared__ int hist[256];
  __shared__ int sh[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int tid = threadIdx.x, bd = blockDim.x;
  // validity check of every score (finite, non-negative); the keys are staged on the way
  bool bad = false;
  for (int i = tid; i < n; i += bd) {
    const float v = scores[i];
    if (!(v >= 0.0f) || isinf(v)) bad = true;
    if (SMEM) skey[i] = score_key(v);
  }
  if (bad) atomicOr(&g_err_mem, ERRBIT_NONFINITE);
  if (k <= 0) return;
  if (k >= n) {
    for (int i = tid; i < n; i += bd) emit(i, i);
    return;
  }
  auto key_at = [&](int i) -> uint32_t { return SMEM ? skey[i] : score_key(scores[i]); };
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += bd) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += bd) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // warp-parallel search, from the top digit down, for the digit holding the
      // remaining-th largest key: lane l owns digits 255-8l .. 248-8l
      const int lane = tid;
      int cnt[8], own = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = hist[255 - 8 * lane - i];
        own += cnt[i];
      }
      int incl = own;   // inclusive prefix over lanes = keys in digits >= this lane's lowest
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - own;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
      if (lane == __ffs(hit) - 1) {
        int cum = excl, dsel = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + cnt[i] >= remaining) {
            dsel = 255 - 8 * lane - i;
            break;
          }
          cum += cnt[i];
        }
        s_prefix = prefix | ((uint32_t)dsel << shift);
        s_remaining = remaining - cum;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
    __syncthreads();
  }
  // every key > T, and the first `remaining` keys == T in index order
  if (SMEM) {
    // one block scan: thread t owns keys [t E, t E + E); counts of keys > T and == T packed
    // in one int (n <= kTopkSmemKeys < 2^16)
    const int E = (n + bd - 1) / bd;
    const int i0 = min(n, tid * E), i1 = min(n, i0 + E);
    int gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = skey[i];
      gt += key > prefix;
      eq += key == prefix;
    }
    int tot;
    const int before = block_excl_scan(gt | (eq << 16), &tot, sh);
    int eq_seen = before >> 16;
    int pos = (before & 0xFFFF) + min(eq_seen, remaining);
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = skey[i];
      if (key > prefix) {
        emit(pos++, i);
      } else if (key == prefix) {
        if (eq_seen < remaining) emit(pos++, i);
        ++eq_seen;
      }
    }
    return;
  }
  int eq_base = 0, out_base = 0;
  for (int i0 = 0; i0 < n; i0 += bd) {
    const int i = i0 + tid;
    const uint32_t key = i < n ? score_key(scores[i]) : 0u;
    const int gt = (i < n) && key > prefix;
    const int eq = (i < n) && key == prefix;
    int eq_tot;
    const int eq_rank = block_excl_scan(eq, &eq_tot, sh);
    const int take = gt || (eq && (eq_base + eq_rank) < remaining);
    int take_tot;
    const int pos = block_excl_scan(take, &take_tot, sh);
    if (take) emit(out_base + pos, i);
    eq_base += eq_tot;
    out_base += take_tot;
  }
}

static cudaError_t topk_launch(const float* scores, int n, int k, int32_t* out_ord, const SelOut& so,
                               cudaStream_t s) {
  if (n <= kTopkSmemKeys) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    bool set = false;
    if (dev >= 0 && dev < 64) {
      std::lock_guard<std::mutex> g(g_mem_mu);
      set = g_topk_attr[dev];
    }
    if (!set) {
      e = cudaFuncSetAttribute(k_topk<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkSmemKeys * 4);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> g(g_mem_mu);
        g_topk_attr[dev] = true;
      }
    }
    { const cudaError_t e_ = launch_k(k_topk<true>, dim3(1), dim3(1024), (size_t)n * 4, s, scores, n, k, out_ord, so); if (e_ != cudaSuccess) return e_; }
  } else {
    { const cudaError_t e_ = launch_k(k_topk<false>, dim3(1), dim3(1024), 0, s, scores, n, k, out_ord, so); if (e_ != cudaSuccess) return e_; }
  }
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* scores, int n, int k, int32_t* out_ord, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return topk_launch(scores, n, k, out_ord, SelOut{nullptr, 0, 0, 0, nullptr, nullptr}, s);
}

cudaError_t launch_topk_sel(const float* scores, int n, int k, const int32_t* cand_row, int32_t forced_row0,
                            int32_t forced_pos0, int n_forced, int32_t* s_out, int32_t* keep_out, cudaStream_t s) {
  if (n == 0 && n_forced == 0) return cudaSuccess;
  return topk_launch(scores, n, k, nullptr, SelOut{cand_row, forced_row0, forced_pos0, n_forced, s_out, keep_out}, s);
}

// out[i] = map[ord[i]] (map null: ord[i])
__global__ void k_map_rows(const int32_t* ord, int k, const int32_t* map, int32_t* out) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < k) out[i] = map ? map[ord[i]] : ord[i];
}

cudaError_t launch_map_rows(const int32_t* ord, int k, const int32_t* map, int32_t* out,
                            cudaStream_t s) {
  if (k == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_map_rows, dim3((k + 255) / 256), dim3(256), 0, s, ord, k, map, out); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// Selected set S = (candidate rows of the top-k ordinals) ++ (forced rows), ascending by
// construction since every forced row lies above every candidate row.  keep_out gives each
// row's position inside the layer's input row set.
__global__ void k_build_sel(const int32_t* ord, int k, const int32_t* cand_row, int32_t forced_row0,
                            int32_t forced_pos0, int n_forced, int32_t* s_out, int32_t* keep_out) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < k) {
    const int o = ord[i];
    s_out[i] = cand_row ? cand_row[o] : o;
    if (keep_out) keep_out[i] = o;
  } else if (i < k + n_forced) {
    const int f = i - k;
    s_out[i] = forced_row0 + f;
    if (keep_out) keep_out[i] = forced_pos0 + f;
  }
}

cudaError_t launch_build_sel(const int32_t* ord, int k, const int32_t* cand_row,
                             int32_t forced_row0, int32_t forced_pos0, int n_forced,
                             int32_t* s_out, int32_t* keep_out, cudaStream_t s) {
  const int n = k + n_forced;
  if (n == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_build_sel, dim3((n + 255) / 256), dim3(256), 0, s, ord, k, cand_row, forced_row0, forced_pos0, n_forced,
                                             s_out, keep_out); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// General row sets (uncached spans anywhere in the request): splits the ascending input
// set rows_in[0..m) (null: 0..m-1) by the forced-row mask into the candidates (cached,
// unforced) and the forced rows, each list ascending with the rows' positions in the input
// set.  One block walks the set in tiles with a block scan; a forced count other than
// n_forced, or a row outside the mask, records ERRBIT_INDEX.
__global__ void __launch_bounds__(1024) k_split_rows(const int32_t* __restrict__ rows_in, int m,
                                                     const uint8_t* __restrict__ mask, int64_t mask_len,
                                                     int n_forced, int32_t* __restrict__ cand_pos,
                                                     int32_t* __restrict__ cand_rows,
                                                     int32_t* __restrict__ forced_pos,
                                                     int32_t* __restrict__ forced_rows) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sh[32];
  int base_f = 0, base_c = 0;
  const int n_cand = m - n_forced;
  for (int t0 = 0; t0 < m; t0 += blockDim.x) {
    const int i = t0 + threadIdx.x;
    int r = -1, f = 0;
    if (i < m) {
      r = rows_in ? rows_in[i] : i;
      if (r < 0 || r >= mask_len) {
        atomicOr(&g_err_mem, ERRBIT_INDEX);
        f = 1;
      } else {
        f = mask[r] != 0;
      }
    }
    int tot;
    const int pf = block_excl_scan(f, &tot, sh);
    if (i < m) {
      if (f) {
        const int o = base_f + pf;
        if (o < n_forced) {
          forced_pos[o] = i;
          forced_rows[o] = r;
        }
      } else {
        const int o = base_c + (i - t0) - pf;
        if (o < n_cand) {
          cand_pos[o] = i;
          cand_rows[o] = r;
        }
      }
    }
    base_f += tot;
    base_c += min((int)blockDim.x, m - t0) - tot;
  }
  if (threadIdx.x == 0 && base_f != n_forced) atomicOr(&g_err_mem, ERRBIT_INDEX);
}

cudaError_t launch_split_rows(const int32_t* rows_in, int m, const uint8_t* mask, int64_t mask_len,
                              int n_forced, int32_t* cand_pos, int32_t* cand_rows, int32_t* forced_pos,
                              int32_t* forced_rows, cudaStream_t s) {
  if (m == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_split_rows, dim3(1), dim3(1024), 0, s, rows_in, m, mask, mask_len, n_forced, cand_pos, cand_rows, forced_pos, forced_rows); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// S = candidate rows of the top-k ordinals merged with the forced rows, ascending; keep_out
// gives each row's position in the layer's input set.  Both lists are ascending and
// disjoint, so an element's output index is its own index plus the number of elements of
// the other list below it (a binary search).
__global__ void k_merge_sel(const int32_t* __restrict__ ord, int k, const int32_t* __restrict__ cand_rows,
                            const int32_t* __restrict__ cand_pos, const int32_t* __restrict__ forced_rows,
                            const int32_t* __restrict__ forced_pos, int nf, int32_t* __restrict__ s_out,
                            int32_t* __restrict__ keep_out) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < k) {
    const int o = ord[i];
    const int r = cand_rows[o];
    int lo = 0, hi = nf;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (forced_rows[mid] < r) lo = mid + 1; else hi = mid;
    }
    s_out[i + lo] = r;
    if (keep_out) keep_out[i + lo] = cand_pos[o];
  } else if (i < k + nf) {
    const int j = i - k;
    const int r = forced_rows[j];
    int lo = 0, hi = k;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (cand_rows[ord[mid]] < r) lo = mid + 1; else hi = mid;
    }
    s_out[j + lo] = r;
    if (keep_out) keep_out[j + lo] = forced_pos[j];
  }
}

cudaError_t launch_merge_sel(const int32_t* ord, int k, const int32_t* cand_rows, const int32_t* cand_pos,
                             const int32_t* forced_rows, const int32_t* forced_pos, int nf, int32_t* s_out,
                             int32_t* keep_out, cudaStream_t s) {
  const int n = k + nf;
  if (n == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_merge_sel, dim3((n + 255) / 256), dim3(256), 0, s, ord, k, cand_rows, cand_pos, forced_rows, forced_pos, nf, s_out, keep_out); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// pos_out[i] = position of rows[i] inside the ascending s_in[0..m_in) (s_in null: rows[i]
// itself, checked < m_in).  A row that is absent records ERRBIT_INDEX and maps to 0.
__global__ void k_rows_to_positions(const int32_t* rows, int k, const int32_t* s_in, int m_in,
                                    int32_t* pos_out) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= k) return;
  const int r = rows[i];
  if (!s_in) {
    if (r < 0 || r >= m_in) {
      atomicOr(&g_err_mem, ERRBIT_INDEX);
      pos_out[i] = 0;
    } else {
      pos_out[i] = r;
    }
    return;
  }
  int lo = 0, hi = m_in;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_in[mid] < r) lo = mid + 1; else hi = mid;
  }
  if (lo < m_in && s_in[lo] == r) {
    pos_out[i] = lo;
  } else {
    atomicOr(&g_err_mem, ERRBIT_INDEX);
    pos_out[i] = 0;
  }
}

cudaError_t launch_rows_to_positions(const int32_t* rows, int k, const int32_t* s_in, int m_in,
                                     int32_t* pos_out, cudaStream_t s) {
  if (k == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_rows_to_positions, dim3((k + 255) / 256), dim3(256), 0, s, rows, k, s_in, m_in, pos_out); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

__global__ void k_iota(int32_t* out, int n, int32_t start) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = start + i;
}

cudaError_t launch_iota(int32_t* out, int n, int32_t start, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_iota, dim3((n + 255) / 256), dim3(256), 0, s, out, n, start); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// kv_row[i] = r * n_tok + s_in[i] for the rows i of request r, [row0[r], row0[r+1]): each
// selected row's place in the requests' caches laid back to back.  A position outside
// [0, n_tok) records ERRBIT_INDEX and maps to -1, which the K/V epilogue does not write.
__global__ void k_batch_kv_rows(const int32_t* __restrict__ s_in, int m_total, int64_t n_tok, const BatchRows b,
                                int32_t* __restrict__ kv_row) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m_total) return;
  int r = 0;
  while (r + 1 < b.n_req && i >= b.row0[r + 1]) ++r;
  const int32_t p = s_in[i];
  if (p < 0 || p >= n_tok) {
    atomicOr(&g_err_mem, ERRBIT_INDEX);
    kv_row[i] = -1;
    return;
  }
  kv_row[i] = (int32_t)(r * n_tok + p);
}

cudaError_t launch_batch_kv_rows(const int32_t* s_in, int m_total, int64_t n_tok, const BatchRows& b,
                                 int32_t* kv_row, cudaStream_t s) {
  if (m_total == 0) return cudaSuccess;
  { const cudaError_t e_ = launch_k(k_batch_kv_rows, dim3((m_total + 255) / 256), dim3(256), 0, s, s_in, m_total, n_tok, b, kv_row); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ SwiGLU (SIMT path)
// out[m][j] = silu(gu[m][j]) * gu[m][F + j]
template <typename T>
__global__ void k_swiglu(T* __restrict__ out, const T* __restrict__ gu, int64_t M, int F) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = M * F;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = t / F, j = t - m * F;
    const float g = to_f(gu[m * 2 * F + j]);
    const float u = to_f(gu[m * 2 * F + F + j]);
    out[t] = from_f<T>(silu_f(g) * u);
  }
}

cudaError_t launch_swiglu(int dt, void* out, const void* gu, int64_t M, int F, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const unsigned grid = dt == DT_BF16 ? grid_for(k_swiglu<bf16>, M * F, 256) : grid_for(k_swiglu<float>, M * F, 256);
  if (dt == DT_BF16)
    { const cudaError_t e_ = launch_k(k_swiglu<bf16>, dim3(grid), dim3(256), 0, s, (bf16*)out, (const bf16*)gu, M, F); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_swiglu<float>, dim3(grid), dim3(256), 0, s, (float*)out, (const float*)gu, M, F); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ lm_head
// argmax with ties to the lowest index: maximise (ordered float bits, ~index) as a u64
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
  return ((unsigned long long)ordered_bits(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, v, o);
    v = y > v ? y : v;
  }
  return v;
}

// logits[v] = hn . w[v]; one warp per vocabulary row, 16-byte weight loads.  Each block
// also leaves the best (logit, lowest index) key of its rows in block_best[blockIdx.x].
template <typename T>
__global__ void __launch_bounds__(256) k_lm_gemv(float* __restrict__ logits, const float* __restrict__ hn,
                                                 const T* __restrict__ w, int V, int d, int rows_per_warp,
                                                 unsigned long long* __restrict__ block_best,
                                                 unsigned long long* span) {
  pdl_wait();
  pdl_trigger();
  span_begin(span);
  __shared__ unsigned long long red[8];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // each warp owns rows_per_warp consecutive rows; the grid is sized so that every warp is
  // resident at once and all of them finish together (no partial last round of rows)
  const int r0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * rows_per_warp;
  const int r1 = min(V, r0 + rows_per_warp);
  unsigned long long best = 0ull;
  // two rows at a time: eight 16-byte weight loads in flight per lane, and each normalised
  // hidden value loaded once for both rows; each row's sum is taken in the same order as
  // one row alone
  for (int r = r0; r < r1; r += 2) {
    const bool two = r + 1 < r1;
    const T* wr0 = w + (int64_t)r * d;
    const T* wr1 = two ? wr0 + d : wr0;
    float acc0[2] = {0.f, 0.f}, acc1[2] = {0.f, 0.f};
    int c = lane * 8;
    for (; c + 768 < d; c += 1024) {
      uint4 raw[2][4][sizeof(T) / 2];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < (int)(sizeof(T) / 2); ++q) {
          raw[0][u][q] = reinterpret_cast<const uint4*>(wr0 + c + 256 * u)[q];
          raw[1][u][q] = reinterpret_cast<const uint4*>(wr1 + c + 256 * u)[q];
        }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float b[8];
        ld8(hn + c + 256 * u, b);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float a[8];
          if constexpr (sizeof(T) == 2) {
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[j][u][0]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(h2[i]);
              a[2 * i] = f.x;
              a[2 * i + 1] = f.y;
            }
          } else {
            const float* f = reinterpret_cast<const float*>(&raw[j][u][0]);
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = f[i];
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (u & 1) acc1[j] = fmaf(a[i], b[i], acc1[j]);
            else acc0[j] = fmaf(a[i], b[i], acc0[j]);
          }
        }
      }
    }
    for (; c < d; c += 256) {
      float a0[8], a1[8], b[8];
      ld8(wr0 + c, a0);
      ld8(wr1 + c, a1);
      ld8(hn + c, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc0[0] = fmaf(a0[i], b[i], acc0[0]);
        acc0[1] = fmaf(a1[i], b[i], acc0[1]);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j == 1 && !two) break;
      const float acc = warp_sum(acc0[j] + acc1[j]);
      if (lane == 0) logits[r + j] = acc;
      const unsigned long long key = argmax_key(acc, r + j);
      best = key > best ? key : best;
    }
  }
  if (lane == 0) red[wid] = best;
  __syncthreads();
  if (wid == 0) {
    unsigned long long b = lane < (int)(blockDim.x >> 5) ? red[lane] : 0ull;
    b = warp_max_u64(b);
    if (lane == 0) block_best[blockIdx.x] = b;
  }
  if (span) {   // uniform; every thread of the block reaches this point
    __syncthreads();
    span_end(span);
  }
}

// 256-thread blocks of the GEMV resident per SM (register-limited)
static int lm_blocks_per_sm(int dt) {
  return dt == DT_BF16 ? resident_blocks(reinterpret_cast<const void*>(k_lm_gemv<bf16>), 256)
                       : resident_blocks(reinterpret_cast<const void*>(k_lm_gemv<float>), 256);
}
// rows per warp: the fewest that cover the vocabulary with the warps that are resident at
// once; the grid then holds just enough warps for that, so every warp runs from the start
// and all of them finish together (no partial last round of rows)
static int lm_rows_per_warp(int V, int dt) {
  const int64_t warps = (int64_t)sm_count() * lm_blocks_per_sm(dt) * 8;
  return (int)std::max<int64_t>(1, (V + warps - 1) / warps);
}
static unsigned lm_grid(int V, int dt) {
  const int rpw = lm_rows_per_warp(V, dt);
  const int64_t warps = (V + rpw - 1) / rpw;
  return (unsigned)std::max<int64_t>(1, (warps + 7) / 8);
}

size_t lm_block_best_count(int V) { return std::max(lm_grid(V, DT_BF16), lm_grid(V, DT_F32)); }
size_t lm_block_count(int V, int dt) { return lm_grid(V, dt); }

cudaError_t launch_lm_gemv(int dt, float* logits, const float* hn, const void* w, int V, int d,
                           unsigned long long* block_best, cudaStream_t s) {
  const unsigned grid = lm_grid(V, dt);
  const int rpw = lm_rows_per_warp(V, dt);
  if (dt == DT_BF16)
    { const cudaError_t e_ = launch_k(k_lm_gemv<bf16>, dim3(grid), dim3(256), 0, s, logits, hn, (const bf16*)w, V, d, rpw, block_best, prof_span_slot()); if (e_ != cudaSuccess) return e_; }
  else
    { const cudaError_t e_ = launch_k(k_lm_gemv<float>, dim3(grid), dim3(256), 0, s, logits, hn, (const float*)w, V, d, rpw, block_best, prof_span_slot()); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// token = index of the largest block key
__global__ void __launch_bounds__(1024) k_argmax_keys(const unsigned long long* __restrict__ keys, int n,
                                                      int32_t* token) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long red[32];
  unsigned long long best = 0ull;
  for (int i = threadIdx.x; i < n; i += blockDim.x) best = keys[i] > best ? keys[i] : best;
  best = warp_max_u64(best);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) red[w] = best;
  __syncthreads();
  if (w == 0) {
    best = lane < (int)(blockDim.x >> 5) ? red[lane] : 0ull;
    best = warp_max_u64(best);
    if (lane == 0) token[0] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
  }
}

cudaError_t launch_argmax_keys(const unsigned long long* keys, int n, int32_t* token, cudaStream_t s) {
  { const cudaError_t e_ = launch_k(k_argmax_keys, dim3(1), dim3(1024), 0, s, keys, n, token); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ allocation-free variant
// Scratch of the deviation/top-k entry point for callers that cannot allocate device memory:
// one fixed array per device, 8 bytes per candidate (fp32 score + int32 ordinal), held for
// the life of the process by every device that loads the library.  Every call shares it.
constexpr int kNoAllocMaxCand = 65536;
static __device__ __align__(256) unsigned char g_noalloc_scratch[(size_t)kNoAllocMaxCand * 8];

int noalloc_max_candidates() { return kNoAllocMaxCand; }

// The array's name is only a host-side stand-in in host code; its device address is looked
// up once per device (with that device current, in the context current then: the primary
// context for callers that use the runtime API) and reused until reset_mem_caches().
static cudaError_t noalloc_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mem_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

// Same kernels as the workspace path; scores (when the caller passes none) and the top-k
// ordinals live in the fixed array.  Both are fully written before they are read, so
// nothing in it has to start at zero.  n_cand <= kNoAllocMaxCand is checked by the caller.
cudaError_t launch_deviation_topk_noalloc(int dt, const void* kn, const void* vn, const void* kr,
                                          const void* vr, const int32_t* new_row,
                                          const int32_t* ref_row, int n_cand, int64_t n_new, int64_t n_ref,
                                          int k, int W, int use_v, float* scores, int32_t* sel,
                                          cudaStream_t s) {
  void* base = nullptr;
  cudaError_t e = noalloc_scratch_address(&base);
  if (e != cudaSuccess) return e;
  float* sc = scores ? scores : static_cast<float*>(base);
  int32_t* ord = reinterpret_cast<int32_t*>(static_cast<char*>(base) + (size_t)kNoAllocMaxCand * 4);
  e = launch_deviation(dt, kn, vn, kr, vr, new_row, ref_row, n_cand, n_new, n_ref, W, use_v, sc, s);
  if (e != cudaSuccess || k <= 0) return e;
  e = launch_topk(sc, n_cand, k, ord, s);
  if (e != cudaSuccess) return e;
  return launch_map_rows(ord, k, ref_row, sel, s);
}

}  // namespace cb
