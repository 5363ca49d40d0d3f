// Tensor-core attention of selected queries over the whole causal KV (bf16, head_dim 64 or
// 128): CacheBlend explainer (0h-n0.github.io/posts/paper-2312-03052) §Selective
// recomputation Step 4 — the selected tokens attend over the entire blended input.
//
// One CTA per (128-query tile, query head).  Per 128-key tile j:
//   S_j = Q K_j^T          tcgen05.mma, A = Q (K-major), B = K_j (K-major), into TMEM
//   P_j = exp2(S_j * log2(e)/sqrt(hd) - m)   softmax warps, row = TMEM lane, key t of a
//                          row visible iff t <= q_pos[row]; P staged to shared memory in
//                          the 128-byte-swizzled K-major layout
//   O  += P_j V_j          tcgen05.mma, A = P (K-major), B = V_j (MN-major), TMEM accum
// The running max m is raised lazily: O (in TMEM) is rescaled only when a row's max grows by
// more than 2^8, so most tiles never touch O.  S is double-buffered in TMEM so the MMA warp
// computes S_{j+1} while the softmax warps work on S_j; K/V tiles stream through a 2-stage
// TMA ring.  Warp roles: 0 = TMA producer, 1 = TMEM allocator + MMA issuer, 2..5 = softmax
// and epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
#include <cuda.h>
#include <math.h>

#include "cb_common.cuh"
#include "cb_internal.h"
#include "cb_tc.cuh"

namespace cb {

static __device__ uint32_t g_err_attn_tc;

uint32_t take_error_attn_tc() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_attn_tc, sizeof(v)) != cudaSuccess) return ERRBIT_INDEX;
  cudaMemcpyToSymbol(g_err_attn_tc, &z, sizeof(z));
  return v;
}

namespace {

constexpr int BM = 128;              // queries per CTA
constexpr int BN = 128;              // keys per tile
constexpr int SLAB = 128 * 128;      // bytes of one [128 rows x 64 bf16] swizzled slab
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;  // S0 | S1 | O
constexpr uint32_t TM_S0 = 0, TM_O = 256;
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
struct Layout {
  static constexpr int NSLAB = HD / 64;
  static constexpr int Q_BYTES = NSLAB * SLAB;
  static constexpr int KV_BYTES = NSLAB * SLAB;
  static constexpr int P_BYTES = 2 * SLAB;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;           // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;      // 2 stages
  static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int BYTES = OFF_BAR + 256;
  // one CTA per SM: it owns all 512 TMEM columns
  static constexpr int SMEM = (BYTES + 1024) > 120 * 1024 ? (BYTES + 1024) : 120 * 1024;
};

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const int32_t* __restrict__ q_pos, int M,
              int64_t n_kv, int H, int Hkv, bf16* __restrict__ out, float scale_log2) {
  using L = Layout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* sQ = base + L::OFF_Q;
  uint8_t* sK = base + L::OFF_K;
  uint8_t* sV = base + L::OFF_V;
  uint8_t* sP = base + L::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* v_full = bars + 3;     // [2]
  uint64_t* kv_empty = bars + 5;   // [2]
  uint64_t* s_full = bars + 7;     // [2]
  uint64_t* s_free = bars + 9;     // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* pv_done = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);
  int* s_qmax = reinterpret_cast<int*>(bars + 14);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = gridDim.x - 1 - blockIdx.x;      // the longest (latest) query tiles first
  const int h = blockIdx.y;
  const int g = h / (H / Hkv);
  const int m0 = qt * BM;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&k_full[i], 1);
      tc::mbar_init(&v_full[i], 1);
      tc::mbar_init(&kv_empty[i], 1);
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&s_free[i], 4);
    }
    tc::mbar_init(p_full, 4);
    tc::mbar_init(pv_done, 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmQ);
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    // furthest key any query of this tile may see
    int mx = 0;
    for (int i = lane; i < BM; i += 32) {
      const int m = m0 + i;
      if (m < M) {
        int p = q_pos[m];
        if (p < 0 || p >= n_kv) {
          atomicOr(&g_err_attn_tc, ERRBIT_INDEX);
          p = p < 0 ? 0 : (int)(n_kv - 1);
        }
        mx = p > mx ? p : mx;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int y = __shfl_xor_sync(0xffffffffu, mx, o);
      mx = y > mx ? y : mx;
    }
    if (lane == 0) *s_qmax = mx;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int T = *s_qmax / BN + 1;   // key tiles to visit

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    tc::mbar_expect_tx(q_full, L::Q_BYTES);
    for (int s = 0; s < L::NSLAB; ++s) tc::tma_load_2d(sQ + s * SLAB, &tmQ, q_full, h * HD + 64 * s, m0);
    for (int j = 0; j < T; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!tc::mbar_wait(&kv_empty[st], ph ^ 1)) {
        atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
        break;
      }
      tc::mbar_expect_tx(&k_full[st], L::KV_BYTES);
      for (int s = 0; s < L::NSLAB; ++s)
        tc::tma_load_2d(sK + st * L::KV_BYTES + s * SLAB, &tmK, &k_full[st], g * HD + 64 * s, j * BN);
      tc::mbar_expect_tx(&v_full[st], L::KV_BYTES);
      for (int s = 0; s < L::NSLAB; ++s)
        tc::tma_load_2d(sV + st * L::KV_BYTES + s * SLAB, &tmV, &v_full[st], g * HD + 64 * s, j * BN);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(BM, HD, true);
    bool ok = tc::mbar_wait(q_full, 0);
    for (int j = 0; ok && j <= T; ++j) {
      if (j < T) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!tc::mbar_wait(&k_full[st], ph) || !tc::mbar_wait(&s_free[st], ph ^ 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k & 3) * 32;
          const uint64_t a = tc::desc_sw128(tc::smem_u32(sQ + (k >> 2) * SLAB) + off);
          const uint64_t b = tc::desc_sw128(tc::smem_u32(sK + st * L::KV_BYTES + (k >> 2) * SLAB) + off);
          tc::mma_bf16(tmem + TM_S0 + st * BN, a, b, idesc_s, k > 0);
        }
        tc::mma_commit(&s_full[st]);
      }
      if (j >= 1) {
        const int jj = j - 1;
        const int st = jj & 1;
        if (!tc::mbar_wait(p_full, jj & 1) || !tc::mbar_wait(&v_full[st], (jj >> 1) & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t a = tc::desc_sw128(tc::smem_u32(sP + (k >> 2) * SLAB) + (k & 3) * 32);
          const uint64_t b = tc::desc_sw128_mn(tc::smem_u32(sV + st * L::KV_BYTES) + k * 16 * 128, SLAB);
          tc::mma_bf16(tmem + TM_O, a, b, idesc_o, (jj > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit(pv_done);
        tc::mma_commit(&kv_empty[st]);
      }
    }
    if (!ok) atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int lane_base = (warp & 3) * 32;
    const int r = lane_base + lane;
    const int m = m0 + r;
    int qp = 0;
    if (m < M) {
      qp = q_pos[m];
      qp = qp < 0 ? 0 : (qp >= n_kv ? (int)(n_kv - 1) : qp);
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>(lane_base) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    uint8_t* prow = sP + r * 128;
    for (int j = 0; j < T; ++j) {
      const int sb = j & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&s_full[sb], (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t ts = trow + TM_S0 + sb * BN;
      const int key0 = j * BN;
      // pass 1: row max of the visible scores (log2 units)
      float mt = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tc::tmem_ld16(ts + c * 16, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x = (key0 + c * 16 + i <= qp) ? v[i] * scale_log2 : -INFINITY;
          mt = fmaxf(mt, x);
        }
      }
      // P buffer free and O stable once the previous P.V has completed
      if (j >= 1) {
        if (!__all_sync(0xffffffffu, tc::mbar_wait(pv_done, (j - 1) & 1))) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
      }
      const float m_new = fmaxf(m_used, mt);
      if (j == 0) {
        m_used = m_new;
      } else {
        const bool need = m_new > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? tc::ex2_approx(m_used - m_new) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < HD / 16; ++c) {
            float o[16];
            tc::tmem_ld16(trow + TM_O + c * 16, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tc::tmem_st16(trow + TM_O + c * 16, o);
          }
          l *= alpha;
          if (need) m_used = m_new;
        }
      }
      // pass 2: P = exp2(x - m_used) in bf16, row sum of the rounded values, swizzled store
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tc::tmem_ld16(ts + c * 16, v);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int k0 = key0 + c * 16 + 2 * i;
          const float p0 = (k0 <= qp) ? tc::ex2_approx(v[2 * i] * scale_log2 - m_used) : 0.f;
          const float p1 = (k0 + 1 <= qp) ? tc::ex2_approx(v[2 * i + 1] * scale_log2 - m_used) : 0.f;
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
          const float2 back = __bfloat1622float2(b2);
          l += back.x + back.y;
          pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        // keys c*16 .. c*16+15 are 16-byte chunks 2c and 2c+1 of the row (slab = chunk / 8)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int chunk = 2 * c + h2;
          const int slab = chunk >> 3, cc = chunk & 7;
          uint4* dst = reinterpret_cast<uint4*>(prow + slab * SLAB + ((cc ^ (r & 7)) << 4));
          *dst = make_uint4(pk[4 * h2], pk[4 * h2 + 1], pk[4 * h2 + 2], pk[4 * h2 + 3]);
        }
      }
      tc::tc_fence_before();
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&s_free[sb]);
        tc::mbar_arrive(p_full);
      }
    }
    if (ok && __all_sync(0xffffffffu, tc::mbar_wait(pv_done, (T - 1) & 1))) {
      tc::tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      bf16* orow = out + (int64_t)m * H * HD + (int64_t)h * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 16; ++c) {
        float o[16];
        tc::tmem_ld16(trow + TM_O + c * 16, o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] *= inv;
        if (m < M) {
          st8(orow + c * 16, o);
          st8(orow + c * 16 + 8, o + 8);
        }
      }
    } else if (lane == 0) {
      atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [rows, cols] bf16, row stride ld elements, box 128 rows x 64 columns, 128-byte swizzle
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
cudaError_t launch_hd(const void* q, const int32_t* q_pos, int M, const void* kc, const void* vc, int64_t n_kv,
                      int H, int Hkv, void* out, cudaStream_t s) {
  using Ly = Layout<HD>;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, M, (int64_t)H * HD, (int64_t)H * HD) ||
      !make_map(&tk, kc, n_kv, (int64_t)Hkv * HD, (int64_t)Hkv * HD) ||
      !make_map(&tv, vc, n_kv, (int64_t)Hkv * HD, (int64_t)Hkv * HD))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  dim3 grid((M + BM - 1) / BM, H);
  k_attn_tc<HD><<<grid, THREADS, Ly::SMEM, s>>>(tq, tk, tv, q_pos, M, n_kv, H, Hkv, static_cast<bf16*>(out),
                                                scale_log2);
  return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(int hd) { return hd == 64 || hd == 128; }

cudaError_t launch_attention_tc(const void* q, const int32_t* q_pos, int M, const void* kc, const void* vc,
                                int64_t n_kv, int H, int Hkv, int hd, void* out, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  if (((uintptr_t)q & 15) || ((uintptr_t)kc & 15) || ((uintptr_t)vc & 15)) return cudaErrorInvalidValue;
  if (hd == 128) return launch_hd<128>(q, q_pos, M, kc, vc, n_kv, H, Hkv, out, s);
  if (hd == 64) return launch_hd<64>(q, q_pos, M, kc, vc, n_kv, H, Hkv, out, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
