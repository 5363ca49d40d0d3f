// bf16 GEMM on the 5th-generation tensor cores: TMA-fed shared-memory pipeline, tcgen05.mma
// into a TMEM accumulator, fused epilogues (RoPE + KV scatter, residual add, SwiGLU, the
// check layer's KV deviation, and the RMSNorm row scale / row sums of squares of the folded
// norms).
//
//   acc[m][n] = sum_k A[m][k] * B[n][k]      A: activations [M, K], B: weight rows [N, K]
//
// Persistent: one CTA per SM walks 128 x BN output tiles (BN 256, 224, 208 or 192 chosen per
// launch; SwiGLU: BN/2 gate + BN/2 up columns -> BN/2 outputs), K consumed in 64-element
// (128-byte) slabs through a 4- or 5-stage ring; two TMEM accumulators let the epilogue of one
// tile overlap the next tile's MMAs.  The CTA-pair variant below computes 256 x BN tiles on two
// SMs with tcgen05.mma.cta_group::2.
// Warp roles:
//   warp 0 lane 0 : TMA producer     warp 1 : TMEM allocator; the whole warp runs the MMA
//                                             issue loop, its elected lane issues
//   warps 2..9    : epilogue; warp w reads the 32 TMEM lanes (rows) of quadrant w % 4 and
//                   one half of the accumulator columns, so two warps share each row band.
#include <cuda.h>

#include <cstdlib>
#include <mutex>

#include "cb_common.cuh"
#include "cb_epilogue.cuh"
#include "cb_internal.h"
#include "cb_tc.cuh"

namespace cb {

static __device__ uint32_t g_err_tc;

uint32_t take_error_gemm_tc() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(v)) != cudaSuccess) return ERRBIT_INDEX;
  cudaMemcpyToSymbol(g_err_tc, &z, sizeof(z));
  return v;
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;   // two accumulators of up to 256 columns, 256 apart

// Tile width BN (accumulator columns): 256, or 224 / 192 where the narrower tile needs fewer
// waves over the SMs (a 512-tile GEMM is 3.37 waves of 152 SMs at 256 columns, exactly 4 at
// 224).  A narrower tile leaves room for a fifth ring stage.
template <int BN>
struct TileCfg {
  static_assert(BN % 16 == 0 && BN <= 256, "the epilogue takes 16-column chunks");
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGES = BN == 256 ? 4 : 5;
  static constexpr int SMEM_BYTES = STAGES * (A_BYTES + B_BYTES) + 1024 /*align slack*/ + 256 /*barriers*/;
};

// Fused RMSNorm: row m's scale 1/rms from the partial sums of squares its producer left
// (1 without them).  Read before the epilogue waits for its accumulator, so the loads are
// hidden under the tile's main loop; eight are in flight at a time, summed in a fixed order.
__device__ __forceinline__ float row_scale(const GemmDesc& g, int m) {
  const EpiParams& p = g.epi;
  if (p.rs_in == nullptr || m >= g.M) return 1.f;
  const int64_t sm = p.rs_row ? (int64_t)p.rs_row[m] : (int64_t)m;
  if (sm < 0 || sm >= p.rs_ld) {
    atomicOr(&g_err_tc, ERRBIT_INDEX);
    return 1.f;
  }
  float sum = 0.f;
  for (int p0 = 0; p0 < p.rs_parts; p0 += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = p0 + i < p.rs_parts ? p.rs_in[(int64_t)(p0 + i) * p.rs_ld + sm] : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += v[i];
  }
  return rsqrtf(sum * p.rs_inv_d + p.rs_eps);
}

// Side inputs of the plain epilogue, per 16-column chunk: the residual row's 16 values (two
// 16-byte words) or the RoPE cos/sin of the row's position for the chunk's 8 pairs (four
// words).  They are loaded a few chunks ahead of their use, the first ones before the
// accumulator is ready, so the loads' latency overlaps the tile's main loop instead of
// following each TMEM read.
template <int WORDS, int AHEAD>
struct SideRing {
  uint4 w[AHEAD][WORDS];
  __device__ __forceinline__ void load(int slot, const uint4* src) {
    if (src) {
#pragma unroll
      for (int i = 0; i < WORDS; ++i) w[slot][i] = __ldg(src + i);
    }
  }
};

// Epilogue of one output tile for one epilogue warp: this lane's accumulator row m (TMEM row
// band at trow), the warp's half of the tile's columns [n0, n0 + BN); rs scales the row
// (fused RMSNorm, see row_scale).  The loads that do not depend on the accumulator are
// issued first; wait_acc() then waits for it (false: the wait gave up, nothing is written).
template <int BN, typename WaitFn>
__device__ __forceinline__ bool epilogue_tile(const GemmDesc& g, int m, int n0, int half, uint32_t trow,
                                              int swiglu, float rs, WaitFn wait_acc) {
  constexpr int CH = BN / 32;              // 16-column chunks per warp
  const bool scaled = g.epi.rs_in != nullptr;
  const EpiParams& p = g.epi;
  if (!swiglu && p.dev_part != nullptr) {
    // K/V columns with the deviation against the cached row: the cached values of the
    // chunk DEV_AHEAD further on are loaded while this chunk is processed
    int64_t rr = -1;
    if (m < g.M) {
      rr = p.ref_row ? (int64_t)p.ref_row[m] : (int64_t)m;
      if (rr < 0 || rr >= p.ref_rows) {
        atomicOr(&g_err_tc, ERRBIT_INDEX);
        rr = -1;
      }
    }
    auto ref_ptr = [&](int c) -> const uint4* {
      const int n = n0 + (half * CH + c) * 16;
      if (rr < 0 || n >= g.N) return nullptr;
      const int gc = p.col0 + n;
      if (gc < p.q_cols) return nullptr;
      const bool is_v = gc >= p.q_cols + p.kv_cols;
      if (is_v && !p.dev_use_v) return nullptr;
      return reinterpret_cast<const uint4*>(static_cast<const bf16*>(is_v ? p.v_ref : p.k_ref) + rr * p.ldkv +
                                            (gc - p.q_cols - (is_v ? p.kv_cols : 0)));
    };
    constexpr int DEV_AHEAD = 4;
    SideRing<2, DEV_AHEAD> ring;
#pragma unroll
    for (int c = 0; c < DEV_AHEAD; ++c) ring.load(c, ref_ptr(c));
    if (!wait_acc()) return false;
    float dsum = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      float v[16];
      tc::tmem_ld16(trow + (half * CH + c) * 16, v);
      if (scaled) {
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] *= rs;
      }
      const int n = n0 + (half * CH + c) * 16;
      if (m < g.M && n < g.N) {
        if (!epi_apply<bf16, 16>(p, m, n, v)) atomicOr(&g_err_tc, ERRBIT_INDEX);
      }
      if (ref_ptr(c)) dsum += sq_dev16(v, ring.w[c % DEV_AHEAD]);
      if (c + DEV_AHEAD < CH) ring.load(c % DEV_AHEAD, ref_ptr(c + DEV_AHEAD));
    }
    if (m < g.M) p.dev_part[((int64_t)(n0 / BN) * 2 + half) * p.dev_ld + m] = dsum;
    return true;
  }
  if (swiglu) {
    if (!wait_acc()) return false;
    for (int c = half * (CH / 2); c < (half + 1) * (CH / 2); ++c) {
      float gt[16], up[16];
      tc::tmem_ld16(trow + c * 16, gt);
      tc::tmem_ld16(trow + BN / 2 + c * 16, up);
      if (scaled) {
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          gt[q] *= rs;
          up[q] *= rs;
        }
      }
      const int j = n0 + c * 16;
      if (m < g.M && j < g.N) {
#pragma unroll
        for (int q = 0; q < 16; ++q) gt[q] = silu_f(gt[q]) * up[q];
        st_vec<bf16, 16>(static_cast<bf16*>(p.out) + (int64_t)m * p.ldo + j, gt);
      }
    }
    return true;
  }
  // the two warps of a row band split the tile's 16-column chunks (7 + 6 at 208 columns)
  constexpr int NCH = BN / 16, H0 = (NCH + 1) / 2;
  const int c_lo = half ? H0 : 0, c_hi = half ? NCH : H0;
  if (p.kind == EPI_RESID) {
    // residual add (and, for the next layer's norm, the squares of the values as stored)
    const int64_t rr = m < g.M ? (p.resid_row ? (int64_t)p.resid_row[m] : (int64_t)m) : -1;
    const bool row_ok = m < g.M && rr >= 0 && (p.resid_rows < 0 || rr < p.resid_rows);
    if (m < g.M && !row_ok) atomicOr(&g_err_tc, ERRBIT_INDEX);
    const bf16* rrow = row_ok ? static_cast<const bf16*>(p.resid) + rr * p.ldr : nullptr;
    const bool vec = rrow != nullptr && ((reinterpret_cast<uintptr_t>(rrow + n0) & 15) == 0);
    SideRing<2, 2> ring;
    auto src = [&](int c) -> const uint4* {
      const int n = n0 + c * 16;
      return (vec && c < c_hi && n < g.N) ? reinterpret_cast<const uint4*>(rrow + n) : nullptr;
    };
    ring.load(0, src(c_lo));
    ring.load(1, src(c_lo + 1));
    if (!wait_acc()) return false;
    float ssq = 0.f;
    // chunks in pairs, so ring slot = chunk parity at compile time with two chunk bodies of code;
    // chunk c + 2's side input is requested while chunk c is processed
    for (int c2 = c_lo; c2 < c_hi; c2 += 2) {
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int c = c2 + a;
        if (c >= c_hi) break;
        float v[16];
        tc::tmem_ld16(trow + c * 16, v);
        if (scaled) {
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] *= rs;
        }
        const int n = n0 + c * 16;
        if (row_ok && n < g.N) {
          float r[16];
          if (vec) {
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(ring.w[a]);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float2 f = __bfloat1622float2(h2[q]);
              r[2 * q] = f.x;
              r[2 * q + 1] = f.y;
            }
          } else {
            ld_vec<bf16, 16>(rrow + n, r);
          }
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] += r[q];
          if (p.ssq_out != nullptr) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float b = __bfloat162float(__float2bfloat16_rn(v[q]));
              ssq = fmaf(b, b, ssq);
            }
          }
          st_vec<bf16, 16>(static_cast<bf16*>(p.out) + (int64_t)m * p.ldo + n, v);
        }
        ring.load(a, src(c + 2));
      }
    }
    if (p.ssq_out != nullptr && m < g.M) p.ssq_out[((int64_t)(n0 / BN) * 2 + half) * p.ssq_ld + m] = ssq;
    return true;
  }
  if (p.kind == EPI_QKV) {
    // RoPE on Q and K columns at the row's position, then Q / K / V stores (K and V into the
    // rows kv_row names, when given)
    const int hhalf = p.hd >> 1;
    const int n_lo = n0 + c_lo * 16, n_hi = min(n0 + c_hi * 16, g.N);   // this warp's columns
    const bool rot = n_lo < n_hi && p.col0 + n_lo < p.q_cols + p.kv_cols;   // some chunk is rotated
    const bool has_kv = n_lo < n_hi && p.col0 + n_hi > p.q_cols;              // some chunk is K or V
    bool pos_ok = m < g.M, kv_ok = m < g.M;
    int pos = 0;
    int64_t kr = 0;
    if (m < g.M && rot) {
      pos = p.pos[m];
      pos_ok = pos >= 0 && pos < p.max_pos;
    }
    if (m < g.M && has_kv) {
      kr = p.kv_row ? (int64_t)p.kv_row[m] : (int64_t)m;
      kv_ok = kr >= 0 && (p.kv_bound < 0 || kr < p.kv_bound);
    }
    if (m < g.M && (!pos_ok || !kv_ok)) atomicOr(&g_err_tc, ERRBIT_INDEX);
    const float2* cs_row =
        pos_ok && rot ? reinterpret_cast<const float2*>(p.rope) + (int64_t)pos * hhalf : nullptr;
    const bool vec = cs_row != nullptr && ((reinterpret_cast<uintptr_t>(cs_row) & 15) == 0) && (hhalf % 2) == 0;
    SideRing<4, 2> ring;
    auto src = [&](int c) -> const uint4* {
      const int n = n0 + c * 16, gc = p.col0 + n;
      if (!vec || c >= c_hi || n >= g.N || gc >= p.q_cols + p.kv_cols) return nullptr;
      const int seg = gc < p.q_cols ? gc : gc - p.q_cols;
      return reinterpret_cast<const uint4*>(cs_row + ((seg % p.hd) >> 1));
    };
    ring.load(0, src(c_lo));
    ring.load(1, src(c_lo + 1));
    if (!wait_acc()) return false;
    for (int c2 = c_lo; c2 < c_hi; c2 += 2) {   // in pairs: ring slot = chunk parity, as above
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int c = c2 + a;
        if (c >= c_hi) break;
        float v[16];
        tc::tmem_ld16(trow + c * 16, v);
        if (scaled) {
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] *= rs;
        }
        const int n = n0 + c * 16;
        const int gc = p.col0 + n;
        const bool rotated = gc < p.q_cols + p.kv_cols;
        if (m < g.M && n < g.N && (!rotated || pos_ok) && (gc < p.q_cols || kv_ok)) {
          if (rotated) {
            const int seg = gc < p.q_cols ? gc : gc - p.q_cols;
            const float2* cs = vec ? reinterpret_cast<const float2*>(ring.w[a]) : cs_row + ((seg % p.hd) >> 1);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float2 t = cs[q];
              const float x0 = v[2 * q], x1 = v[2 * q + 1];
              v[2 * q] = x0 * t.x - x1 * t.y;
              v[2 * q + 1] = x0 * t.y + x1 * t.x;
            }
          }
          if (gc < p.q_cols)
            st_vec<bf16, 16>(static_cast<bf16*>(p.q) + (int64_t)m * p.ldq + gc, v);
          else if (gc < p.q_cols + p.kv_cols)
            st_vec<bf16, 16>(static_cast<bf16*>(p.k) + kr * p.ldkv + (gc - p.q_cols), v);
          else
            st_vec<bf16, 16>(static_cast<bf16*>(p.v) + kr * p.ldkv + (gc - p.q_cols - p.kv_cols), v);
        }
        ring.load(a, src(c + 2));
      }
    }
    return true;
  }
  // plain store
  if (!wait_acc()) return false;
  for (int c = c_lo; c < c_hi; ++c) {
    float v[16];
    tc::tmem_ld16(trow + c * 16, v);
    if (scaled) {
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] *= rs;
    }
    const int n = n0 + c * 16;
    if (m < g.M && n < g.N) {
      if (!epi_apply<bf16, 16>(p, m, n, v)) atomicOr(&g_err_tc, ERRBIT_INDEX);
    }
  }
  return true;
}

template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
              const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
              const GemmDesc g0, const GemmDesc g1, int n_prob, int swiglu, unsigned long long* span) {
  constexpr int STAGES = TileCfg<BN>::STAGES;
  constexpr int B_BYTES = TileCfg<BN>::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the 128-byte-swizzled tiles
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* smA = base;
  uint8_t* smB = base + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + STAGES * (A_BYTES + B_BYTES));
  uint64_t* full = bars;                     // [STAGES] TMA -> MMA
  uint64_t* empty = bars + STAGES;           // [STAGES] MMA -> TMA
  uint64_t* acc_full = bars + 2 * STAGES;    // [2] MMA -> epilogue
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2] epilogue -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // one or two independent problems share the launch: problem 0's tiles come first, then
  // problem 1's, so a short second GEMM fills the first one's partial last wave
  const int out_cols = swiglu ? BN / 2 : BN;
  const int num_m0 = (g0.M + BM - 1) / BM;
  const int t0 = num_m0 * ((g0.N + out_cols - 1) / out_cols);
  const int num_m1 = n_prob > 1 ? (g1.M + BM - 1) / BM : 1;
  const int total = t0 + (n_prob > 1 ? num_m1 * ((g1.N + out_cols - 1) / out_cols) : 0);
  const int kb0 = (g0.K + BK - 1) / BK, kb1 = n_prob > 1 ? (g1.K + BK - 1) / BK : kb0;
  // tile t -> problem, first row and first output column (M-fastest inside a problem)
  auto locate = [&](int t, int& pr, int& m0, int& n0) {
    pr = t >= t0;
    const int u = pr ? t - t0 : t;
    const int nm = pr ? num_m1 : num_m0;
    m0 = (u % nm) * BM;
    n0 = (u / nm) * out_cols;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], EPI_WARPS);
    }
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmA0);
    tc::tma_prefetch_desc(&tmB0);
    if (n_prob > 1) {
      tc::tma_prefetch_desc(&tmA1);
      tc::tma_prefetch_desc(&tmB1);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the prologue above overlaps the previous kernel's tail; inputs are read only from here
  pdl_wait();
  pdl_trigger();
  span_begin(span);

  // Tiles are visited M-fastest: the CTAs in flight share a few weight tiles and the whole
  // (small) activation matrix, so both stay in L2 and each is read from HBM about once.
  if (warp == 0 && lane == 0) {
    // ---------------- producer
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
      int pr, m0, n0;
      locate(t, pr, m0, n0);
      const CUtensorMap* tmA = pr ? &tmA1 : &tmA0;
      const CUtensorMap* tmB = pr ? &tmB1 : &tmB0;
      const int KB = pr ? kb1 : kb0;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&empty[s], ph ^ 1)) {
          atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
          ok = false;
          break;
        }
        tc::mbar_expect_tx(&full[s], A_BYTES + B_BYTES);
        tc::tma_load_2d(smA + s * A_BYTES, tmA, &full[s], kb * BK, m0);
        if (swiglu) {
          tc::tma_load_2d(smB + s * B_BYTES, tmB, &full[s], kb * BK, n0);
          tc::tma_load_2d(smB + s * B_BYTES + B_BYTES / 2, tmB, &full[s], kb * BK, (int)g0.b_up_row + n0);
        } else {
          tc::tma_load_2d(smB + s * B_BYTES, tmB, &full[s], kb * BK, n0);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (warp 1; the elected lane issues, all lanes wait, so the
    // loop stays warp-uniform): accumulator b = local tile index & 1
    constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
    // stage-0 descriptors; the address field (bytes >> 4) advances by plain addition
    const uint64_t a_desc0 = tc::desc_sw128(tc::smem_u32(smA));
    const uint64_t b_desc0 = tc::desc_sw128(tc::smem_u32(smB));
    uint32_t it = 0, i = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++i) {
      const uint32_t b = i & 1;
      const int KB = t >= t0 ? kb1 : kb0;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&acc_empty[b], ((i >> 1) & 1) ^ 1))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t d_tmem = tmem + b * 256;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&full[s], ph))) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        if (tc::elect_one()) {
          const uint64_t a_desc = a_desc0 + (uint64_t)((s * A_BYTES) >> 4);
          const uint64_t b_desc = b_desc0 + (uint64_t)((s * B_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // advance 16 bf16 = 32 bytes along K inside the swizzled 128-byte row
            tc::mma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, (kb | k) != 0);
          }
          tc::mma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (ok) {
        if (tc::elect_one()) tc::mma_commit(&acc_full[b]);
        __syncwarp();
      }
    }
    if (!ok && lane == 0) atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
  } else if (warp >= 2) {
    // ---------------- epilogue: drains accumulator b while the MMAs fill the other one
    const int lane_base = (warp & 3) * 32;
    const int half = (warp - 2) >> 2;        // which half of the accumulator columns
    uint32_t i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const uint32_t b = i & 1;
      int pr, m0, n0;
      locate(t, pr, m0, n0);
      const GemmDesc& g = pr ? g1 : g0;
      const int m = m0 + lane_base + lane;
      const float rs = row_scale(g, m);
      const uint32_t trow = tmem + b * 256 + (static_cast<uint32_t>(lane_base) << 16);
      // every lane waits, then the warp re-converges before the .sync.aligned TMEM loads
      const bool done = epilogue_tile<BN>(g, m, n0, half, trow, swiglu, rs, [&] {
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (i >> 1) & 1))) return false;
        tc::tc_fence_after();
        return true;
      });
      if (!done) {
        if (lane == 0) atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
        break;
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  span_end(span);
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- two-SM variant: 256 x BN tiles computed by a CTA pair ------------------------------
// A cluster of two CTAs on two SMs shares each tile: CTA r stages A rows [m0 + 128 r, +128)
// and half of the B tile (rows n0 + r BN/2; for SwiGLU CTA 0 the gate rows, CTA 1 the up
// rows) and receives accumulator rows [m0 + 128 r, +128) in its own TMEM; the even CTA issues
// tcgen05.mma.cta_group::2 on both CTAs' stages.  Each SM thus stages and feeds its tensor
// core half of B per tile instead of all of it.  Both CTAs' loads complete on the even CTA's
// "full" barrier; the MMA completions arrive on both CTAs' "empty" and "accumulator full"
// barriers; both CTAs' epilogue warps release an accumulator on the even CTA's barrier.
template <int BN>
struct PairCfg {
  static_assert(BN == 256 || BN == 224 || BN == 192, "pair tiles are 256, 224 or 192 columns wide");
  static constexpr int B_BYTES = (BN / 2) * BK * 2;   // this CTA's half of the B tile
  static constexpr int STAGES = BN == 256 ? 6 : 7;
  static constexpr int SMEM_BYTES = STAGES * (A_BYTES + B_BYTES) + 1024 /*align slack*/ + 256 /*barriers*/;
};
constexpr int PAIR_BM = 2 * BM;

template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_tc_pair(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const GemmDesc g0, const GemmDesc g1, int n_prob, int swiglu, unsigned long long* span) {
  constexpr int STAGES = PairCfg<BN>::STAGES;
  constexpr int B_BYTES = PairCfg<BN>::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  // the same 1024-byte aligned layout in both CTAs (the pair MMA addresses both by offset)
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* smA = base;
  uint8_t* smB = base + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + STAGES * (A_BYTES + B_BYTES));
  uint64_t* full = bars;                        // [STAGES] both CTAs' TMA -> MMA (even CTA's copy used)
  uint64_t* empty = bars + STAGES;              // [STAGES] MMA -> this CTA's TMA
  uint64_t* acc_full = bars + 2 * STAGES;       // [2] MMA -> this CTA's epilogue
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2] both CTAs' epilogues -> MMA (even CTA's copy used)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const int pair = (int)tc::cluster_id_x(), n_pairs = (int)tc::n_clusters_x();
  const int out_cols = swiglu ? BN / 2 : BN;
  const int num_m0 = (g0.M + PAIR_BM - 1) / PAIR_BM;
  const int t0 = num_m0 * ((g0.N + out_cols - 1) / out_cols);
  const int num_m1 = n_prob > 1 ? (g1.M + PAIR_BM - 1) / PAIR_BM : 1;
  const int total = t0 + (n_prob > 1 ? num_m1 * ((g1.N + out_cols - 1) / out_cols) : 0);
  const int kb0 = (g0.K + BK - 1) / BK, kb1 = n_prob > 1 ? (g1.K + BK - 1) / BK : kb0;
  auto locate = [&](int t, int& pr, int& m0, int& n0) {
    pr = t >= t0;
    const int u = pr ? t - t0 : t;
    const int nm = pr ? num_m1 : num_m0;
    m0 = (u % nm) * PAIR_BM;
    n0 = (u / nm) * out_cols;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 2 * EPI_WARPS);
    }
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmA0);
    tc::tma_prefetch_desc(&tmB0);
    if (n_prob > 1) {
      tc::tma_prefetch_desc(&tmA1);
      tc::tma_prefetch_desc(&tmB1);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish_pair();
  }
  tc::tc_fence_before();
  // both CTAs' barriers are initialised and both TMEM allocations made before either CTA
  // signals the other
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  span_begin(span);

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // ---------------- producer (both CTAs)
    uint32_t it = 0;
    for (int t = pair; ok && t < total; t += n_pairs) {
      int pr, m0, n0;
      locate(t, pr, m0, n0);
      const CUtensorMap* tmA = pr ? &tmA1 : &tmA0;
      const CUtensorMap* tmB = pr ? &tmB1 : &tmB0;
      const int KB = pr ? kb1 : kb0;
      const int brow = swiglu ? (rank ? (int)g0.b_up_row + n0 : n0) : n0 + (int)rank * (BN / 2);
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&empty[s], ph ^ 1)) {
          ok = false;
          break;
        }
        // the even CTA's barrier counts the bytes of both CTAs' loads
        if (rank == 0) tc::mbar_expect_tx(&full[s], 2 * (A_BYTES + B_BYTES));
        const uint32_t fb = tc::mapa_shared(tc::smem_u32(&full[s]), 0);
        tc::tma_load_2d_pair(smA + s * A_BYTES, tmA, fb, kb * BK, m0 + (int)rank * BM);
        tc::tma_load_2d_pair(smB + s * B_BYTES, tmB, fb, kb * BK, brow);
      }
    }
    // wait until the MMAs have released every stage, so that no completion is still on its
    // way to this CTA's barriers when it exits
    for (uint32_t j = 0; ok && j < (uint32_t)STAGES; ++j, ++it)
      ok = tc::mbar_wait(&empty[it % STAGES], ((it / STAGES) & 1) ^ 1);
    if (!ok) atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
  } else if (warp == 1 && rank == 0) {
    // ---------------- pair MMA issuer (even CTA; the elected lane issues)
    constexpr uint32_t idesc = tc::idesc_bf16_f32(PAIR_BM, BN);
    const uint64_t a_desc0 = tc::desc_sw128(tc::smem_u32(smA));
    const uint64_t b_desc0 = tc::desc_sw128(tc::smem_u32(smB));
    uint32_t it = 0, i = 0;
    for (int t = pair; ok && t < total; t += n_pairs, ++i) {
      const uint32_t b = i & 1;
      const int KB = t >= t0 ? kb1 : kb0;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&acc_empty[b], ((i >> 1) & 1) ^ 1))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t d_tmem = tmem + b * 256;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&full[s], ph))) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        if (tc::elect_one()) {
          const uint64_t a_desc = a_desc0 + (uint64_t)((s * A_BYTES) >> 4);
          const uint64_t b_desc = b_desc0 + (uint64_t)((s * B_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_bf16_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, (kb | k) != 0);
          tc::mma_commit_pair(&empty[s], 0x3);
        }
        __syncwarp();
      }
      if (ok) {
        if (tc::elect_one()) tc::mma_commit_pair(&acc_full[b], 0x3);
        __syncwarp();
      }
    }
    if (!ok && lane == 0) atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs): this CTA's 128 rows of each tile
    const int lane_base = (warp & 3) * 32;
    const int half = (warp - 2) >> 2;
    const uint32_t release0 = tc::mapa_shared(tc::smem_u32(&acc_empty[0]), 0);
    const uint32_t release1 = tc::mapa_shared(tc::smem_u32(&acc_empty[1]), 0);
    uint32_t i = 0;
    for (int t = pair; t < total; t += n_pairs, ++i) {
      const uint32_t b = i & 1;
      int pr, m0, n0;
      locate(t, pr, m0, n0);
      const GemmDesc& g = pr ? g1 : g0;
      const int m = m0 + (int)rank * BM + lane_base + lane;
      const float rs = row_scale(g, m);
      const uint32_t trow = tmem + b * 256 + (static_cast<uint32_t>(lane_base) << 16);
      const bool done = epilogue_tile<BN>(g, m, n0, half, trow, swiglu, rs, [&] {
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (i >> 1) & 1))) return false;
        tc::tc_fence_after();
        return true;
      });
      if (!done) {
        if (lane == 0) atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
        break;
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(b ? release1 : release0);
    }
  }
  __syncwarp();
  tc::tc_fence_before();
  // neither CTA frees its TMEM (or exits) before the pair's last MMA and epilogue are done
  tc::cluster_sync();
  span_end(span);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// Failure-path self test of the bounded waits every tcgen05 kernel uses: an mbarrier that
// completes (arrive != 0) or that nothing completes; the wait gives up after max_polls
// tries, records ERRBIT_TIMEOUT and the kernel returns, leaving the context usable.
__global__ void k_wait_selftest(uint32_t max_polls, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) tc::mbar_arrive(&bar);
    if (!tc::mbar_wait_n(&bar, 0, max_polls)) atomicOr(&g_err_tc, ERRBIT_TIMEOUT);
  }
}

// ---- host: tensor maps through the driver entry point (no libcuda link dependency)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// looked up once per process (a function-local static: thread-safe initialisation)
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess) return reinterpret_cast<EncodeTiledFn>(p);
    if (e != cudaSuccess) cudaGetLastError();   // clears the error of this lookup only
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// rows x cols (cols innermost, contiguous), row stride ld elements; box = box_rows x 64
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
              int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t max_polls, int arrive, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(max_polls, arrive);
  return cudaGetLastError();
}

namespace {

// Host-side caches of this file, per device: SM count, which kernel variants have their
// shared-memory limit set (one bit each), co-resident CTA pairs.  One mutex guards them
// (calls may come from several host threads); a failed query is not cached, and
// reset_gemm_tc_caches() empties them.
std::mutex g_tc_mu;
int g_tc_sms[64];
uint32_t g_tc_attr[64];
int g_pair_slots[64];
bool g_pair_done[64];

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  {
    std::lock_guard<std::mutex> g(g_tc_mu);
    if (g_tc_sms[dev]) return g_tc_sms[dev];
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();   // clears the error of the call just made
    return 148;
  }
  if (n <= 0) return 148;
  std::lock_guard<std::mutex> g(g_tc_mu);
  g_tc_sms[dev] = n;
  return n;
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` once per device (bit `bit` of the
// device's mask records it).
cudaError_t ensure_smem_attr(const void* kernel, int bytes, int bit) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    std::lock_guard<std::mutex> g(g_tc_mu);
    if ((g_tc_attr[dev] >> bit) & 1u) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (cached) {
    std::lock_guard<std::mutex> g(g_tc_mu);
    g_tc_attr[dev] |= 1u << bit;
  }
  return cudaSuccess;
}
constexpr int attr_bit_single(int bn) { return bn == 256 ? 0 : bn == 224 ? 1 : bn == 208 ? 2 : 3; }
constexpr int attr_bit_pair(int bn) { return 4 + (bn == 256 ? 0 : bn == 224 ? 1 : 2); }

int tiles_for(const GemmDesc* gs, int n, int out_cols) {
  int tiles = 0;
  for (int p = 0; p < n; ++p) tiles += ((gs[p].N + out_cols - 1) / out_cols) * ((gs[p].M + BM - 1) / BM);
  return tiles;
}

// Tile width for one launch: each SM's share of the work is ceil(tiles / SMs) tiles of BN
// columns, so pick the BN with the smallest product; a narrower tile must save at least 5%
// (it moves more operand bytes per FLOP).  208 fits one wave of 7 x 20 tiles (832 x 4096)
// where 224 leaves 19 SMs idle.  SwiGLU (gate and up halves of 16-column chunks per epilogue
// warp) keeps 256; the fused deviation (one partial per half tile of whole 32-column pairs
// of chunks) takes 256, 224 or 192.
int pick_tile_n(const GemmDesc* gs, int n, int n_sm) {
  if (gs[0].epi.kind == EPI_SWIGLU) return 256;
  bool dev = false;
  for (int p = 0; p < n; ++p) dev = dev || gs[p].epi.dev_part != nullptr;
  const int cand[4] = {256, 224, 208, 192};
  int best = 256;
  int64_t best_cost = 0;
  for (int c = 0; c < 4; ++c) {
    if (dev && cand[c] == 208) continue;
    const int64_t cost = (int64_t)((tiles_for(gs, n, cand[c]) + n_sm - 1) / n_sm) * cand[c];
    if (c == 0 || cost * 20 <= best_cost * 19) {
      if (c == 0 || cost < best_cost) {
        best = cand[c];
        best_cost = cost;
      }
    }
  }
  return best;
}

template <int BN>
cudaError_t launch_tiles(const GemmDesc* gs, int n, bool swiglu, int n_sm, cudaStream_t s) {
  constexpr int SMEM_BYTES = TileCfg<BN>::SMEM_BYTES;
  CUtensorMap tmA[2], tmB[2];
  const int out_cols = swiglu ? BN / 2 : BN;
  for (int p = 0; p < n; ++p) {
    const GemmDesc& g = gs[p];
    if (!make_map(&tmA[p], g.A, g.M, g.K, g.lda, BM)) return cudaErrorInvalidValue;
    const int64_t b_rows = swiglu ? g.b_up_row + g.N : g.N;
    if (!make_map(&tmB[p], g.B, b_rows, g.K, g.ldb, swiglu ? BN / 2 : BN)) return cudaErrorInvalidValue;
  }
  if (n == 1) {
    tmA[1] = tmA[0];
    tmB[1] = tmB[0];
  }
  {
    const cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_gemm_tc<BN>), SMEM_BYTES, attr_bit_single(BN));
    if (e != cudaSuccess) return e;
  }
  const int tiles = tiles_for(gs, n, out_cols);
  const int grid = tiles < n_sm ? tiles : n_sm;
  const cudaError_t e = launch_k(k_gemm_tc<BN>, dim3(grid), dim3(THREADS), SMEM_BYTES, s, tmA[0], tmB[0], tmA[1],
                                 tmB[1], gs[0], n > 1 ? gs[1] : gs[0], n, swiglu ? 1 : 0, prof_span_slot());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int pair_tiles_for(const GemmDesc* gs, int n, int out_cols) {
  int tiles = 0;
  for (int p = 0; p < n; ++p)
    tiles += ((gs[p].N + out_cols - 1) / out_cols) * ((gs[p].M + PAIR_BM - 1) / PAIR_BM);
  return tiles;
}

template <int BN>
cudaError_t pair_attr() {
  return ensure_smem_attr(reinterpret_cast<const void*>(k_gemm_tc_pair<BN>), PairCfg<BN>::SMEM_BYTES,
                          attr_bit_pair(BN));
}

cudaLaunchConfig_t pair_config(cudaLaunchAttribute* attr, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cfg;
}

// Co-resident CTA pairs on this device (one CTA per SM), once per device; 0 if pair launches
// are unavailable.  Also sets the pair kernels' shared-memory limits.  A failed query gives 0
// for this call only (it is asked again next time); only its own error is cleared.
int pair_slots() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  {
    std::lock_guard<std::mutex> g(g_tc_mu);
    if (g_pair_done[dev]) return g_pair_slots[dev];
  }
  if (pair_attr<256>() != cudaSuccess || pair_attr<224>() != cudaSuccess || pair_attr<192>() != cudaSuccess) {
    cudaGetLastError();   // clears the error of the call that just failed
    return 0;
  }
  int mp = 0;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(attr, 0);
  cfg.dynamicSmemBytes = PairCfg<256>::SMEM_BYTES;
  cfg.gridDim = dim3(2 * (sm_count() / 2));
  if (cudaOccupancyMaxActiveClusters(&mp, k_gemm_tc_pair<256>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> g(g_tc_mu);
  g_pair_slots[dev] = mp;
  g_pair_done[dev] = true;
  return mp;
}

template <int BN>
cudaError_t launch_pair(const GemmDesc* gs, int n, bool swiglu, int n_pairs, cudaStream_t s) {
  CUtensorMap tmA[2], tmB[2];
  for (int p = 0; p < n; ++p) {
    const GemmDesc& g = gs[p];
    if (!make_map(&tmA[p], g.A, g.M, g.K, g.lda, BM)) return cudaErrorInvalidValue;
    const int64_t b_rows = swiglu ? g.b_up_row + g.N : g.N;
    if (!make_map(&tmB[p], g.B, b_rows, g.K, g.ldb, BN / 2)) return cudaErrorInvalidValue;
  }
  if (n == 1) {
    tmA[1] = tmA[0];
    tmB[1] = tmB[0];
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(attr, s);
  cfg.dynamicSmemBytes = PairCfg<BN>::SMEM_BYTES;
  const int tiles = pair_tiles_for(gs, n, swiglu ? BN / 2 : BN);
  cfg.gridDim = dim3(2 * (tiles < n_pairs ? tiles : n_pairs));
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_tc_pair<BN>, tmA[0], tmB[0], tmA[1], tmB[1], gs[0],
                                           n > 1 ? gs[1] : gs[0], n, swiglu ? 1 : 0, prof_span_slot());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// CB_GEMM_PAIR=0 forces single-SM tiles, =1 pair tiles wherever a pair launch is possible
// (for measurement); unset, plan_tiles decides.
int pair_mode() {
  static const int mode = [] {
    const char* v = getenv("CB_GEMM_PAIR");
    return (v && v[0] == '0') ? 0 : (v && v[0] == '1') ? 1 : -1;
  }();
  return mode;
}

struct TilePlan {
  bool pair;
  int bn;
};

// Kernel and tile width of one launch.  A launch takes about (waves of tiles over the
// co-resident CTAs, or pairs) x BN per SM.  A pair tile does the same per-SM work as a
// single-SM tile of its width in about 1/1.12 of the time (measured at equal wave counts:
// 4096 x 8192 x 4096 and 8192^3 ran 13-15% faster as pairs), but pads M to 256 rows: pairs
// are taken only with at least two waves and at most 8% more padded rows than single tiles
// (832 rows pad to 1024 as pairs, 14% more than 896; 1664 rows to 1792, 7.7% more, where the
// 1664 x 13824 SwiGLU runs 430 -> 405 us as pairs), and there where their cost is lower.
// SwiGLU keeps 256 columns either way.
TilePlan plan_tiles(const GemmDesc* gs, int n, int n_sm, int n_pairs) {
  TilePlan tp{false, pick_tile_n(gs, n, n_sm)};
  const int mode = pair_mode();
  if (mode == 0 || n_pairs < 1) return tp;
  const bool fixed = gs[0].epi.kind == EPI_SWIGLU;
  const int cand[3] = {256, 224, 192};
  int pbn = 256;
  int64_t pcost = 0, pwaves = 0;
  for (int c = 0; c < (fixed ? 1 : 3); ++c) {
    const int out = gs[0].epi.kind == EPI_SWIGLU ? cand[c] / 2 : cand[c];
    const int64_t waves = (pair_tiles_for(gs, n, out) + n_pairs - 1) / n_pairs;
    const int64_t cost = waves * cand[c];
    if (c == 0 || (cost * 20 <= pcost * 19 && cost < pcost)) {
      pbn = cand[c];
      pcost = cost;
      pwaves = waves;
    }
  }
  if (mode == 1) return TilePlan{true, pbn};
  int64_t rows_single = 0, rows_pair = 0;
  for (int p = 0; p < n; ++p) {
    rows_single += (int64_t)((gs[p].M + BM - 1) / BM) * BM;
    rows_pair += (int64_t)((gs[p].M + PAIR_BM - 1) / PAIR_BM) * PAIR_BM;
  }
  const int out_s = gs[0].epi.kind == EPI_SWIGLU ? tp.bn / 2 : tp.bn;
  const int64_t scost = (int64_t)((tiles_for(gs, n, out_s) + n_sm - 1) / n_sm) * tp.bn;
  if (pwaves >= 2 && rows_pair * 100 <= rows_single * 108 && pcost * 100 < scost * 112) return TilePlan{true, pbn};
  return tp;
}

}  // namespace

void reset_gemm_tc_caches() {
  std::lock_guard<std::mutex> g(g_tc_mu);
  for (int i = 0; i < 64; ++i) {
    g_tc_sms[i] = 0;
    g_tc_attr[i] = 0;
    g_pair_slots[i] = 0;
    g_pair_done[i] = false;
  }
}

// The tile width (output columns per tile, SwiGLU: gate + up) launch_gemm_tc_group will use
// for this launch; the fused deviation's partials are laid out per half tile of this width.
int gemm_tc_tile_n(const GemmDesc* gs, int n) {
  return plan_tiles(gs, n, sm_count(), pair_slots()).bn;
}

// Host preconditions (checked by the caller's validation, re-checked here): K % 8 == 0,
// lda/ldb % 8 == 0, A and B 16-byte aligned, N % 16 == 0.
cudaError_t launch_gemm_tc_group(const GemmDesc* gs, int n, cudaStream_t s) {
  if (n < 1 || n > 2) return cudaErrorInvalidValue;
  const bool swiglu = gs[0].epi.kind == EPI_SWIGLU;
  if (n > 1 && (swiglu || gs[1].epi.kind == EPI_SWIGLU)) return cudaErrorInvalidValue;
  for (int p = 0; p < n; ++p) {
    const GemmDesc& g = gs[p];
    if (g.K % 8 || g.lda % 8 || g.ldb % 8 || g.N % 16 || ((uintptr_t)g.A & 15) || ((uintptr_t)g.B & 15))
      return cudaErrorInvalidValue;
  }
  const int n_sm = sm_count();
  const int n_pairs = pair_slots();
  const TilePlan tp = plan_tiles(gs, n, n_sm, n_pairs);
  if (tp.pair) {
    switch (tp.bn) {
      case 224:
        return launch_pair<224>(gs, n, swiglu, n_pairs, s);
      case 192:
        return launch_pair<192>(gs, n, swiglu, n_pairs, s);
      default:
        return launch_pair<256>(gs, n, swiglu, n_pairs, s);
    }
  }
  switch (tp.bn) {
    case 224:
      return launch_tiles<224>(gs, n, swiglu, n_sm, s);
    case 208:
      return launch_tiles<208>(gs, n, swiglu, n_sm, s);
    case 192:
      return launch_tiles<192>(gs, n, swiglu, n_sm, s);
    default:
      return launch_tiles<256>(gs, n, swiglu, n_sm, s);
  }
}

cudaError_t launch_gemm_tc(const GemmDesc& g, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  return launch_gemm_tc_group(&g, 1, s);
}

}  // namespace cb
