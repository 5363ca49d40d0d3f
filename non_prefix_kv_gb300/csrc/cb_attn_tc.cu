// Tensor-core attention of selected queries over the whole causal KV (bf16, head_dim 64 or
// 128): CacheBlend explainer (0h-n0.github.io/posts/paper-2312-03052) §Selective
// recomputation Step 4 — the selected tokens attend over the entire blended input.
//
// Per 128-query tile and query head, over 128-key tiles j:
//   S_j = Q K_j^T          tcgen05.mma, A = Q (K-major), B = K_j (K-major), into TMEM
//   P_j = exp2(S_j * log2(e)/sqrt(hd) - m)   softmax warps, row = TMEM lane, key t of a
//                          row visible iff t <= q_pos[row]
//   O  += P_j V_j          tcgen05.mma, A = P_j from TMEM, B = V_j (MN-major), fp32 in TMEM
// Two softmax groups take alternate key tiles, each with its own S buffer, running max, row
// sum and O accumulator (TMEM: S_0 | S_1 | O_0 | O_1); one thread owns one query row of its
// group's tiles, so no warp waits for another until the two halves of the key range are
// merged at the end.  The running max is raised lazily: O is rescaled only when a row's max
// grows by more than 2^8.  One CTA per (128-query tile, query head); K and V stream through
// a TMA ring.  Warp roles: 0 = TMA producer, 1 = TMEM allocator + MMA issuer (the whole warp
// runs the issue loop, the elected lane issues), 2..9 = softmax groups and epilogue; warp w
// reads TMEM lanes 32*(w%4)..+31.  A second kernel (k_attn_tc2) takes two query tiles per
// CTA, one per softmax group, for dense launches with many query tiles.
#include <cuda.h>
#include <math.h>

#include <mutex>

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
constexpr int NSOFT = 8;             // softmax warps: two groups of one per TMEM lane quarter
constexpr int THREADS = 32 * (2 + NSOFT);
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleLog2 = 8.0f;

// Packed fp32 pairs (sm_100+): one instruction updates two score elements.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// three-input maximum (NaN inputs are ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One key tile of a softmax group, shared by both attention kernels; a thread owns one query
// row of the group's S and O in TMEM.  Pass 1 takes the row's maximum over the tile, the
// running max is raised lazily (O_g rescaled only when it grows by more than 2^8), pass 2
// writes P over S and adds it to the row sum, then the group's P_j is signalled.  u is the
// tile's index among the group's tiles (the barriers' phases; u = 0 starts O_g).  Returns
// false when a wait gave up.
template <int HD>
__device__ __forceinline__ bool softmax_tile(uint64_t* s_full_g, uint64_t* p_full_g, uint64_t* pv_done_g, uint32_t u,
                                             int key0, int qp, uint32_t tS, uint32_t tO, float scale_log2,
                                             float& m_used, float& l, int lane) {
  if (!__all_sync(0xffffffffu, tc::mbar_wait(s_full_g, u & 1))) return false;
  // every key of this tile lies beyond all 32 rows' positions: no load, P = 0
  const bool none = __all_sync(0xffffffffu, key0 > qp);
  const bool full_row = key0 + BN - 1 <= qp;
  // pass 1: the row's maximum over the tile, 64 columns at a time (a whole 128-column row
  // does not fit in the registers three warps per sub-partition leave)
  float pmx[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) pmx[a] = -INFINITY;
  if (!none) {
    tc::tc_fence_after();
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t sr[64];
      tc::tmem_ld32_nowait(tS + hf * 64, sr);
      tc::tmem_ld32_nowait(tS + hf * 64 + 32, sr + 32);
      tc::tmem_wait_ld();
      if (full_row) {
#pragma unroll
        for (int i = 0; i < 64; i += 8) {
#pragma unroll
          for (int a = 0; a < 4; ++a)
            pmx[a] = fmax3(pmx[a], __uint_as_float(sr[i + 2 * a]), __uint_as_float(sr[i + 2 * a + 1]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (key0 + hf * 64 + i <= qp) pmx[i & 3] = fmaxf(pmx[i & 3], __uint_as_float(sr[i]));
      }
    }
  }
  const float mt = fmaxf(fmaxf(pmx[0], pmx[1]), fmaxf(pmx[2], pmx[3])) * scale_log2;
  const float m_new = fmaxf(m_used, mt);
  if (u == 0) {
    m_used = m_new;            // O_g is written, not added to, by this tile's P.V
  } else {
    const bool need = m_new > m_used + kRescaleLog2;
    if (__any_sync(0xffffffffu, need)) {
      // O_g must be stable: the group's previous P.V has completed
      if (!__all_sync(0xffffffffu, tc::mbar_wait(pv_done_g, (u - 1) & 1))) return false;
      tc::tc_fence_after();
      const float alpha = need ? tc::ex2_approx(m_used - m_new) : 1.0f;
#pragma unroll 1
      for (int c = 0; c < HD / 16; ++c) {
        float o[16];
        tc::tmem_ld16(tO + c * 16, o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] *= alpha;
        tc::tmem_st16(tO + c * 16, o);
      }
      l *= alpha;
      if (need) m_used = m_new;
    }
  }
  // pass 2: P = 2^(s * log2(e)/sqrt(hd) - m), two scores per packed instruction; keys 2w,
  // 2w+1 go to P column w (bf16 pair).  Keys 0..63 are read again and their P written to
  // columns 0..31 before keys 64..127 are read; P of those lands in columns 32..63, whose
  // scores were read in the first half.
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_used, -m_used);
  uint64_t ls2[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) ls2[a] = 0ull;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t sr[64];
    if (!none) {
      tc::tmem_ld32_nowait(tS + hf * 64, sr);
      tc::tmem_ld32_nowait(tS + hf * 64 + 32, sr + 32);
      tc::tmem_wait_ld();
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t pk[16];
      if (none) {
#pragma unroll
        for (int w = 0; w < 16; ++w) pk[w] = 0u;
      } else {
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const int k0 = c * 32 + 2 * w;
          const int key = key0 + hf * 64 + k0;
          const float2 z =
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k0]), __uint_as_float(sr[k0 + 1])), sc2, nm2));
          float p0 = tc::ex2_approx(z.x);
          float p1 = tc::ex2_approx(z.y);
          if (!full_row) {
            p0 = (key <= qp) ? p0 : 0.f;
            p1 = (key + 1 <= qp) ? p1 : 0.f;
          }
          ls2[w & 3] = f2_add(ls2[w & 3], f2_pack(p0, p1));
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
          pk[w] = *reinterpret_cast<const uint32_t*>(&b2);
        }
      }
      tc::tmem_st16u_nowait(tS + hf * 32 + c * 16, pk);
    }
  }
  {
    const float2 a = f2_unpack(f2_add(ls2[0], ls2[1])), c = f2_unpack(f2_add(ls2[2], ls2[3]));
    l += (a.x + a.y) + (c.x + c.y);
  }
  tc::tmem_wait_st();
  tc::tc_fence_before();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(p_full_g);
  return true;
}

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, %0;" ::"n"(NSOFT * 32) : "memory"); }

// ---- two softmax groups on alternating key tiles ------------------------------------------
// TMEM: S_0 | S_1 | O_0 | O_1.  Group g (warps 2 + 4g .. 5 + 4g, one per TMEM lane quarter)
// owns the key tiles j = g, g + 2, ...: each of its threads reads one query row's 128 scores
// of S_g, keeps that row's running maximum and sum for the group's tiles, writes P_j (bf16
// pairs) over S_g and the tensor core adds P_j V_j into O_g.  Neither group waits for the
// other until the end, where the two partial results are merged per row:
//   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)),  m = max(m_0, m_1),
// the same online-softmax algebra that joins consecutive tiles, applied to two interleaved
// halves of the key range.  While one group exponentiates, the tensor core works on the
// other group's tiles; S(j + 2) reuses S_g once P.V(j) has completed.
template <int HD>
struct Layout {
  static constexpr int NSLAB = HD / 64;
  static constexpr int Q_BYTES = NSLAB * SLAB;
  static constexpr int KV_BYTES = NSLAB * SLAB;
  static constexpr int KV_STAGES = HD == 128 ? 5 : 10;      // ring K_0, V_0, K_1, V_1, ...
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + Q_BYTES;
  static constexpr int OFF_X = OFF_KV + KV_STAGES * KV_BYTES;  // per group: row max, row sum
  static constexpr int X_BYTES = 2 * 2 * BM * 4;
  static constexpr int OFF_BAR = OFF_X + X_BYTES;
  static constexpr int BYTES = OFF_BAR + 256;
  static constexpr int SMEM = BYTES + 1024;
  static_assert((1 + 6 + 2 * KV_STAGES) * 8 + 8 <= 256, "barriers exceed their region");
};
constexpr uint32_t TM2_O = 2 * BN;   // O_0 at column 256, O_1 right after it

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const int32_t* __restrict__ q_pos, int M,
               int64_t n_kv, int H, int Hkv, bf16* __restrict__ out, float scale_log2,
               unsigned long long* span) {
  pdl_wait();
  pdl_trigger();
  span_begin(span);
  using L = Layout<HD>;
  constexpr int NST = L::KV_STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* sQ = base + L::OFF_Q;
  uint8_t* sKV = base + L::OFF_KV;
  float* xm = reinterpret_cast<float*>(base + L::OFF_X);   // [2 groups][BM] row max
  float* xl = xm + 2 * BM;                                  // [2 groups][BM] row sum
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;     // [2] per group: S_g holds tile j's scores
  uint64_t* p_full = bars + 3;     // [2] the group's four warps wrote P_j
  uint64_t* pv_done = bars + 5;    // [2] P_j V_j into O_g completed
  uint64_t* kv_full = bars + 7;    // [NST]
  uint64_t* kv_empty = kv_full + NST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(kv_empty + NST);
  int* s_qmax = reinterpret_cast<int*>(kv_empty + NST) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Query tiles are cut from the end of the (position-sorted) rows: tile y holds rows
  // [M - 128 (y + 1), M - 128 y), so a partial tile, if any, is the one with the smallest
  // positions (the cheapest) rather than the last one (which sees every key).  Heads vary
  // fastest in launch order and the latest (longest) query tiles come first, so every
  // head's heavy tiles start in the first wave and the short ones fill in behind.
  const int h = blockIdx.x;
  const int g_kv = h / (H / Hkv);
  const int m0 = M - (int)(blockIdx.y + 1) * BM;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], 4);
      tc::mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < NST; ++i) {
      tc::mbar_init(&kv_full[i], 1);
      tc::mbar_init(&kv_empty[i], 1);
    }
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmQ);
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    int mx = 0;
    for (int i = lane; i < BM; i += 32) {
      const int m = m0 + i;
      if (m >= 0 && m < M) {
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
    for (int i = 0; i < 2 * T; ++i) {
      const int st = i % NST;
      if (!tc::mbar_wait(&kv_empty[st], ((i / NST) & 1) ^ 1)) {
        atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
        break;
      }
      tc::mbar_expect_tx(&kv_full[st], L::KV_BYTES);
      const CUtensorMap* map = (i & 1) ? &tmV : &tmK;
      for (int s = 0; s < L::NSLAB; ++s)
        tc::tma_load_2d(sKV + st * L::KV_BYTES + s * SLAB, map, &kv_full[st], g_kv * HD + 64 * s, (i >> 1) * BN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (warp 1)
    // S(0), S(1); then per key tile j: P.V(j) once its group wrote P, and S(j + 2) into the
    // same group's buffer once that P.V has completed.
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(BM, HD, true);
    const uint64_t kv_desc = tc::desc_sw128(tc::smem_u32(sKV));
    const uint64_t v_desc = tc::desc_sw128_mn(tc::smem_u32(sKV), SLAB);
    const uint64_t q_desc = tc::desc_sw128(tc::smem_u32(sQ));
    bool ok = __all_sync(0xffffffffu, tc::mbar_wait(q_full, 0));
    auto issue_s = [&](int jj) {
      const int b = jj & 1, i = 2 * jj, st = i % NST;
      ok = ok && __all_sync(0xffffffffu, tc::mbar_wait(&kv_full[st], (i / NST) & 1) &&
                                             (jj < 2 || tc::mbar_wait(&pv_done[b], ((jj - 2) >> 1) & 1)));
      if (!ok) return;
      tc::tc_fence_after();
      if (tc::elect_one()) {
        const uint64_t kd = kv_desc + (uint64_t)((st * L::KV_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = ((k >> 2) * SLAB + (k & 3) * 32) >> 4;
          tc::mma_bf16(tmem + b * BN, q_desc + off, kd + off, idesc_s, k > 0);
        }
        tc::mma_commit(&s_full[b]);
        tc::mma_commit(&kv_empty[st]);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int jj) {
      const int b = jj & 1, i = 2 * jj + 1, st = i % NST;
      ok = ok && __all_sync(0xffffffffu, tc::mbar_wait(&p_full[b], (jj >> 1) & 1) &&
                                             tc::mbar_wait(&kv_full[st], (i / NST) & 1));
      if (!ok) return;
      tc::tc_fence_after();
      if (tc::elect_one()) {
        const uint64_t vd = v_desc + (uint64_t)((st * L::KV_BYTES) >> 4);
        const uint32_t pa = tmem + b * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          tc::mma_bf16_ts(tmem + TM2_O + b * HD, pa + k * 8, vd + (uint64_t)((k * 16 * 128) >> 4), idesc_o,
                          (jj >= 2 || k > 0) ? 1u : 0u);
        tc::mma_commit(&pv_done[b]);
        tc::mma_commit(&kv_empty[st]);
      }
      __syncwarp();
    };
    issue_s(0);
    if (T > 1) issue_s(1);
    for (int jj = 0; ok && jj < T; ++jj) {
      issue_pv(jj);
      if (jj + 2 < T) issue_s(jj + 2);
    }
    if (!ok && lane == 0) atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ softmax groups
    const int grp = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int m = m0 + r;
    const bool row_valid = m >= 0 && m < M;
    int qp = 0;
    if (row_valid) {
      qp = q_pos[m];
      qp = qp < 0 ? 0 : (qp >= n_kv ? (int)(n_kv - 1) : qp);
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tS = trow + grp * BN;
    const uint32_t tO = trow + TM2_O + grp * HD;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;   // warp-uniform; a failed wait stops the work, never the loop
    int u = 0;        // this group's tile count
    for (int j = grp; j < T; j += 2, ++u)
      if (ok) ok = softmax_tile<HD>(&s_full[grp], &p_full[grp], &pv_done[grp], (uint32_t)u, j * BN, qp, tS, tO,
                                    scale_log2, m_used, l, lane);
    // the group's last P.V, then both groups' row statistics meet in shared memory
    const bool done = ok && (u == 0 || __all_sync(0xffffffffu, tc::mbar_wait(&pv_done[grp], (u - 1) & 1)));
    xm[grp * BM + r] = m_used;
    xl[grp * BM + r] = l;
    tc::tc_fence_before();
    softmax_bar();   // every softmax warp reaches this barrier exactly once
    if (done) {
      tc::tc_fence_after();
      const bool has1 = T > 1;       // group 1 saw at least one tile (else O_1 was never written)
      const float ma = xm[r], mb = has1 ? xm[BM + r] : -INFINITY;
      const float mm = fmaxf(ma, mb);
      const float a0 = ma == -INFINITY ? 0.f : tc::ex2_approx(ma - mm);
      const float a1 = mb == -INFINITY ? 0.f : tc::ex2_approx(mb - mm);
      const float lt = xl[r] * a0 + (has1 ? xl[BM + r] * a1 : 0.f);
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      // group g finalises output columns [g HD/2, (g + 1) HD/2) of its rows
      bf16* orow = out + (int64_t)(row_valid ? m : 0) * H * HD + (int64_t)h * HD + grp * (HD / 2);
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        const uint32_t col = TM2_O + grp * (HD / 2) + c * 16;
        float o0[16], o1[16];
        tc::tmem_ld16(trow + col, o0);
        if (has1) {
          tc::tmem_ld16(trow + col + HD, o1);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o1[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) o0[i] = (o0[i] * a0 + o1[i] * a1) * inv;
        if (row_valid) {
          if ((reinterpret_cast<uintptr_t>(orow + c * 16) & 31) == 0) {
            st16_v8(orow + c * 16, o0);
          } else {
            st8(orow + c * 16, o0);
            st8(orow + c * 16 + 8, o0 + 8);
          }
        }
      }
    } else if (lane == 0) {
      atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
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

// ---- two query tiles per CTA --------------------------------------------------------------
// For launches with many query tiles per head.  Group g owns query tile y_g = 2 p + g of the
// CTA's pair p (tile 2 p is the later, longer one) and walks every key tile up to its own
// bound; both groups' S use the same K_j from shared memory and both P.V the same V_j.  Each
// group's row statistics and O_g then cover its whole key range, so the epilogue needs no
// merge.  TMEM is laid out as in the kernel above (S_0 | S_1 | O_0 | O_1).  Per key tile and
// query tile the work is the same as there; the CTAs, and with them the ramp at the start and
// the drain at the end of every CTA's chain of hand-offs, are half as many, and every K/V
// tile is loaded once for two query tiles.
template <int HD>
struct Layout2 {
  static constexpr int NSLAB = HD / 64;
  static constexpr int Q_BYTES = NSLAB * SLAB;                // one query tile
  static constexpr int KV_BYTES = NSLAB * SLAB;
  static constexpr int KV_STAGES = HD == 128 ? 5 : 10;
  static constexpr int OFF_Q = 0;                             // [2 query tiles]
  static constexpr int OFF_KV = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_BAR = OFF_KV + KV_STAGES * KV_BYTES;
  static constexpr int BYTES = OFF_BAR + 256;
  static constexpr int SMEM = BYTES + 1024;
  static_assert((1 + 6 + 2 * KV_STAGES) * 8 + 16 <= 256, "barriers exceed their region");
  static_assert(SMEM <= 227 * 1024, "shared memory exceeds the per-block limit");
};

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    k_attn_tc2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const int32_t* __restrict__ q_pos, int M,
               int64_t n_kv, int H, int Hkv, bf16* __restrict__ out, float scale_log2,
               unsigned long long* span) {
  pdl_wait();
  pdl_trigger();
  span_begin(span);
  using L = Layout2<HD>;
  constexpr int NST = L::KV_STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* sQ = base + L::OFF_Q;
  uint8_t* sKV = base + L::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;     // [2] per group: S_g holds key tile j's scores
  uint64_t* p_full = bars + 3;     // [2] the group's four warps wrote P_j
  uint64_t* pv_done = bars + 5;    // [2] P_j V_j into O_g completed
  uint64_t* kv_full = bars + 7;    // [NST]
  uint64_t* kv_empty = kv_full + NST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(kv_empty + NST);
  int* s_tmax = reinterpret_cast<int*>(kv_empty + NST) + 1;   // [2] key tiles per group

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int g_kv = h / (H / Hkv);
  const int n_qt = (M + BM - 1) / BM;
  // query tile y holds rows [M - 128 (y + 1), M - 128 y): tile 0 is the latest (longest)
  const int y0 = 2 * (int)blockIdx.y, y1 = y0 + 1;
  const bool has1 = y1 < n_qt;
  const int m00 = M - (y0 + 1) * BM, m01 = M - (y1 + 1) * BM;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], 4);
      tc::mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < NST; ++i) {
      tc::mbar_init(&kv_full[i], 1);
      tc::mbar_init(&kv_empty[i], 1);
    }
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmQ);
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    // key tiles each query tile visits: up to its largest position
    for (int g = 0; g < 2; ++g) {
      const int m0 = g ? m01 : m00;
      int mx = -1;
      if (g == 0 || has1) {
        for (int i = lane; i < BM; i += 32) {
          const int m = m0 + i;
          if (m >= 0 && m < M) {
            int p = q_pos[m];
            if (p < 0 || p >= n_kv) {
              atomicOr(&g_err_attn_tc, ERRBIT_INDEX);
              p = p < 0 ? 0 : (int)(n_kv - 1);
            }
            mx = p > mx ? p : mx;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const int y = __shfl_xor_sync(0xffffffffu, mx, o);
        mx = y > mx ? y : mx;
      }
      if (lane == 0) s_tmax[g] = mx < 0 ? 0 : mx / BN + 1;
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
  const int T0 = s_tmax[0], T1 = s_tmax[1];   // T1 = 0: no second query tile
  const int Tm = T0 > T1 ? T0 : T1;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    tc::mbar_expect_tx(q_full, (T1 > 0 ? 2 : 1) * L::Q_BYTES);
    for (int s = 0; s < L::NSLAB; ++s) tc::tma_load_2d(sQ + s * SLAB, &tmQ, q_full, h * HD + 64 * s, m00);
    if (T1 > 0)
      for (int s = 0; s < L::NSLAB; ++s)
        tc::tma_load_2d(sQ + L::Q_BYTES + s * SLAB, &tmQ, q_full, h * HD + 64 * s, m01);
    for (int i = 0; i < 2 * Tm; ++i) {
      const int st = i % NST;
      if (!tc::mbar_wait(&kv_empty[st], ((i / NST) & 1) ^ 1)) {
        atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
        break;
      }
      tc::mbar_expect_tx(&kv_full[st], L::KV_BYTES);
      const CUtensorMap* map = (i & 1) ? &tmV : &tmK;
      for (int s = 0; s < L::NSLAB; ++s)
        tc::tma_load_2d(sKV + st * L::KV_BYTES + s * SLAB, map, &kv_full[st], g_kv * HD + 64 * s, (i >> 1) * BN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (warp 1)
    // S_0(0), S_1(0); then per key tile j: P_0.V(j), S_0(j + 1), P_1.V(j), S_1(j + 1), each
    // group's S(j + 1) once its P.V(j) has completed.  A K or V stage is released by the last
    // MMA that reads it (group 1's while group 1 still has key tiles, else group 0's).
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(BM, HD, true);
    const uint64_t kv_desc = tc::desc_sw128(tc::smem_u32(sKV));
    const uint64_t v_desc = tc::desc_sw128_mn(tc::smem_u32(sKV), SLAB);
    const uint64_t q_desc = tc::desc_sw128(tc::smem_u32(sQ));
    bool ok = __all_sync(0xffffffffu, tc::mbar_wait(q_full, 0));
    auto issue_s = [&](int g, int j) {
      const int i = 2 * j, st = i % NST;
      ok = ok && __all_sync(0xffffffffu, tc::mbar_wait(&kv_full[st], (i / NST) & 1) &&
                                             (j == 0 || tc::mbar_wait(&pv_done[g], (j - 1) & 1)));
      if (!ok) return;
      tc::tc_fence_after();
      if (tc::elect_one()) {
        const uint64_t kd = kv_desc + (uint64_t)((st * L::KV_BYTES) >> 4);
        const uint64_t qd = q_desc + (uint64_t)((g * L::Q_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = ((k >> 2) * SLAB + (k & 3) * 32) >> 4;
          tc::mma_bf16(tmem + g * BN, qd + off, kd + off, idesc_s, k > 0);
        }
        tc::mma_commit(&s_full[g]);
        if (g == 1 || j >= T1) tc::mma_commit(&kv_empty[st]);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int g, int j) {
      const int i = 2 * j + 1, st = i % NST;
      ok = ok && __all_sync(0xffffffffu, tc::mbar_wait(&p_full[g], j & 1) &&
                                             tc::mbar_wait(&kv_full[st], (i / NST) & 1));
      if (!ok) return;
      tc::tc_fence_after();
      if (tc::elect_one()) {
        const uint64_t vd = v_desc + (uint64_t)((st * L::KV_BYTES) >> 4);
        const uint32_t pa = tmem + g * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          tc::mma_bf16_ts(tmem + TM2_O + g * HD, pa + k * 8, vd + (uint64_t)((k * 16 * 128) >> 4), idesc_o,
                          (j > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&pv_done[g]);
        if (g == 1 || j >= T1) tc::mma_commit(&kv_empty[st]);
      }
      __syncwarp();
    };
    issue_s(0, 0);
    if (T1 > 0) issue_s(1, 0);
    for (int j = 0; ok && j < Tm; ++j) {
      if (j < T0) {
        issue_pv(0, j);
        if (j + 1 < T0) issue_s(0, j + 1);
      }
      if (j < T1) {
        issue_pv(1, j);
        if (j + 1 < T1) issue_s(1, j + 1);
      }
    }
    if (!ok && lane == 0) atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ softmax groups
    const int grp = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int m = (grp ? m01 : m00) + r;
    const int T = grp ? T1 : T0;
    const bool row_valid = (grp == 0 || has1) && m >= 0 && m < M;
    int qp = 0;
    if (row_valid) {
      qp = q_pos[m];
      qp = qp < 0 ? 0 : (qp >= n_kv ? (int)(n_kv - 1) : qp);
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tS = trow + grp * BN;
    const uint32_t tO = trow + TM2_O + grp * HD;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;   // warp-uniform; a failed wait stops the work, never the loop
    for (int j = 0; j < T; ++j)
      if (ok) ok = softmax_tile<HD>(&s_full[grp], &p_full[grp], &pv_done[grp], (uint32_t)j, j * BN, qp, tS, tO,
                                    scale_log2, m_used, l, lane);
    // the group's last P.V; then O_g / l is this tile's output (no second half to merge)
    const bool done = ok && (T == 0 || __all_sync(0xffffffffu, tc::mbar_wait(&pv_done[grp], (T - 1) & 1)));
    if (done && T > 0) {
      tc::tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      bf16* orow = out + (int64_t)(row_valid ? m : 0) * H * HD + (int64_t)h * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 16; ++c) {
        float o[16];
        tc::tmem_ld16(tO + c * 16, o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] *= inv;
        if (row_valid) {
          if ((reinterpret_cast<uintptr_t>(orow + c * 16) & 31) == 0) {
            st16_v8(orow + c * 16, o);
          } else {
            st8(orow + c * 16, o);
            st8(orow + c * 16 + 8, o + 8);
          }
        }
      }
    } else if (!done && lane == 0) {
      atomicOr(&g_err_attn_tc, ERRBIT_TIMEOUT);
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

// which kernel variants have their shared-memory limit set, per device (one bit per head
// size), guarded for calls from several host threads; emptied by reset_attn_tc_caches()
std::mutex g_attn_mu;
uint32_t g_attn_attr[64];

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

// CB_ATTN_PAIR=0 keeps one query tile per CTA, =1 takes two wherever possible (for
// measurement and tests).  Unset, two are taken when a head has at least kPairMinTiles query
// tiles and the queries cover at least half the keys: there the two tiles of a CTA visit
// nearly the same key tiles (dense causal: one apart).  A sparse selection spreads a pair's
// bounds apart, one group idles while the other finishes, and with fewer, longer CTAs the
// packing onto the SMs is coarser (measured: 3328 of 16384 rows 662 -> 692 us; dense 4096
// 149 -> 137 us, 8192 495 -> 467 us).
constexpr int kPairMinTiles = 8;
int attn_pair_mode() {
  static const int mode = [] {
    const char* v = getenv("CB_ATTN_PAIR");
    return v && v[0] == '0' ? 0 : (v && v[0] == '1' ? 1 : -1);
  }();
  return mode;
}

template <int HD>
cudaError_t launch_hd(const void* q, const int32_t* q_pos, int M, const void* kc, const void* vc, int64_t n_kv,
                      int H, int Hkv, void* out, cudaStream_t s) {
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, M, (int64_t)H * HD, (int64_t)H * HD) ||
      !make_map(&tk, kc, n_kv, (int64_t)Hkv * HD, (int64_t)Hkv * HD) ||
      !make_map(&tv, vc, n_kv, (int64_t)Hkv * HD, (int64_t)Hkv * HD))
    return cudaErrorInvalidValue;
  const int n_qt = (M + BM - 1) / BM;
  const int mode = attn_pair_mode();
  const bool pair = mode == 1 ? n_qt >= 2 : (mode == 0 ? false : n_qt >= kPairMinTiles && 2 * (int64_t)M >= n_kv);
  auto kern = pair ? k_attn_tc2<HD> : k_attn_tc<HD>;
  const int smem = pair ? Layout2<HD>::SMEM : Layout<HD>::SMEM;
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < 64;
    const uint32_t bit = (HD == 128 ? 1u : 2u) << (pair ? 2 : 0);
    bool set = false;
    if (cached) {
      std::lock_guard<std::mutex> g(g_attn_mu);
      set = (g_attn_attr[dev] & bit) != 0;
    }
    if (!set) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      if (cached) {
        std::lock_guard<std::mutex> g(g_attn_mu);
        g_attn_attr[dev] |= bit;
      }
    }
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  dim3 grid(H, pair ? (n_qt + 1) / 2 : n_qt);
  { const cudaError_t e_ = launch_k(kern, dim3(grid), dim3(THREADS), smem, s, tq, tk, tv, q_pos, M, n_kv, H, Hkv,
                                    static_cast<bf16*>(out), scale_log2, prof_span_slot());
    if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(int hd) { return hd == 64 || hd == 128; }

void reset_attn_tc_caches() {
  std::lock_guard<std::mutex> g(g_attn_mu);
  for (int i = 0; i < 64; ++i) g_attn_attr[i] = 0;
}

cudaError_t launch_attention_tc(const void* q, const int32_t* q_pos, int M, const void* kc, const void* vc,
                                int64_t n_kv, int H, int Hkv, int hd, void* out, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  if (((uintptr_t)q & 15) || ((uintptr_t)kc & 15) || ((uintptr_t)vc & 15)) return cudaErrorInvalidValue;
  if (hd == 128) return launch_hd<128>(q, q_pos, M, kc, vc, n_kv, H, Hkv, out, s);
  if (hd == 64) return launch_hd<64>(q, q_pos, M, kc, vc, n_kv, H, Hkv, out, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
