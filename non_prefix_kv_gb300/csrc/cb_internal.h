// Internal launcher interface between the C ABI layer and the kernel translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace cb {

enum DType { DT_F32 = 0, DT_BF16 = 1 };

// bits of the sticky device error words
enum : uint32_t {
  ERRBIT_NONFINITE = 1u,   // a deviation score was NaN/Inf (or negative)
  ERRBIT_INDEX = 2u,       // an index or position fell outside its buffer
  ERRBIT_TIMEOUT = 4u,     // a bounded device wait gave up
};

// GEMM epilogues.  The GEMM computes acc[m][n] = sum_k A[m][k] * B[n][k] (B = weight rows,
// output-major), then hands groups of consecutive columns of one row to the epilogue.
enum EpiKind {
  EPI_STORE = 0,   // out[m][n] = acc
  EPI_RESID = 1,   // out[m][n] = acc + resid[m][n]
  EPI_QKV = 2,     // column n + col0 of the fused Wqkv: q | k | v segments, RoPE on q, k
  EPI_SWIGLU = 3,  // out[m][j] = silu(gate_j) * up_j  (tensor-core path only)
};

struct EpiParams {
  int kind = EPI_STORE;
  void* out = nullptr;
  int64_t ldo = 0;
  const void* resid = nullptr;
  int64_t ldr = 0;
  const int32_t* resid_row = nullptr;  // EPI_RESID: row of resid added to output row m, or null (m)
  int64_t resid_rows = -1;             // rows of resid for the check of resid_row (< 0: unchecked)
  // EPI_QKV
  int col0 = 0;        // first Wqkv row covered by this launch
  int q_cols = 0;      // H * hd
  int kv_cols = 0;     // Hkv * hd
  int hd = 0;
  void* q = nullptr;   // [M, q_cols]
  int64_t ldq = 0;
  void* k = nullptr;   // rows kv_row[m] (or m) of [*, kv_cols]
  void* v = nullptr;
  int64_t ldkv = 0;
  const int32_t* pos = nullptr;     // [M] RoPE position per row
  const int32_t* kv_row = nullptr;  // [M] destination row of k/v, or null
  int64_t kv_bound = -1;            // rows of k/v for the check of kv_row (< 0: unchecked)
  const float* rope = nullptr;      // cos/sin table [max_pos][hd/2][2]
  int max_pos = 0;
  // EPI_QKV on the tensor-core path: squared deviation of the (bf16-rounded) K/V columns
  // from the cached rows, one partial per output row and half of a BN-column tile (BN the
  // launch's tile width, gemm_tc_tile_n)
  float* dev_part = nullptr;        // [2 * ceil(N / BN)][dev_ld]
  int64_t dev_ld = 0;
  const void* k_ref = nullptr;      // rows ref_row[m] (or m) of [ref_rows, kv_cols]
  const void* v_ref = nullptr;
  const int32_t* ref_row = nullptr;
  int64_t ref_rows = 0;
  int dev_use_v = 1;
  // A fused RMSNorm (tensor-core path, unit gains).  Producer (EPI_RESID): each warp writes
  // the sum of squares of its stored (bf16) output values of row m over its half of the tile
  // to ssq_out[(tile * 2 + half) * ssq_ld + m].  Consumer: its A operand holds the rows
  // before the norm; row m's accumulator is multiplied by
  // 1 / sqrt(sum_{p < rs_parts} rs_in[p * rs_ld + m] * rs_inv_d + rs_eps) first.
  float* ssq_out = nullptr;
  int64_t ssq_ld = 0;
  const float* rs_in = nullptr;
  const int32_t* rs_row = nullptr;  // row of rs_in's statistics for output row m, or null (m)
  int rs_parts = 0;
  int64_t rs_ld = 0;
  float rs_inv_d = 0.f;
  float rs_eps = 0.f;
};

constexpr int kGemmTileN = 256;     // widest tensor-core GEMM tile (output columns)
constexpr int kGemmTileNMinDev = 192;   // narrowest tile a fused-deviation launch takes

struct GemmDesc {
  int M = 0, N = 0, K = 0;
  const void* A = nullptr;  // [M, K], row stride lda elements
  int64_t lda = 0;
  const void* B = nullptr;  // [N, K] rows, stride ldb elements
  int64_t ldb = 0;
  int64_t b_up_row = 0;     // EPI_SWIGLU: row of B holding the 'up' partner of row 0
  EpiParams epi;
};

// ---- cb_gemm_tc.cu --------------------------------------------------------------------
// tile width (output columns) the tensor-core GEMM launch of these problems will use
int gemm_tc_tile_n(const GemmDesc* gs, int n);

// ---- cb_mem.cu ------------------------------------------------------------------------
cudaError_t launch_rope_table(float* tab, int max_pos, int hd, double base, cudaStream_t s);
cudaError_t launch_rope_shift(int dt, void* kd, void* vd, const void* ks, const void* vs,
                              const int32_t* src_row, int64_t n_src, const int32_t* delta,
                              int64_t n_rows, int W, int hd, const float* tab, int max_pos,
                              cudaStream_t s);
cudaError_t launch_kv_quantize(int dt, const void* x, int64_t n, int W, uint8_t* q, float* scale,
                               float* zero, cudaStream_t s);
cudaError_t launch_rope_shift_q8(int dt, void* kd, void* vd, const uint8_t* kq, const uint8_t* vq,
                                 const float* ks, const float* kz, const float* vs, const float* vz,
                                 const int32_t* src_row, int64_t n_src, const int32_t* qrow, int n_q,
                                 const int32_t* delta, int64_t n_rows, int W, int hd, const float* tab,
                                 int max_pos, cudaStream_t s);
cudaError_t launch_copy_rows(void* dst, const int32_t* dst_idx, const void* src,
                             const int32_t* src_idx, int64_t n, int64_t row_bytes,
                             int64_t dst_bound, int64_t src_bound, cudaStream_t s);
// rows index x; n_src is x's row count for the index check (< 0: unchecked)
cudaError_t launch_rmsnorm(int dt_in, int dt_out, void* out, const void* x,
                           const int32_t* rows, int64_t n_src, const void* g, int64_t n, int d,
                           float eps, cudaStream_t s);
cudaError_t launch_dev_reduce(const float* part, int part_lo, int n_parts, int64_t ld, int n_cand,
                              const int32_t* cand_pos, float* scores, cudaStream_t s);
constexpr int kMaxCopyJobs = 4;
struct CopyJobs {          // row copies of 16-byte words: dst[di[r]] = src[si[r]] (null index: r)
  void* dst[kMaxCopyJobs];
  const void* src[kMaxCopyJobs];
  const int32_t* di[kMaxCopyJobs];
  const int32_t* si[kMaxCopyJobs];
  int64_t rv[kMaxCopyJobs];       // 16-byte words per row
  int64_t dbound[kMaxCopyJobs];   // row bounds for the index checks (< 0: unchecked)
  int64_t sbound[kMaxCopyJobs];
  int64_t row_end[kMaxCopyJobs];  // inclusive prefix sums of the jobs' row counts
  int n;
};
// beside = true: small low-register blocks for a copy that runs beside a GEMM on another stream
cudaError_t launch_copy_rows_multi(const CopyJobs& J, cudaStream_t s, bool beside = false);
cudaError_t launch_wait_selftest(uint32_t max_polls, int arrive, cudaStream_t s);
cudaError_t launch_split_rows(const int32_t* rows_in, int m, const uint8_t* mask, int64_t mask_len,
                              int n_forced, int32_t* cand_pos, int32_t* cand_rows, int32_t* forced_pos,
                              int32_t* forced_rows, cudaStream_t s);
cudaError_t launch_merge_sel(const int32_t* ord, int k, const int32_t* cand_rows, const int32_t* cand_pos,
                             const int32_t* forced_rows, const int32_t* forced_pos, int nf, int32_t* s_out,
                             int32_t* keep_out, cudaStream_t s);
// n_new / n_ref: row counts of the new and cached K/V for the index checks (< 0: unchecked)
cudaError_t launch_deviation(int dt, const void* kn, const void* vn, const void* kr,
                             const void* vr, const int32_t* new_row, const int32_t* ref_row,
                             int n_cand, int64_t n_new, int64_t n_ref, int W, int use_v,
                             float* scores, cudaStream_t s);
cudaError_t launch_topk(const float* scores, int n, int k, int32_t* out_ord, cudaStream_t s);
// top-k fused with the selection build of the default layout (see launch_build_sel)
cudaError_t launch_topk_sel(const float* scores, int n, int k, const int32_t* cand_row, int32_t forced_row0,
                            int32_t forced_pos0, int n_forced, int32_t* s_out, int32_t* keep_out, cudaStream_t s);
cudaError_t launch_map_rows(const int32_t* ord, int k, const int32_t* map, int32_t* out,
                            cudaStream_t s);
cudaError_t launch_build_sel(const int32_t* ord, int k, const int32_t* cand_row,
                             int32_t forced_row0, int32_t forced_pos0, int n_forced,
                             int32_t* s_out, int32_t* keep_out, cudaStream_t s);
cudaError_t launch_rows_to_positions(const int32_t* rows, int k, const int32_t* s_in, int m_in,
                                     int32_t* pos_out, cudaStream_t s);
cudaError_t launch_iota(int32_t* out, int n, int32_t start, cudaStream_t s);
// row offsets of the requests of a batched steady layer (request r owns rows [row0[r], row0[r+1]))
constexpr int kMaxBatch = 64;
struct BatchRows {
  int32_t row0[kMaxBatch + 1];
  int n_req;
};
cudaError_t launch_batch_kv_rows(const int32_t* s_in, int m_total, int64_t n_tok, const BatchRows& b,
                                 int32_t* kv_row, cudaStream_t s);
cudaError_t launch_swiglu(int dt, void* out, const void* gu, int64_t M, int F, cudaStream_t s);
size_t lm_block_best_count(int V);          // workspace entries (either type)
size_t lm_block_count(int V, int dt);       // entries the GEMV of this type writes
cudaError_t launch_lm_gemv(int dt, float* logits, const float* hn, const void* w, int V, int d,
                           unsigned long long* block_best, cudaStream_t s);
cudaError_t launch_argmax_keys(const unsigned long long* keys, int n, int32_t* token, cudaStream_t s);
uint32_t take_error_mem();
int noalloc_max_candidates();
cudaError_t launch_deviation_topk_noalloc(int dt, const void* kn, const void* vn, const void* kr,
                                          const void* vr, const int32_t* new_row,
                                          const int32_t* ref_row, int n_cand, int64_t n_new,
                                          int64_t n_ref, int k, int W, int use_v, float* scores,
                                          int32_t* sel, cudaStream_t s);
// empty the host-side per-device caches of each translation unit (cb_shutdown)
void reset_mem_caches();
void reset_gemm_tc_caches();
void reset_attn_tc_caches();

// ---- cb_gemm.cu -----------------------------------------------------------------------
// The span slot of the launch being made by this thread (span profiling on), else NULL.
unsigned long long* prof_span_slot();
cudaError_t launch_gemm(int dt, const GemmDesc& g, cudaStream_t s);
cudaError_t launch_gemm_pair(int dt, const GemmDesc& a, const GemmDesc& b, cudaStream_t s);
uint32_t take_error_gemm();

// ---- cb_attn.cu -----------------------------------------------------------------------
size_t attention_ws_bytes(int dt, int64_t M, int H, int hd);
cudaError_t launch_attention(int dt, const void* q, const int32_t* q_pos, int M,
                             const void* kc, const void* vc, int64_t n_kv, int H, int Hkv,
                             int hd, void* out, void* ws, size_t ws_bytes, cudaStream_t s);
uint32_t take_error_attn();

}  // namespace cb
