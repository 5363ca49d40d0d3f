// C ABI of the selective-KV-recompute library: host-side validation, workspace carving and
// the per-layer orchestration of the kernels.  Every argument check happens before the first
// launch, so a call that returns an error has enqueued nothing.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <time.h>

#include <algorithm>
#include <atomic>
#include <initializer_list>
#include <vector>

#include "../../include/cacheblend.h"
#include "cb_internal.h"

namespace cb {
uint32_t take_error_gemm_tc();
uint32_t take_error_attn_tc();
}  // namespace cb

using namespace cb;

namespace {

thread_local char g_msg[512] = "";
thread_local char g_cuda_msg[256] = "";   // the last failing CUDA call on this thread

// records a failing CUDA call for cb_last_cuda_error
void note_cuda(cudaError_t e, const char* what) {
  snprintf(g_cuda_msg, sizeof(g_cuda_msg), "%s (%s): %s", cudaGetErrorName(e), cudaGetErrorString(e), what);
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

#define CB_CUDA(expr)                                                                    \
  do {                                                                                   \
    cudaError_t e__ = (expr);                                                            \
    if (e__ != cudaSuccess) {                                                            \
      note_cuda(e__, #expr);                                                             \
      return fail(CB_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e__));         \
    }                                                                                    \
  } while (0)

inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

// ---- launch accounting and optional per-launch CUDA-event timing (calling thread only)
std::atomic<long long> g_launches{0};

struct ProfState {
  bool on = false;
  bool spans = false;                 // span mode: kernel-side timestamps instead of events
  int cap = 0;
  std::vector<cudaEvent_t> ev;        // 2 per record, created once and reused
  std::vector<cb_prof_record> rec;
  unsigned long long* span_base = nullptr;
};
thread_local ProfState g_prof;

// span slots: two words per record (earliest start, latest end; %globaltimer ns)
constexpr int kSpanMax = 8192;
__device__ unsigned long long g_span_buf[2 * kSpanMax];
thread_local unsigned long long* g_cur_span = nullptr;
std::atomic<bool> g_span_taken{false};   // the slot buffer serves one host thread at a time

struct ProfScope {
  int idx = -1;
  cudaStream_t s;
  ProfScope(int kind, int aux, int64_t m, int64_t n, int64_t k, double flops, double bytes, cudaStream_t st)
      : s(st) {
    if (m <= 0) return;          // the launcher returns without launching
    g_launches.fetch_add(1, std::memory_order_relaxed);
    ProfState& P = g_prof;
    if (!P.on || (int)P.rec.size() >= P.cap) return;
    idx = (int)P.rec.size();
    cb_prof_record r{};
    r.kind = kind;
    r.aux = aux;
    r.m = m;
    r.n = n;
    r.k = k;
    r.flops = flops;
    r.bytes = bytes;
    P.rec.push_back(r);
    if (P.spans)
      g_cur_span = P.span_base + 2 * idx;
    else
      cudaEventRecord(P.ev[2 * idx], s);
  }
  ~ProfScope() {
    if (idx < 0) return;
    if (g_prof.spans)
      g_cur_span = nullptr;
    else
      cudaEventRecord(g_prof.ev[2 * idx + 1], s);
  }
};

// wraps one kernel launch: counts it and, when profiling, brackets it with events
#define CB_LAUNCH(kind, aux, m, n, k, flops, bytes, stream, expr)         \
  do {                                                                    \
    ProfScope ps__(kind, aux, m, n, k, flops, bytes, stream);             \
    CB_CUDA(expr);                                                        \
  } while (0)

inline size_t esize(int dt) { return dt == CB_BF16 ? 2 : 4; }

double gemm_flops(const GemmDesc& g) {
  return 2.0 * g.M * g.N * g.K * (g.epi.kind == EPI_SWIGLU ? 2 : 1);
}
// compulsory HBM traffic of one GEMM launch: A, B (both halves for SwiGLU), C (+ residual)
double gemm_bytes(int dt, const GemmDesc& g) {
  const double B = (double)esize(dt);
  const double nb = (g.epi.kind == EPI_SWIGLU ? 2.0 : 1.0) * g.N;
  double b = B * ((double)g.M * g.K + nb * g.K + (double)g.M * g.N);
  if (g.epi.kind == EPI_RESID) b += B * (double)g.M * g.N;
  return b;
}

#define L_GEMM(dt, gexpr, s)                                                                  \
  do {                                                                                        \
    const GemmDesc g__ = (gexpr);                                                             \
    CB_LAUNCH(CB_PROF_GEMM, g__.epi.kind, g__.M, g__.N, g__.K, gemm_flops(g__), gemm_bytes(dt, g__), s, \
              launch_gemm(dt, g__, s));                                                       \
  } while (0)
#define L_GEMM2(dt, ga, gb, s)                                                                   \
  do {                                                                                        \
    const GemmDesc a__ = (ga), b__ = (gb);                                                    \
    CB_LAUNCH(CB_PROF_GEMM, 100 + a__.epi.kind, a__.M + b__.M, a__.N, a__.K,                  \
              gemm_flops(a__) + gemm_flops(b__), gemm_bytes(dt, a__) + gemm_bytes(dt, b__), s,  \
              launch_gemm_pair(dt, a__, b__, s));                                             \
  } while (0)
#define L_IOTA(out, n, start, s) \
  CB_LAUNCH(CB_PROF_INDEX, 0, (n), 0, 0, 0.0, 4.0 * (n), s, launch_iota(out, n, start, s))
#define L_RMSNORM(dti, dto, out, x, rows, g, n, d, eps, s) L_RMSNORM_B(dti, dto, out, x, rows, -1, g, n, d, eps, s)
#define L_RMSNORM_B(dti, dto, out, x, rows, nsrc, g, n, d, eps, s)                               \
  CB_LAUNCH(CB_PROF_RMSNORM, 0, (n), (d), 0, 3.0 * (n) * (d),                                    \
            (double)(n) * (d) * (esize(dti) + esize(dto)), s,                                    \
            launch_rmsnorm(dti, dto, out, x, rows, nsrc, g, n, d, eps, s))
#define L_ATTN(dt, q, qpos, M, kc, vc, nkv, H, Hkv, hd, out, ws, wsb, s)                         \
  CB_LAUNCH(CB_PROF_ATTENTION, 0, (M), (nkv), (H), 0.0, 0.0, s,                                  \
            launch_attention(dt, q, qpos, M, kc, vc, nkv, H, Hkv, hd, out, ws, wsb, s))
#define L_COPY(dst, di, src, si, n, rb, db, sb, s)                                               \
  CB_LAUNCH(CB_PROF_COPY_ROWS, 0, (n), (rb), 0, 0.0, 2.0 * (n) * (rb), s,                        \
            launch_copy_rows(dst, di, src, si, n, rb, db, sb, s))
#define L_DEV(dt, kn, vn, kr, vr, nr, rr, nc, nnew, nref, W, usev, sc, s)                       \
  CB_LAUNCH(CB_PROF_DEVIATION, 0, (nc), (W), (usev), 3.0 * (nc) * (W) * ((usev) ? 2 : 1),        \
            (double)(nc) * (W) * esize(dt) * ((usev) ? 4 : 2) + 4.0 * (nc), s,                   \
            launch_deviation(dt, kn, vn, kr, vr, nr, rr, nc, nnew, nref, W, usev, sc, s))
#define L_DEVRED(part, plo, np, ld, nc, cpos, W, usev, sc, s)                                    \
  CB_LAUNCH(CB_PROF_DEVIATION, 1, (nc), (W), (usev), (double)(nc) * ((np) - (plo)),                 \
            4.0 * (nc) * ((np) - (plo) + 1), s, launch_dev_reduce(part, plo, np, ld, nc, cpos, sc, s))
#define L_SPLIT(rows, m, mask, mlen, nf, cp, cr, fp, fr, s)                                      \
  CB_LAUNCH(CB_PROF_INDEX, 1, (m), 0, 0, 0.0, 21.0 * (m), s,                                      \
            launch_split_rows(rows, m, mask, mlen, nf, cp, cr, fp, fr, s))
#define L_MERGE(ord, k, cr, cp, fr, fp, nf, so, ko, s)                                           \
  CB_LAUNCH(CB_PROF_INDEX, 2, (k) + (nf), 0, 0, 0.0, 16.0 * ((k) + (nf)), s,                     \
            launch_merge_sel(ord, k, cr, cp, fr, fp, nf, so, ko, s))
#define L_TOPK(sc, n, k, ord, s) \
  CB_LAUNCH(CB_PROF_TOPK, 0, (n), (k), 0, 0.0, 4.0 * (n) + 4.0 * (k), s, launch_topk(sc, n, k, ord, s))
#define L_MAP(ord, k, map, out, s) \
  CB_LAUNCH(CB_PROF_INDEX, 0, (k), 0, 0, 0.0, 12.0 * (k), s, launch_map_rows(ord, k, map, out, s))
#define L_TOPK_SEL(sc, n, k, cr, f0, fp0, nf, so, ko, s)                                          \
  CB_LAUNCH(CB_PROF_TOPK, 0, (n), (k), 0, 0.0, 4.0 * (n) + 8.0 * ((k) + (nf)), s,                \
            launch_topk_sel(sc, n, k, cr, f0, fp0, nf, so, ko, s))
#define L_BUILD_SEL(ord, k, cr, f0, fp0, nf, so, ko, s)                                          \
  CB_LAUNCH(CB_PROF_INDEX, 0, (k) + (nf), 0, 0, 0.0, 16.0 * ((k) + (nf)), s,                     \
            launch_build_sel(ord, k, cr, f0, fp0, nf, so, ko, s))
#define L_R2P(rows, k, sin, m, out, s) \
  CB_LAUNCH(CB_PROF_INDEX, 0, (k), 0, 0, 0.0, 8.0 * (k), s, launch_rows_to_positions(rows, k, sin, m, out, s))
#define L_ROPE_SHIFT(dt, kd, vd, ks, vs, sr, nsrc, dl, n, W, hd, tab, mp, s)                     \
  CB_LAUNCH(CB_PROF_ROPE_SHIFT, 0, (n), (W), 0, 3.0 * (n) * (W),                                 \
            (double)(n) * (W) * esize(dt) * ((vd) ? 4 : 2) + 4.0 * (n), s,                       \
            launch_rope_shift(dt, kd, vd, ks, vs, sr, nsrc, dl, n, W, hd, tab, mp, s))
#define L_LMGEMV(dt, lg, hn, w, V, d, bb, s)                                                     \
  CB_LAUNCH(CB_PROF_LMHEAD, 0, (V), (d), 0, 2.0 * (V) * (d), (double)(V) * (d) * esize(dt) + 4.0 * (V), s, \
            launch_lm_gemv(dt, lg, hn, w, V, d, bb, s))
#define L_ARGMAX(bb, n, tok, s) \
  CB_LAUNCH(CB_PROF_ARGMAX, 0, (n), 0, 0, 0.0, 8.0 * (n), s, launch_argmax_keys(bb, n, tok, s))
#define L_ROPE_TABLE(tab, mp, hd, base, s)                                                       \
  CB_LAUNCH(CB_PROF_ROPE_TABLE, 0, (int64_t)(mp) * (hd) / 2, (hd), 0, 0.0, 4.0 * (mp) * (hd), s, \
            launch_rope_table(tab, mp, hd, base, s))

int check_dims(const cb_dims* d) {
  if (!d) return fail(CB_ERR_INVALID_ARG, "dims is NULL");
  if (d->dtype != CB_F32 && d->dtype != CB_BF16) return fail(CB_ERR_DTYPE, "dtype %d", d->dtype);
  if (d->d_model <= 0 || d->n_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 || d->d_ff <= 0 ||
      d->vocab <= 0)
    return fail(CB_ERR_SHAPE, "non-positive dimension");
  if (d->n_heads % d->n_kv_heads) return fail(CB_ERR_SHAPE, "n_heads %% n_kv_heads != 0");
  if (d->head_dim % 32 || d->head_dim > 256)
    return fail(CB_ERR_UNSUPPORTED, "head_dim must be a multiple of 32, at most 256");
  if (d->d_model % 16 || d->d_ff % 16)
    return fail(CB_ERR_UNSUPPORTED, "d_model and d_ff must be multiples of 16");
  if (!(d->rope_base > 1.0) || !(d->rms_eps >= 0.0f)) return fail(CB_ERR_INVALID_ARG, "rope_base/rms_eps");
  return CB_OK;
}

// A source the kernels read may live in pinned host memory (zero-copy over the host link)
// only if that memory is mapped into the device address space at the same address.
int check_readable(const void* p, const char* what) {
  if (!p) return CB_OK;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return fail(CB_ERR_INVALID_ARG, "%s: not a CUDA-visible pointer", what);
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return CB_OK;
  if (a.type == cudaMemoryTypeHost && a.devicePointer == p) return CB_OK;
  return fail(CB_ERR_INVALID_ARG, "%s: host memory not mapped at the same device address", what);
}

// Device buffers that kernels read or write in 16-byte vectors (activation rows, KV caches,
// weights, tables, workspaces) must start on a 16-byte boundary; every row width the library
// accepts keeps later rows on one.  A misaligned base is refused here, before any launch,
// rather than faulting on the GPU.  NULL entries (optional buffers) pass.
int check_al16(std::initializer_list<const void*> ps, const char* what) {
  for (const void* p : ps)
    if (reinterpret_cast<uintptr_t>(p) & 15) return fail(CB_ERR_INVALID_ARG, "%s: buffer not 16-byte aligned", what);
  return CB_OK;
}

// the norm gains may be NULL (unit gains); the matrices may not
int check_w(const cb_layer_w* w) {
  if (!w || !w->wqkv || !w->wo || !w->w_gate_up || !w->w_down)
    return fail(CB_ERR_INVALID_ARG, "layer weight pointer is NULL");
  if (int st = check_al16({w->attn_norm, w->wqkv, w->wo, w->ffn_norm, w->w_gate_up, w->w_down}, "layer weights"))
    return st;
  return CB_OK;
}

// bump allocator over the caller's workspace; base == nullptr measures only
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

struct LayerWs {
  void *a, *q, *knew, *vnew, *attn, *h, *b, *act, *ag, *qg, *xa, *xb, *attn_ws;
  float *scores, *hn, *logits, *dev_part, *ssq;
  int32_t *ord, *keep, *pos, *rows, *cpos, *crows, *fpos, *frows;
};

// deviation partials per row of a GEMM over ncols Wqkv columns in tiles of bn columns: one
// per half tile (the workspace holds enough for the narrowest tile)
int dev_parts(int ncols, int bn = kGemmTileNMinDev) { return 2 * ((ncols + bn - 1) / bn); }
int qkv_cols(const cb_dims* d) { return (d->n_heads + 2 * d->n_kv_heads) * d->head_dim; }

// R = rows entering the layer, M = rows selected (M <= R)
LayerWs carve_layer(Carver& c, const cb_dims* d, int64_t R, int64_t M) {
  const size_t B = esize(d->dtype);
  const int64_t qc = (int64_t)d->n_heads * d->head_dim, W = (int64_t)d->n_kv_heads * d->head_dim;
  LayerWs w{};
  w.a = c.take(R * d->d_model * B);
  w.q = c.take(std::max(R, M) * qc * B);
  w.knew = c.take(R * W * B);
  w.vnew = c.take(R * W * B);
  w.attn = c.take(std::max(R, M) * qc * B);
  w.h = c.take(std::max(R, M) * d->d_model * B);
  w.b = c.take(std::max(R, M) * d->d_model * B);
  w.act = c.take(std::max(R, M) * d->d_ff * B);
  w.ag = c.take(M * d->d_model * B);
  w.xa = c.take(R * d->d_model * B);
  w.xb = c.take(R * d->d_model * B);
  w.scores = static_cast<float*>(c.take(R * 4));
  w.dev_part = static_cast<float*>(c.take((size_t)dev_parts(qkv_cols(d)) * R * 4));
  w.ssq = static_cast<float*>(c.take((size_t)dev_parts(d->d_model) * std::max(R, M) * 4));
  w.qg = c.take(M * qc * B);
  w.ord = static_cast<int32_t*>(c.take(R * 4));
  w.keep = static_cast<int32_t*>(c.take(R * 4));
  w.pos = static_cast<int32_t*>(c.take(R * 4));
  w.rows = static_cast<int32_t*>(c.take(R * 4));
  w.cpos = static_cast<int32_t*>(c.take(R * 4));
  w.crows = static_cast<int32_t*>(c.take(R * 4));
  w.fpos = static_cast<int32_t*>(c.take(R * 4));
  w.frows = static_cast<int32_t*>(c.take(R * 4));
  w.hn = static_cast<float*>(c.take(d->d_model * 4));
  w.logits = static_cast<float*>(c.take((size_t)d->vocab * 4));
  const size_t aw = attention_ws_bytes(d->dtype, std::max(R, M), d->n_heads, d->head_dim);
  w.attn_ws = c.take(aw);
  return w;
}

size_t layer_ws_bytes(const cb_dims* d, int64_t R, int64_t M) {
  Carver c(nullptr);
  carve_layer(c, d, R, M);
  return c.off + 256;
}

int need_ws(const cb_dims* d, int64_t R, int64_t M, void* ws, size_t ws_bytes, LayerWs* out) {
  const size_t need = layer_ws_bytes(d, R, M);
  if (!ws) return fail(CB_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (ws_bytes < need) return fail(CB_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  Carver c(ws);
  *out = carve_layer(c, d, R, M);
  return CB_OK;
}

// Row copies batched into one launch when every row is a whole number of 16-byte words
// at 16-byte aligned bases; otherwise one launch per copy.
struct RowCopies {
  CopyJobs J{};
  struct One { void* d; const int32_t* di; const void* src; const int32_t* si; int64_t n, rb, db, sb; };
  One list[kMaxCopyJobs];
  int n = 0;
  void add(void* d, const int32_t* di, const void* src, const int32_t* si, int64_t rows, int64_t rb, int64_t db,
           int64_t sb) {
    list[n++] = One{d, di, src, si, rows, rb, db, sb};
  }
  int launch(cudaStream_t s, bool beside = false) {
    bool vec = true;
    int64_t acc = 0, bytes = 0, rows = 0;
    int m = 0;
    for (int i = 0; i < n; ++i) {
      const One& o = list[i];
      if (o.n == 0) continue;
      vec = vec && o.rb % 16 == 0 && ((uintptr_t)o.d & 15) == 0 && ((uintptr_t)o.src & 15) == 0;
      J.dst[m] = o.d;
      J.src[m] = o.src;
      J.di[m] = o.di;
      J.si[m] = o.si;
      J.rv[m] = o.rb / 16;
      J.dbound[m] = o.db;
      J.sbound[m] = o.sb;
      acc += o.n;
      J.row_end[m] = acc;
      bytes += 2 * o.n * o.rb;
      rows += o.n;
      ++m;
    }
    J.n = m;
    if (m == 0) return CB_OK;
    if (!vec) {
      for (int i = 0; i < n; ++i) {
        const One& o = list[i];
        L_COPY(o.d, o.di, o.src, o.si, o.n, o.rb, o.db, o.sb, s);
      }
      return CB_OK;
    }
    CB_LAUNCH(CB_PROF_COPY_ROWS, m, rows, 0, 0, 0.0, (double)bytes, s, launch_copy_rows_multi(J, s, beside));
    return CB_OK;
  }
};

GemmDesc make_gemm(int M, int N, int K, const void* A, int64_t lda, const void* B, int64_t ldb) {
  GemmDesc g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.A = A;
  g.lda = lda;
  g.B = B;
  g.ldb = ldb;
  return g;
}

// Q/K/V GEMM over columns [col0, col0 + ncols) of Wqkv for M rows of normalised input a.
GemmDesc qkv_desc(const cb_dims* d, const cb_layer_w* w, const void* a, int M, int col0, int ncols, void* q,
                  void* k, void* v, const int32_t* pos, const int32_t* kv_row, const float* tab, int max_pos) {
  const size_t B = esize(d->dtype);
  const int qc = d->n_heads * d->head_dim, W = d->n_kv_heads * d->head_dim;
  GemmDesc g = make_gemm(M, ncols, d->d_model, a, d->d_model,
                         static_cast<const char*>(w->wqkv) + (size_t)col0 * d->d_model * B, d->d_model);
  g.epi.kind = EPI_QKV;
  g.epi.col0 = col0;
  g.epi.q_cols = qc;
  g.epi.kv_cols = W;
  g.epi.hd = d->head_dim;
  g.epi.q = q;
  g.epi.ldq = qc;
  g.epi.k = k;
  g.epi.v = v;
  g.epi.ldkv = W;
  g.epi.pos = pos;
  g.epi.kv_row = kv_row;
  g.epi.rope = tab;
  g.epi.max_pos = max_pos;
  return g;
}

// h = x_res[res_row[m]] + attn Wo^T ; x_out = h + (silu(b Wg^T) * b Wu^T) Wd^T, b = RMSNorm(h) g.
// res_row null: row m of x_res; otherwise rows of x_res (res_rows of them) read in place, so the
// residual rows of a selection need no gather.
// x_ssq / x_ssq_parts_host (optional): the bf16 path writes each x_out row's partial sums
// of squares there (for the next layer's norm) and their count on the host.
int o_ffn(const cb_dims* d, const cb_layer_w* w, const void* attn, const void* x_res, int M, void* x_out,
          const LayerWs& ws, cudaStream_t s, const int32_t* res_row = nullptr, int64_t res_rows = -1,
          float* x_ssq = nullptr, int32_t* x_ssq_parts_host = nullptr) {
  if (M == 0) return CB_OK;
  const int qc = d->n_heads * d->head_dim;
  // with unit FFN-norm gains (ffn_norm NULL) the bf16 path folds the norm into the GEMMs:
  // the O-projection leaves each row's partial sums of squares of h, the gate/up GEMM reads h
  // itself and scales its rows by 1/rms in the epilogue (no separate norm pass)
  const bool fuse = d->dtype == CB_BF16 && w->ffn_norm == nullptr;
  GemmDesc go = make_gemm(M, d->d_model, qc, attn, qc, w->wo, qc);
  go.epi.kind = EPI_RESID;
  go.epi.out = ws.h;
  go.epi.ldo = d->d_model;
  go.epi.resid = x_res;
  go.epi.ldr = d->d_model;
  go.epi.resid_row = res_row;
  go.epi.resid_rows = res_rows;
  if (fuse) {
    go.epi.ssq_out = ws.ssq;
    go.epi.ssq_ld = M;
  }
  L_GEMM(d->dtype, go, s);
  if (!fuse) L_RMSNORM(d->dtype, d->dtype, ws.b, ws.h, nullptr, w->ffn_norm, M, d->d_model, d->rms_eps, s);
  GemmDesc gu = make_gemm(M, d->d_ff, d->d_model, fuse ? ws.h : ws.b, d->d_model, w->w_gate_up, d->d_model);
  gu.b_up_row = d->d_ff;
  gu.epi.kind = EPI_SWIGLU;
  gu.epi.out = ws.act;
  gu.epi.ldo = d->d_ff;
  if (fuse) {
    gu.epi.rs_in = ws.ssq;
    gu.epi.rs_parts = dev_parts(d->d_model, gemm_tc_tile_n(&go, 1));
    gu.epi.rs_ld = M;
    gu.epi.rs_inv_d = 1.0f / (float)d->d_model;
    gu.epi.rs_eps = d->rms_eps;
  }
  L_GEMM(d->dtype, gu, s);
  GemmDesc gd = make_gemm(M, d->d_model, d->d_ff, ws.act, d->d_ff, w->w_down, d->d_ff);
  gd.epi.kind = EPI_RESID;
  gd.epi.out = x_out;
  gd.epi.ldo = d->d_model;
  gd.epi.resid = ws.h;
  gd.epi.ldr = d->d_model;
  const bool stats = d->dtype == CB_BF16 && x_ssq != nullptr;
  if (stats) {
    gd.epi.ssq_out = x_ssq;
    gd.epi.ssq_ld = M;
  }
  if (x_ssq_parts_host) *x_ssq_parts_host = stats ? dev_parts(d->d_model, gemm_tc_tile_n(&gd, 1)) : 0;
  L_GEMM(d->dtype, gd, s);
  return CB_OK;
}

double now_s() {
  timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec + 1e-9 * ts.tv_nsec;
}

}  // namespace

namespace cb {
unsigned long long* prof_span_slot() { return g_cur_span; }
}  // namespace cb

extern "C" {

const char* cb_status_string(int status) {
  switch (status) {
    case CB_OK: return "ok";
    case CB_ERR_INVALID_ARG: return "invalid argument";
    case CB_ERR_SHAPE: return "inconsistent shape";
    case CB_ERR_DTYPE: return "unsupported dtype";
    case CB_ERR_WORKSPACE: return "workspace too small";
    case CB_ERR_NONFINITE: return "non-finite deviation score";
    case CB_ERR_CUDA: return "CUDA error";
    case CB_ERR_TIMEOUT: return "timed out";
    case CB_ERR_UNSUPPORTED: return "unsupported shape";
    case CB_ERR_DEVICE: return "device-side index or wait error";
    case CB_ERR_IO: return "storage read failed";
    default: return "unknown status";
  }
}

const char* cb_last_error_message(void) { return g_msg; }

const char* cb_last_cuda_error(void) { return g_cuda_msg; }

int cb_sync(void* stream, double timeout_s) {
  const double t0 = now_s();
  for (;;) {
    cudaError_t e = cudaStreamQuery(S(stream));
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) {
      note_cuda(e, "cudaStreamQuery");
      return fail(CB_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
    }
    if (timeout_s > 0 && now_s() - t0 > timeout_s)
      return fail(CB_ERR_TIMEOUT, "stream not idle after %.3f s", timeout_s);
    timespec ts{0, 50000};
    nanosleep(&ts, nullptr);
  }
  const uint32_t bits = take_error_mem() | take_error_gemm() | take_error_gemm_tc() | take_error_attn() |
                        take_error_attn_tc();
  if (bits & ERRBIT_NONFINITE) return fail(CB_ERR_NONFINITE, "a deviation score was NaN/Inf");
  if (bits & ERRBIT_INDEX) return fail(CB_ERR_DEVICE, "a kernel met an out-of-range index");
  if (bits & ERRBIT_TIMEOUT) return fail(CB_ERR_DEVICE, "a kernel's bounded wait expired");
  return CB_OK;
}

int cb_selftest_wait(int32_t max_polls, int32_t arrive, void* stream) {
  if (max_polls < 1 || max_polls > (1 << 20)) return fail(CB_ERR_INVALID_ARG, "max_polls outside [1, 2^20]");
  CB_CUDA(launch_wait_selftest((uint32_t)max_polls, arrive ? 1 : 0, S(stream)));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return CB_OK;
}

int cb_workspace_bytes(const cb_dims* dims, int64_t n_tok, int64_t m_max, size_t* out_host) {
  int st = check_dims(dims);
  if (st) return st;
  if (!out_host || n_tok < 1 || m_max < 0) return fail(CB_ERR_INVALID_ARG, "workspace query arguments");
  *out_host = layer_ws_bytes(dims, n_tok, std::max<int64_t>(m_max, n_tok));
  return CB_OK;
}

int64_t cb_hkvd_budget(int64_t n_cached, double ratio, int64_t n_cand) {
  if (n_cached < 0 || n_cand < 0 || !(ratio >= 0.0) || ratio > 1.0) return -1;
  if (ratio == 0.0) return 0;
  int64_t k = (int64_t)floor((double)n_cached * ratio);
  if (k < 1) k = 1;
  if (k > n_cand) k = n_cand;
  return k;
}

double cb_gradual_ratio(double r, int32_t layer, int32_t check_layer, double r1_factor) {
  if (layer < check_layer) return -1.0;
  const double r1 = std::min(1.0, r1_factor * r);
  return r + (r1 - r) * ldexp(1.0, -(layer - check_layer));
}

double cb_load_controller_ratio(double r_min, double t_load_s, double t_prefill_s) {
  if (!(t_prefill_s > 0.0)) return r_min;
  return std::max(r_min, t_load_s / t_prefill_s);
}

int cb_rope_table(float* cos_sin, int32_t max_pos, int32_t head_dim, double base, void* stream) {
  if (!cos_sin || max_pos < 1 || head_dim < 2 || head_dim % 2 || !(base > 1.0))
    return fail(CB_ERR_INVALID_ARG, "rope table arguments");
  L_ROPE_TABLE(cos_sin, max_pos, head_dim, base, S(stream));
  return CB_OK;
}

int cb_rope_shift(void* k_dst, void* v_dst, const void* k_src, const void* v_src, const int32_t* src_row,
                  int64_t n_src_rows, const int32_t* delta, int64_t n_rows, const cb_dims* dims,
                  const float* cos_sin, int32_t max_pos, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (n_rows < 0 || n_src_rows < 0) return fail(CB_ERR_SHAPE, "n_rows < 0 or n_src_rows < 0");
  if (n_rows == 0) return CB_OK;
  if (!src_row && n_src_rows < n_rows) return fail(CB_ERR_SHAPE, "n_src_rows < n_rows with src_row NULL");
  if (!k_dst || !k_src || !delta || !cos_sin || max_pos < 1)
    return fail(CB_ERR_INVALID_ARG, "rope_shift pointer is NULL");
  if ((v_dst == nullptr) != (v_src == nullptr)) return fail(CB_ERR_INVALID_ARG, "v_dst/v_src must both be set or NULL");
  if (k_dst == k_src && src_row) return fail(CB_ERR_INVALID_ARG, "in-place shift needs src_row == NULL");
  if ((st = check_al16({k_dst, v_dst, k_src, v_src, cos_sin}, "rope_shift"))) return st;
  if ((st = check_readable(k_src, "k_src")) || (st = check_readable(v_src, "v_src"))) return st;
  const int W = dims->n_kv_heads * dims->head_dim;
  L_ROPE_SHIFT(dims->dtype, k_dst, v_dst, k_src, v_src, src_row, n_src_rows, delta, n_rows, W, dims->head_dim, cos_sin,
               max_pos, S(stream));
  return CB_OK;
}

int cb_kv_quantize(const void* x, int64_t n_rows, int32_t W, int32_t dtype, uint8_t* codes, float* scale,
                   float* zero, void* stream) {
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_DTYPE, "dtype %d", dtype);
  if (n_rows < 0 || W < 1) return fail(CB_ERR_SHAPE, "need n_rows >= 0, W >= 1");
  if (n_rows == 0) return CB_OK;
  if (!x || !codes || !scale || !zero) return fail(CB_ERR_INVALID_ARG, "kv_quantize pointer is NULL");
  if (int st = check_al16({x, scale, zero}, "kv_quantize")) return st;
  if (reinterpret_cast<uintptr_t>(codes) & 7) return fail(CB_ERR_INVALID_ARG, "kv_quantize: codes not 8-byte aligned");
  CB_LAUNCH(CB_PROF_QUANT, 0, n_rows, W, 0, 0.0, (double)n_rows * W * (2.0 * esize(dtype) + 1.0) + 8.0 * W,
            S(stream), launch_kv_quantize(dtype, x, n_rows, W, codes, scale, zero, S(stream)));
  return CB_OK;
}

int cb_rope_shift_q8(void* k_dst, void* v_dst, const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scale,
                     const float* k_zero, const float* v_scale, const float* v_zero, const int32_t* src_row,
                     int64_t n_src_rows, const int32_t* qrow, int32_t n_qrows, const int32_t* delta, int64_t n_rows,
                     const cb_dims* dims, const float* cos_sin, int32_t max_pos, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (n_rows < 0 || n_src_rows < 0 || n_qrows < 0) return fail(CB_ERR_SHAPE, "negative size");
  if (n_rows == 0) return CB_OK;
  if (!k_dst || !k_codes || !k_scale || !k_zero || !qrow || !delta || !cos_sin || max_pos < 1)
    return fail(CB_ERR_INVALID_ARG, "rope_shift_q8 pointer is NULL");
  if ((v_dst == nullptr) != (v_codes == nullptr) || (v_dst && (!v_scale || !v_zero)))
    return fail(CB_ERR_INVALID_ARG, "v_dst, v_codes, v_scale, v_zero must all be set or all NULL");
  if (!src_row && n_src_rows < n_rows) return fail(CB_ERR_SHAPE, "n_src_rows < n_rows with src_row NULL");
  const uintptr_t a = (uintptr_t)k_codes | (uintptr_t)v_codes;
  const uintptr_t b = (uintptr_t)k_scale | (uintptr_t)k_zero | (uintptr_t)v_scale | (uintptr_t)v_zero;
  if ((a & 7) || (b & 15)) return fail(CB_ERR_INVALID_ARG, "codes need 8-byte, scale/zero 16-byte alignment");
  if ((st = check_al16({k_dst, v_dst, cos_sin}, "rope_shift_q8"))) return st;
  if ((st = check_readable(k_codes, "k_codes")) || (st = check_readable(v_codes, "v_codes"))) return st;
  const int W = dims->n_kv_heads * dims->head_dim;
  const double bytes = (double)n_rows * W * ((v_dst ? 2.0 : 1.0) * (1.0 + esize(dims->dtype))) + 4.0 * n_rows;
  CB_LAUNCH(CB_PROF_ROPE_SHIFT, 1, n_rows, W, 0, 3.0 * n_rows * W, bytes, S(stream),
            launch_rope_shift_q8(dims->dtype, k_dst, v_dst, k_codes, v_codes, k_scale, k_zero, v_scale, v_zero, src_row,
                                 n_src_rows, qrow, n_qrows, delta, n_rows, W, dims->head_dim, cos_sin, max_pos,
                                 S(stream)));
  return CB_OK;
}

// row counts of the new and cached K/V: with a row map every index is checked on the device;
// without one the candidates are rows 0..n_cand-1, which must exist
int check_dev_rows(const int32_t* new_row, const int32_t* ref_row, int32_t n_cand, int64_t n_new_rows,
                   int64_t n_ref_rows) {
  if (n_new_rows < 0 || n_ref_rows < 0) return fail(CB_ERR_SHAPE, "negative row count");
  if ((!new_row && n_new_rows < n_cand) || (!ref_row && n_ref_rows < n_cand))
    return fail(CB_ERR_SHAPE, "fewer rows than candidates without a row map");
  return CB_OK;
}

int cb_kv_deviation_topk(const void* k_new, const void* v_new, int64_t n_new_rows, const void* k_ref,
                         const void* v_ref, int64_t n_ref_rows, const int32_t* new_row, const int32_t* ref_row,
                         int32_t n_cand, int32_t k, int32_t dev_mode, const cb_dims* dims, float* scores,
                         int32_t* sel, void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (n_cand < 0 || k < 0 || k > n_cand) return fail(CB_ERR_SHAPE, "need 0 <= k <= n_cand");
  if ((st = check_dev_rows(new_row, ref_row, n_cand, n_new_rows, n_ref_rows))) return st;
  if (dev_mode != CB_DEV_KV && dev_mode != CB_DEV_K) return fail(CB_ERR_INVALID_ARG, "dev_mode");
  if (n_cand == 0) return CB_OK;
  if (!k_new || !k_ref || (dev_mode == CB_DEV_KV && (!v_new || !v_ref)) || (k > 0 && !sel))
    return fail(CB_ERR_INVALID_ARG, "deviation pointer is NULL");
  if ((st = check_al16({k_new, v_new, k_ref, v_ref, ws}, "kv_deviation_topk"))) return st;
  const size_t need = 256 + (size_t)n_cand * 8 + 512;
  if (!ws || ws_bytes < need) return fail(CB_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  Carver c(ws);
  float* sc = scores ? scores : static_cast<float*>(c.take((size_t)n_cand * 4));
  int32_t* ord = static_cast<int32_t*>(c.take((size_t)n_cand * 4));
  const int W = dims->n_kv_heads * dims->head_dim;
  L_DEV(dims->dtype, k_new, v_new, k_ref, v_ref, new_row, ref_row, n_cand, n_new_rows, n_ref_rows, W,
        dev_mode == CB_DEV_KV, sc, S(stream));
  if (k > 0) {
    L_TOPK(sc, n_cand, k, ord, S(stream));
    L_MAP(ord, k, ref_row, sel, S(stream));
  }
  return CB_OK;
}

int cb_kv_deviation_topk_noalloc(const void* k_new, const void* v_new, int64_t n_new_rows, const void* k_ref,
                                 const void* v_ref, int64_t n_ref_rows, const int32_t* new_row,
                                 const int32_t* ref_row, int32_t n_cand, int32_t k, int32_t dev_mode,
                                 const cb_dims* dims, float* scores, int32_t* sel, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (n_cand < 0 || k < 0 || k > n_cand) return fail(CB_ERR_SHAPE, "need 0 <= k <= n_cand");
  if ((st = check_dev_rows(new_row, ref_row, n_cand, n_new_rows, n_ref_rows))) return st;
  if (n_cand > noalloc_max_candidates())
    return fail(CB_ERR_UNSUPPORTED, "n_cand %d exceeds the fixed scratch of %d candidates", n_cand,
                noalloc_max_candidates());
  if (dev_mode != CB_DEV_KV && dev_mode != CB_DEV_K) return fail(CB_ERR_INVALID_ARG, "dev_mode");
  if (n_cand == 0) return CB_OK;
  if (!k_new || !k_ref || (dev_mode == CB_DEV_KV && (!v_new || !v_ref)) || (k > 0 && !sel))
    return fail(CB_ERR_INVALID_ARG, "deviation pointer is NULL");
  if ((st = check_al16({k_new, v_new, k_ref, v_ref}, "kv_deviation_topk_noalloc"))) return st;
  const int W = dims->n_kv_heads * dims->head_dim;
  CB_CUDA(launch_deviation_topk_noalloc(dims->dtype, k_new, v_new, k_ref, v_ref, new_row, ref_row, n_cand,
                                        n_new_rows, n_ref_rows, k, W, dev_mode == CB_DEV_KV, scores, sel,
                                        S(stream)));
  g_launches.fetch_add(k > 0 ? 3 : 1, std::memory_order_relaxed);
  return CB_OK;
}

int cb_topk_from_scores(const float* scores, const int32_t* cand, int32_t n_cand, int32_t k, int32_t* sel,
                        void* ws, size_t ws_bytes, void* stream) {
  if (n_cand < 0 || k < 0 || k > n_cand) return fail(CB_ERR_SHAPE, "need 0 <= k <= n_cand");
  if (n_cand == 0) return CB_OK;
  if (!scores || (k > 0 && !sel)) return fail(CB_ERR_INVALID_ARG, "topk pointer is NULL");
  if (int st = check_al16({scores, ws}, "topk_from_scores")) return st;
  const size_t need = 256 + (size_t)n_cand * 4;
  if (!ws || ws_bytes < need) return fail(CB_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  Carver c(ws);
  int32_t* ord = static_cast<int32_t*>(c.take((size_t)n_cand * 4));
  L_TOPK(scores, n_cand, k, ord, S(stream));
  if (k > 0) L_MAP(ord, k, cand, sel, S(stream));
  return CB_OK;
}

int cb_rmsnorm(void* out, const void* x, int64_t n_x_rows, const int32_t* rows, int64_t n, int32_t d,
               const void* gain, float eps, int32_t dtype_in, int32_t dtype_out, void* stream) {
  if ((dtype_in != CB_F32 && dtype_in != CB_BF16) || (dtype_out != CB_F32 && dtype_out != CB_BF16) ||
      (dtype_in == CB_F32 && dtype_out == CB_BF16))
    return fail(CB_ERR_DTYPE, "rmsnorm dtypes %d -> %d", dtype_in, dtype_out);
  if (n < 0 || n_x_rows < 0 || d < 8 || d % 8 || !(eps >= 0.0f)) return fail(CB_ERR_SHAPE, "rmsnorm n/d/eps");
  if (n == 0) return CB_OK;
  if (!rows && n_x_rows < n) return fail(CB_ERR_SHAPE, "n_x_rows < n with rows NULL");
  if (!out || !x || !gain) return fail(CB_ERR_INVALID_ARG, "rmsnorm pointer is NULL");
  if (int st = check_al16({out, x, gain}, "rmsnorm")) return st;
  L_RMSNORM_B(dtype_in, dtype_out, out, x, rows, n_x_rows, gain, n, d, eps, S(stream));
  return CB_OK;
}

int cb_gather_rows(void* dst, const void* src, int64_t n_src_rows, const int32_t* idx, int64_t n, int64_t row_bytes,
                   void* stream) {
  if (n < 0 || n_src_rows < 0 || row_bytes < 0 || row_bytes % 4) return fail(CB_ERR_SHAPE, "n/n_src_rows/row_bytes");
  if (n == 0) return CB_OK;
  if (!idx && n_src_rows < n) return fail(CB_ERR_SHAPE, "n_src_rows < n with idx NULL");
  if (!dst || !src) return fail(CB_ERR_INVALID_ARG, "gather pointer is NULL");
  // rows are copied in 16-byte words where both bases allow it, else in 4-byte words
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 3)
    return fail(CB_ERR_INVALID_ARG, "gather: buffer not 4-byte aligned");
  L_COPY(dst, nullptr, src, idx, n, row_bytes, n, n_src_rows, S(stream));
  return CB_OK;
}

int cb_scatter_kv(void* k_cache, void* v_cache, int64_t n_cache_rows, const void* k_rows, const void* v_rows,
                  int64_t n_src_rows, const int32_t* dst_idx, const int32_t* src_idx, int64_t n,
                  const cb_dims* dims, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (n < 0 || n_cache_rows < 0 || n_src_rows < 0) return fail(CB_ERR_SHAPE, "negative size");
  if (n == 0) return CB_OK;
  if (!src_idx && n_src_rows < n) return fail(CB_ERR_SHAPE, "n_src_rows < n with src_idx NULL");
  if (!k_cache || !k_rows || !dst_idx || ((v_cache == nullptr) != (v_rows == nullptr)))
    return fail(CB_ERR_INVALID_ARG, "scatter pointer is NULL");
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_rows) | reinterpret_cast<uintptr_t>(v_rows)) & 3)
    return fail(CB_ERR_INVALID_ARG, "scatter_kv: buffer not 4-byte aligned");
  const int64_t rb = (int64_t)dims->n_kv_heads * dims->head_dim * esize(dims->dtype);
  L_COPY(k_cache, dst_idx, k_rows, src_idx, n, rb, n_cache_rows, n_src_rows, S(stream));
  if (v_cache) L_COPY(v_cache, dst_idx, v_rows, src_idx, n, rb, n_cache_rows, n_src_rows, S(stream));
  return CB_OK;
}

int cb_selective_qkv(const void* x, int64_t n_x_rows, const int32_t* rows, const int32_t* pos, int32_t M,
                     const cb_dims* dims, const cb_layer_w* w, const float* cos_sin, int32_t max_pos, void* q,
                     void* k, void* v, void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st || (st = check_w(w))) return st;
  if (M < 0 || n_x_rows < 0) return fail(CB_ERR_SHAPE, "M < 0 or n_x_rows < 0");
  if (M == 0) return CB_OK;
  if (!rows && n_x_rows < M) return fail(CB_ERR_SHAPE, "n_x_rows < M with rows NULL");
  if (!x || !pos || !cos_sin || (!q && !k) || ((k == nullptr) != (v == nullptr)))
    return fail(CB_ERR_INVALID_ARG, "selective_qkv pointer is NULL");
  if ((st = check_al16({x, q, k, v, cos_sin, ws}, "selective_qkv"))) return st;
  LayerWs L;
  if ((st = need_ws(dims, M, M, ws, ws_bytes, &L))) return st;
  const int qc = dims->n_heads * dims->head_dim, W = dims->n_kv_heads * dims->head_dim;
  L_RMSNORM_B(dims->dtype, dims->dtype, L.a, x, rows, n_x_rows, w->attn_norm, M, dims->d_model, dims->rms_eps,
              S(stream));
  const int col0 = q ? 0 : qc;
  const int ncols = (q ? qc : 0) + (k ? 2 * W : 0);
  L_GEMM(dims->dtype, qkv_desc(dims, w, L.a, M, col0, ncols, q, k, v, pos, nullptr, cos_sin, max_pos), S(stream));
  return CB_OK;
}

int cb_partial_attention(const void* q, const int32_t* q_pos, int32_t M, const void* k_cache, const void* v_cache,
                         int64_t n_kv, const cb_dims* dims, void* out, void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (M < 0 || n_kv < 1) return fail(CB_ERR_SHAPE, "M/n_kv");
  if (M == 0) return CB_OK;
  if (!q || !q_pos || !k_cache || !v_cache || !out) return fail(CB_ERR_INVALID_ARG, "attention pointer is NULL");
  if ((st = check_al16({q, k_cache, v_cache, out, ws}, "partial_attention"))) return st;
  const size_t need = attention_ws_bytes(dims->dtype, M, dims->n_heads, dims->head_dim);
  if (need && (!ws || ws_bytes < need)) return fail(CB_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  L_ATTN(dims->dtype, q, q_pos, M, k_cache, v_cache, n_kv, dims->n_heads, dims->n_kv_heads, dims->head_dim, out, ws, ws_bytes, S(stream));
  return CB_OK;
}

int cb_o_proj_ffn(const void* attn, const void* x_res, int32_t M, const cb_dims* dims, const cb_layer_w* w,
                  void* x_out, void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st || (st = check_w(w))) return st;
  if (M < 0) return fail(CB_ERR_SHAPE, "M < 0");
  if (M == 0) return CB_OK;
  if (!attn || !x_res || !x_out) return fail(CB_ERR_INVALID_ARG, "o_proj_ffn pointer is NULL");
  if ((st = check_al16({attn, x_res, x_out, ws}, "o_proj_ffn"))) return st;
  LayerWs L;
  if ((st = need_ws(dims, M, M, ws, ws_bytes, &L))) return st;
  return o_ffn(dims, w, attn, x_res, M, x_out, L, S(stream));
}

int cb_blend_layer(const cb_dims* dims, const cb_layer_w* w, int32_t mode, const void* x_in, const int32_t* s_in,
                   int32_t m_in, int64_t n_tok, int64_t n_cached, void* k_cache, void* v_cache,
                   const float* cos_sin, int32_t max_pos, int32_t k_budget, int32_t dev_mode,
                   const int32_t* sel_override, void* x_out, int32_t* s_out, int32_t* m_out_host,
                   float* scores_out, const cb_layer_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st || (st = check_w(w))) return st;
  if (!x_in || !k_cache || !v_cache || !cos_sin || !x_out || !s_out || !m_out_host)
    return fail(CB_ERR_INVALID_ARG, "blend_layer pointer is NULL");
  if (x_out == x_in) return fail(CB_ERR_INVALID_ARG, "x_out must not alias x_in");
  if ((st = check_al16({x_in, k_cache, v_cache, cos_sin, x_out, ws}, "blend_layer"))) return st;
  if (n_tok < 1 || n_tok > INT32_MAX || n_cached < 0 || n_cached > n_tok)
    return fail(CB_ERR_SHAPE, "need 0 <= n_cached <= n_tok, n_tok >= 1");
  if (n_tok > max_pos) return fail(CB_ERR_SHAPE, "rope table (%d) shorter than n_tok (%lld)", max_pos, (long long)n_tok);
  if (dev_mode != CB_DEV_KV && dev_mode != CB_DEV_K) return fail(CB_ERR_INVALID_ARG, "dev_mode");
  const int N = (int)n_tok;
  const uint8_t* fmask = opts ? opts->forced_mask : nullptr;
  void* kv_ready = opts ? opts->kv_ready : nullptr;
  const int32_t* x_rows = opts ? opts->x_rows : nullptr;
  const int64_t n_x_rows = opts ? opts->n_x_rows : 0;
  if (x_rows && (mode != CB_LAYER_PRECHECK || n_x_rows < 1))
    return fail(CB_ERR_INVALID_ARG, "x_rows applies to PRECHECK, with n_x_rows >= 1");
  const bool fork = opts && opts->aux_stream;
  float* ssq_out = opts ? opts->x_out_ssq : nullptr;
  int32_t* ssq_out_parts = opts ? opts->x_out_ssq_parts_host : nullptr;
  if (ssq_out && !ssq_out_parts) return fail(CB_ERR_INVALID_ARG, "x_out_ssq needs x_out_ssq_parts_host");
  const float* ssq_in = opts ? opts->x_in_ssq : nullptr;
  const int ssq_in_parts = opts ? opts->x_in_ssq_parts : 0;
  if (ssq_in && (ssq_in_parts < 0 || ssq_in_parts > dev_parts(dims->d_model)))
    return fail(CB_ERR_SHAPE, "x_in_ssq_parts %d outside [0, %d]", ssq_in_parts, dev_parts(dims->d_model));
  // the attention norm folded into the Q/K/V GEMMs: bf16, unit gains, the input's statistics
  const bool fuse_in = ssq_in && ssq_in_parts > 0 && dims->dtype == CB_BF16 && w->attn_norm == nullptr &&
                       mode != CB_LAYER_PRECHECK;
  if (opts && ((opts->aux_stream == nullptr) != (opts->aux_fork == nullptr) ||
               (opts->aux_stream == nullptr) != (opts->aux_join == nullptr)))
    return fail(CB_ERR_INVALID_ARG, "aux_stream, aux_fork and aux_join must all be set or all NULL");
  if (fmask && (opts->n_forced < 1 || opts->n_forced > N))
    return fail(CB_ERR_SHAPE, "n_forced %d outside [1, n_tok]", opts ? opts->n_forced : 0);
  if (opts && opts->recompute_from != 0) {
    if (mode != CB_LAYER_PRECHECK || fmask || opts->recompute_kv)
      return fail(CB_ERR_INVALID_ARG, "recompute_from applies to PRECHECK without forced_mask or recompute_kv");
    if (opts->recompute_from < 0 || opts->recompute_from > n_cached)
      return fail(CB_ERR_SHAPE, "recompute_from %d outside [0, n_cached]", opts->recompute_from);
  }
  // default layout: forced rows [f0, N) (the uncached suffix and the last row)
  const int f0 = (int)std::min<int64_t>(n_cached, n_tok - 1);
  const int n_forced = fmask ? opts->n_forced : N - f0;
  const int qc = dims->n_heads * dims->head_dim, W = dims->n_kv_heads * dims->head_dim;
  const size_t B = esize(dims->dtype);
  const bool use_v = dev_mode == CB_DEV_KV;
  cudaStream_t s = S(stream);
  LayerWs L;
  // the stream waits for the cached rows right before its first access to them
#define WAIT_CACHED_ROWS() \
  do { if (kv_ready) CB_CUDA(cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(kv_ready), 0)); } while (0)

  switch (mode) {
    case CB_LAYER_PRECHECK: {
      if (m_in != N) return fail(CB_ERR_SHAPE, "PRECHECK needs m_in == n_tok");
      if ((st = need_ws(dims, N, N, ws, ws_bytes, &L))) return st;
      *m_out_host = N;
      L_IOTA(s_out, N, 0, s);
      // input row i is x_in[x_rows[i]] when a row map is given (e.g. the embedding table and the
      // token ids): the norm and the residual read the table rows in place
      L_RMSNORM_B(dims->dtype, dims->dtype, L.a, x_in, x_rows, x_rows ? n_x_rows : -1, w->attn_norm, N, dims->d_model,
                  dims->rms_eps, s);
      if (opts && opts->recompute_kv) {
        // every row's Q, K and V in one GEMM; the cached rows are overwritten, not read
        WAIT_CACHED_ROWS();
        GemmDesc g = qkv_desc(dims, w, L.a, N, 0, qc + 2 * W, L.q, k_cache, v_cache, s_out, s_out, cos_sin, max_pos);
        g.epi.kv_bound = N;
        L_GEMM(dims->dtype, g, s);
        L_ATTN(dims->dtype, L.q, s_out, N, k_cache, v_cache, N, dims->n_heads, dims->n_kv_heads, dims->head_dim, L.attn, L.attn_ws, 0, s);
        return o_ffn(dims, w, L.attn, x_in, N, x_out, L, s, x_rows, x_rows ? n_x_rows : -1, ssq_out, ssq_out_parts);
      }
      // Q of every row and K/V of the uncached rows (and of the cached rows from
      // recompute_from on): independent, so one shared launch
      const GemmDesc gq = qkv_desc(dims, w, L.a, N, 0, qc, L.q, nullptr, nullptr, s_out, nullptr, cos_sin, max_pos);
      const int kv0 = (opts && opts->recompute_from > 0) ? opts->recompute_from : (int)n_cached;
      if (fmask) {
        // K/V of the forced rows, wherever they are: gather their normalised rows first
        L_SPLIT(nullptr, N, fmask, N, n_forced, L.cpos, L.crows, L.fpos, L.frows, s);
        L_COPY(L.ag, nullptr, L.a, L.frows, n_forced, (int64_t)dims->d_model * B, n_forced, N, s);
        GemmDesc gkv = qkv_desc(dims, w, L.ag, n_forced, qc, 2 * W, nullptr, k_cache, v_cache, L.frows, L.frows, cos_sin, max_pos);
        gkv.epi.kv_bound = N;
        L_GEMM2(dims->dtype, gq, gkv, s);
      } else if (N > kv0) {
        const int nu = N - kv0;
        const void* a_u = static_cast<const char*>(L.a) + (size_t)kv0 * dims->d_model * B;
        GemmDesc gkv = qkv_desc(dims, w, a_u, nu, qc, 2 * W, nullptr, k_cache, v_cache, s_out + kv0, s_out + kv0, cos_sin, max_pos);
        gkv.epi.kv_bound = N;
        L_GEMM2(dims->dtype, gq, gkv, s);
      } else {
        L_GEMM(dims->dtype, gq, s);
      }
      WAIT_CACHED_ROWS();
      L_ATTN(dims->dtype, L.q, s_out, N, k_cache, v_cache, N, dims->n_heads, dims->n_kv_heads, dims->head_dim, L.attn, L.attn_ws, 0, s);
      return o_ffn(dims, w, L.attn, x_in, N, x_out, L, s, x_rows, x_rows ? n_x_rows : -1, ssq_out, ssq_out_parts);
    }
    case CB_LAYER_CHECK:
    case CB_LAYER_GRADUAL: {
      const bool check = mode == CB_LAYER_CHECK;
      if (check && m_in != N) return fail(CB_ERR_SHAPE, "CHECK needs m_in == n_tok");
      if (!check && (m_in < n_forced || m_in > N)) return fail(CB_ERR_SHAPE, "GRADUAL needs n_forced <= m_in <= n_tok");
      if (!check && !s_in && m_in != N) return fail(CB_ERR_INVALID_ARG, "GRADUAL needs s_in");
      const int n_cand = (check && !fmask) ? f0 : m_in - n_forced;
      if (k_budget < 0 || k_budget > n_cand)
        return fail(CB_ERR_SHAPE, "k_budget %d outside [0, %d]", k_budget, n_cand);
      const int M = k_budget + n_forced;
      if ((st = need_ws(dims, m_in, M, ws, ws_bytes, &L))) return st;
      *m_out_host = M;
      const int32_t* rows_in = s_in;
      if (check || !s_in) {
        L_IOTA(L.rows, m_in, 0, s);
        rows_in = L.rows;
      }
      float* sc = scores_out ? scores_out : L.scores;
      // candidates: positions (GEMM rows) and rows of the cached, unforced incoming rows;
      // without a mask they are the leading n_cand rows of the incoming set
      const int32_t* cpos = nullptr;
      const int32_t* crows = rows_in;
      if (fmask) {
        L_SPLIT(rows_in, m_in, fmask, N, n_forced, L.cpos, L.crows, L.fpos, L.frows, s);
        cpos = L.cpos;
        crows = L.crows;
      }
      if (!fuse_in)
        L_RMSNORM(dims->dtype, dims->dtype, L.a, x_in, nullptr, w->attn_norm, m_in, dims->d_model, dims->rms_eps, s);
      const void* a_in = fuse_in ? x_in : L.a;   // the GEMMs' rows: normalised, or scaled in the epilogue
      auto fold_norm = [&](GemmDesc& g, const int32_t* row_map) {
        if (!fuse_in) return;
        g.epi.rs_in = ssq_in;
        g.epi.rs_row = row_map;
        g.epi.rs_parts = ssq_in_parts;
        g.epi.rs_ld = m_in;
        g.epi.rs_inv_d = 1.0f / (float)dims->d_model;
        g.epi.rs_eps = dims->rms_eps;
      };
      WAIT_CACHED_ROWS();
      // A gradual layer whose incoming set is at most 25% larger than its selection computes
      // Q for every incoming row in the same GEMM (one wider launch) and gathers the
      // selected queries afterwards; otherwise Q is computed for the selected rows only.
      const bool q_all = !check && (int64_t)m_in * 4 <= (int64_t)M * 5;
      const int col0 = q_all ? 0 : qc, ncols = q_all ? qc + 2 * W : 2 * W;
      GemmDesc gkv = qkv_desc(dims, w, a_in, m_in, col0, ncols, q_all ? L.q : nullptr, L.knew, L.vnew, rows_in, nullptr,
                              cos_sin, max_pos);
      fold_norm(gkv, nullptr);
      if (dims->dtype == CB_BF16) {
        // the deviation is taken in the K/V GEMM's epilogue; a small pass sums the tiles
        gkv.epi.dev_part = L.dev_part;
        gkv.epi.dev_ld = m_in;
        gkv.epi.k_ref = k_cache;
        gkv.epi.v_ref = v_cache;
        gkv.epi.ref_row = rows_in;
        gkv.epi.ref_rows = N;
        gkv.epi.dev_use_v = use_v ? 1 : 0;
        const int bn = gemm_tc_tile_n(&gkv, 1);
        L_GEMM(dims->dtype, gkv, s);
        // partials of tiles that hold only Q columns are zero: start at the first tile that
        // holds K columns
        L_DEVRED(L.dev_part, q_all ? 2 * (qc / bn) : 0, dev_parts(ncols, bn), m_in, n_cand, cpos, W, use_v, sc, s);
      } else {
        L_GEMM(dims->dtype, gkv, s);
        L_DEV(dims->dtype, L.knew, L.vnew, k_cache, v_cache, cpos, crows, n_cand, m_in, N, W, use_v, sc, s);
      }
      if (k_budget > 0 && !sel_override && !fmask) {
        // top-k and the selection build (S = candidate rows of the top k ++ forced rows) in
        // one launch
        L_TOPK_SEL(sc, n_cand, k_budget, rows_in, f0, m_in - n_forced, n_forced, s_out, L.keep, s);
      } else {
        if (k_budget > 0) {
          if (sel_override)
            L_R2P(sel_override, k_budget, (check && !fmask) ? nullptr : crows, n_cand, L.ord, s);
          else
            L_TOPK(sc, n_cand, k_budget, L.ord, s);
        }
        if (fmask)
          L_MERGE(L.ord, k_budget, L.crows, L.cpos, L.frows, L.fpos, n_forced, s_out, L.keep, s);
        else
          L_BUILD_SEL(L.ord, k_budget, rows_in, f0, m_in - n_forced, n_forced, s_out, L.keep, s);
      }
      // Step 3, KV expansion (the recomputed K/V of S replace the cached rows), and the
      // gather of S's queries (or normalised rows): one launch, or with an aux stream the
      // expansion there, beside the Q GEMM.  S's residual rows are read in place by the
      // O-projection's epilogue (row map keep).
      {
        // the expansion overlaps only a Q GEMM; with Q already computed, attention waits for it
        const bool fork_kv = fork && !q_all;
        RowCopies rc, kv;
        RowCopies& kvc = fork_kv ? kv : rc;
        kvc.add(k_cache, s_out, L.knew, L.keep, M, (int64_t)W * B, N, m_in);
        kvc.add(v_cache, s_out, L.vnew, L.keep, M, (int64_t)W * B, N, m_in);
        if (q_all)
          rc.add(L.qg, nullptr, L.q, L.keep, M, (int64_t)qc * B, M, m_in);
        else
          rc.add(L.ag, nullptr, a_in, L.keep, M, (int64_t)dims->d_model * B, M, m_in);
        if (fork_kv) {
          cudaStream_t aux = S(opts->aux_stream);
          CB_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(opts->aux_fork), s));
          CB_CUDA(cudaStreamWaitEvent(aux, static_cast<cudaEvent_t>(opts->aux_fork), 0));
          if ((st = kv.launch(aux, /*beside=*/true))) return st;   // runs beside the Q GEMM
          CB_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(opts->aux_join), aux));
        }
        if ((st = rc.launch(s))) return st;
      }
      const void* qsel = q_all ? L.qg : L.q;
      if (!q_all) {
        GemmDesc gq = qkv_desc(dims, w, L.ag, M, 0, qc, L.q, nullptr, nullptr, s_out, nullptr, cos_sin, max_pos);
        fold_norm(gq, L.keep);   // row m of the selection is row keep[m] of the input
        L_GEMM(dims->dtype, gq, s);
      }
      if (fork && !q_all) CB_CUDA(cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(opts->aux_join), 0));
      L_ATTN(dims->dtype, qsel, s_out, M, k_cache, v_cache, N, dims->n_heads, dims->n_kv_heads, dims->head_dim, L.attn, L.attn_ws, 0, s);
      return o_ffn(dims, w, L.attn, x_in, M, x_out, L, s, L.keep, m_in, ssq_out, ssq_out_parts);
    }
    case CB_LAYER_STEADY: {
      if (m_in < 1 || m_in > N) return fail(CB_ERR_SHAPE, "STEADY needs 1 <= m_in <= n_tok");
      if (!s_in && m_in != N) return fail(CB_ERR_INVALID_ARG, "STEADY needs s_in");
      if ((st = need_ws(dims, m_in, m_in, ws, ws_bytes, &L))) return st;
      *m_out_host = m_in;
      if (s_in)
        CB_CUDA(cudaMemcpyAsync(s_out, s_in, (size_t)m_in * 4, cudaMemcpyDeviceToDevice, s));
      else
        L_IOTA(s_out, m_in, 0, s);
      if (!fuse_in)
        L_RMSNORM(dims->dtype, dims->dtype, L.a, x_in, nullptr, w->attn_norm, m_in, dims->d_model, dims->rms_eps, s);
      WAIT_CACHED_ROWS();
      // s_out is the caller's row set: its rows are checked against the cache height
      GemmDesc g = qkv_desc(dims, w, fuse_in ? x_in : L.a, m_in, 0, qc + 2 * W, L.q, k_cache, v_cache, s_out, s_out,
                            cos_sin, max_pos);
      g.epi.kv_bound = N;
      if (fuse_in) {
        g.epi.rs_in = ssq_in;
        g.epi.rs_parts = ssq_in_parts;
        g.epi.rs_ld = m_in;
        g.epi.rs_inv_d = 1.0f / (float)dims->d_model;
        g.epi.rs_eps = dims->rms_eps;
      }
      L_GEMM(dims->dtype, g, s);
      L_ATTN(dims->dtype, L.q, s_out, m_in, k_cache, v_cache, N, dims->n_heads, dims->n_kv_heads, dims->head_dim, L.attn, L.attn_ws, 0, s);
      return o_ffn(dims, w, L.attn, x_in, m_in, x_out, L, s, nullptr, -1, ssq_out, ssq_out_parts);
    }
    default:
      return fail(CB_ERR_INVALID_ARG, "mode %d", mode);
  }
#undef WAIT_CACHED_ROWS
}

int cb_blend_steady_batch(const cb_dims* dims, const cb_layer_w* w, int32_t n_req, const int32_t* row0_host,
                          const void* x_in, const int32_t* s_in, int64_t n_tok, void* k_cache, void* v_cache,
                          const float* cos_sin, int32_t max_pos, void* x_out, void* ws, size_t ws_bytes,
                          void* stream) {
  int st = check_dims(dims);
  if (st || (st = check_w(w))) return st;
  if (!row0_host || !x_in || !s_in || !k_cache || !v_cache || !cos_sin || !x_out)
    return fail(CB_ERR_INVALID_ARG, "blend_steady_batch pointer is NULL");
  if (x_out == x_in) return fail(CB_ERR_INVALID_ARG, "x_out must not alias x_in");
  if ((st = check_al16({x_in, k_cache, v_cache, cos_sin, x_out, ws}, "blend_steady_batch"))) return st;
  if (n_req < 1 || n_req > kMaxBatch) return fail(CB_ERR_SHAPE, "n_req %d outside [1, %d]", n_req, kMaxBatch);
  if (n_tok < 1 || n_tok > max_pos) return fail(CB_ERR_SHAPE, "need 1 <= n_tok <= max_pos");
  if ((int64_t)n_req * n_tok > INT32_MAX) return fail(CB_ERR_SHAPE, "n_req * n_tok exceeds the int32 row range");
  BatchRows br{};
  br.n_req = n_req;
  if (row0_host[0] != 0) return fail(CB_ERR_SHAPE, "row0[0] must be 0");
  for (int r = 0; r <= n_req; ++r) {
    if (r > 0 && (row0_host[r] < row0_host[r - 1] || row0_host[r] - row0_host[r - 1] > n_tok))
      return fail(CB_ERR_SHAPE, "request %d: rows must be non-decreasing, at most n_tok per request", r - 1);
    br.row0[r] = row0_host[r];
  }
  const int M = row0_host[n_req];
  if (M == 0) return CB_OK;
  LayerWs L;
  if ((st = need_ws(dims, M, M, ws, ws_bytes, &L))) return st;
  cudaStream_t s = S(stream);
  const int qc = dims->n_heads * dims->head_dim, W = dims->n_kv_heads * dims->head_dim;
  const size_t B = esize(dims->dtype);
  L_RMSNORM(dims->dtype, dims->dtype, L.a, x_in, nullptr, w->attn_norm, M, dims->d_model, dims->rms_eps, s);
  CB_LAUNCH(CB_PROF_INDEX, 3, M, 0, 0, 0.0, 8.0 * M, s, launch_batch_kv_rows(s_in, M, n_tok, br, L.rows, s));
  // one Q/K/V GEMM over every request's rows: RoPE at each row's position in its request,
  // K/V written straight into its request's cache rows
  GemmDesc g = qkv_desc(dims, w, L.a, M, 0, qc + 2 * W, L.q, k_cache, v_cache, s_in, L.rows, cos_sin, max_pos);
  g.epi.kv_bound = (int64_t)n_req * n_tok;
  L_GEMM(dims->dtype, g, s);
  for (int r = 0; r < n_req; ++r) {
    const int m0 = row0_host[r], mr = row0_host[r + 1] - m0;
    if (mr == 0) continue;
    const size_t off = (size_t)r * n_tok * W * B;
    L_ATTN(dims->dtype, static_cast<const char*>(L.q) + (size_t)m0 * qc * B, s_in + m0, mr,
           static_cast<const char*>(k_cache) + off, static_cast<const char*>(v_cache) + off, n_tok, dims->n_heads,
           dims->n_kv_heads, dims->head_dim, static_cast<char*>(L.attn) + (size_t)m0 * qc * B, L.attn_ws, 0, s);
  }
  return o_ffn(dims, w, L.attn, x_in, M, x_out, L, s);
}

int cb_full_prefill(const cb_dims* dims, int32_t n_layers, const cb_layer_w* layers_host, const void* embed,
                    const int32_t* tokens, int32_t n, int32_t pos0, void* const* k_out_host,
                    void* const* v_out_host, void* h_last, void* x_all, const float* cos_sin, int32_t max_pos,
                    void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (n_layers < 1 || !layers_host || !embed || !tokens || !k_out_host || !v_out_host || !cos_sin)
    return fail(CB_ERR_INVALID_ARG, "full_prefill argument is NULL");
  for (int l = 0; l < n_layers; ++l) {
    if ((st = check_w(&layers_host[l]))) return st;
    if (!k_out_host[l] || !v_out_host[l]) return fail(CB_ERR_INVALID_ARG, "k_out/v_out[%d] is NULL", l);
    if ((st = check_al16({k_out_host[l], v_out_host[l]}, "full_prefill k_out/v_out"))) return st;
  }
  if ((st = check_al16({embed, h_last, x_all, cos_sin, ws}, "full_prefill"))) return st;
  if (n < 1 || pos0 < 0) return fail(CB_ERR_SHAPE, "n >= 1, pos0 >= 0");
  if ((int64_t)pos0 + n > max_pos) return fail(CB_ERR_SHAPE, "rope table shorter than pos0 + n");
  LayerWs L;
  if ((st = need_ws(dims, n, n, ws, ws_bytes, &L))) return st;
  cudaStream_t s = S(stream);
  const size_t B = esize(dims->dtype);
  const int qc = dims->n_heads * dims->head_dim, W = dims->n_kv_heads * dims->head_dim;
  const int64_t row_b = (int64_t)dims->d_model * B;
  L_COPY(L.xa, nullptr, embed, tokens, n, row_b, n, dims->vocab, s);
  L_IOTA(L.pos, n, pos0, s);
  L_IOTA(L.rows, n, 0, s);
  void* x = L.xa;
  void* y = L.xb;
  for (int l = 0; l < n_layers; ++l) {
    const cb_layer_w* w = &layers_host[l];
    L_RMSNORM(dims->dtype, dims->dtype, L.a, x, nullptr, w->attn_norm, n, dims->d_model, dims->rms_eps, s);
    L_GEMM(dims->dtype, qkv_desc(dims, w, L.a, n, 0, qc + 2 * W, L.q, k_out_host[l], v_out_host[l], L.pos, nullptr, cos_sin, max_pos), s);
    L_ATTN(dims->dtype, L.q, L.rows, n, k_out_host[l], v_out_host[l], n, dims->n_heads, dims->n_kv_heads, dims->head_dim, L.attn, L.attn_ws, 0, s);
    if ((st = o_ffn(dims, w, L.attn, x, n, y, L, s))) return st;
    std::swap(x, y);
  }
  if (h_last)
    CB_CUDA(cudaMemcpyAsync(h_last, static_cast<char*>(x) + (size_t)(n - 1) * row_b, row_b, cudaMemcpyDeviceToDevice, s));
  if (x_all) CB_CUDA(cudaMemcpyAsync(x_all, x, (size_t)n * row_b, cudaMemcpyDeviceToDevice, s));
  return CB_OK;
}

int cb_lmhead_argmax(const void* h, const void* final_norm, const void* w_lm, const cb_dims* dims, float* logits,
                     int32_t* token, void* ws, size_t ws_bytes, void* stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!h || !final_norm || !w_lm || !token) return fail(CB_ERR_INVALID_ARG, "lmhead pointer is NULL");
  if ((st = check_al16({h, final_norm, w_lm, logits, ws}, "lmhead_argmax"))) return st;
  const int nb = (int)lm_block_best_count(dims->vocab);
  const size_t need = 256 + (size_t)dims->d_model * 4 + 256 + (size_t)dims->vocab * 4 + 256 + (size_t)nb * 8 + 256;
  if (!ws || ws_bytes < need) return fail(CB_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  Carver c(ws);
  float* hn = static_cast<float*>(c.take((size_t)dims->d_model * 4));
  float* lg = logits ? logits : static_cast<float*>(c.take((size_t)dims->vocab * 4));
  unsigned long long* bb = static_cast<unsigned long long*>(c.take((size_t)nb * 8));
  cudaStream_t s = S(stream);
  L_RMSNORM(dims->dtype, CB_F32, hn, h, nullptr, final_norm, 1, dims->d_model, dims->rms_eps, s);
  L_LMGEMV(dims->dtype, lg, hn, w_lm, dims->vocab, dims->d_model, bb, s);
  L_ARGMAX(bb, (int)lm_block_count(dims->vocab, dims->dtype), token, s);
  return CB_OK;
}

// y = x W^T (plain linear layer) on the same GEMM kernels as the layer path.
int cb_linear(const void* x, const void* w, void* y, int32_t M, int32_t N, int32_t K, int32_t dtype, void* stream) {
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_DTYPE, "dtype %d", dtype);
  if (M < 0 || N < 1 || K < 1) return fail(CB_ERR_SHAPE, "M/N/K");
  if (M == 0) return CB_OK;
  if (!x || !w || !y) return fail(CB_ERR_INVALID_ARG, "linear pointer is NULL");
  if (int st = check_al16({x, w, y}, "linear")) return st;
  if (dtype == CB_BF16 && (N % 16 || K % 8)) return fail(CB_ERR_UNSUPPORTED, "bf16 needs N %% 16 == 0, K %% 8 == 0");
  if (dtype == CB_F32 && N % 4) return fail(CB_ERR_UNSUPPORTED, "fp32 needs N %% 4 == 0");
  GemmDesc g = make_gemm(M, N, K, x, K, w, K);
  g.epi.kind = EPI_STORE;
  g.epi.out = y;
  g.epi.ldo = N;
  L_GEMM(dtype, g, S(stream));
  return CB_OK;
}

int cb_prefetch_layer(void* dev_dst, const void* pinned_src, size_t bytes, void* side_stream, void* done_event) {
  if (bytes > 0 && (!dev_dst || !pinned_src)) return fail(CB_ERR_INVALID_ARG, "prefetch pointer is NULL");
  if (!done_event) return fail(CB_ERR_INVALID_ARG, "done_event is NULL");
  const char* d = static_cast<const char*>(dev_dst);
  const char* h = static_cast<const char*>(pinned_src);
  if (bytes > 0 && d < h + bytes && h < d + bytes) return fail(CB_ERR_INVALID_ARG, "source and destination overlap");
  if (bytes > 0) CB_CUDA(cudaMemcpyAsync(dev_dst, pinned_src, bytes, cudaMemcpyHostToDevice, S(side_stream)));
  CB_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(done_event), S(side_stream)));
  return CB_OK;
}

int cb_copy_async(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return CB_OK;
  if (!dst || !src) return fail(CB_ERR_INVALID_ARG, "copy pointer is NULL");
  CB_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, S(stream)));
  return CB_OK;
}

int cb_stream_wait(void* stream, void* event) {
  if (!event) return fail(CB_ERR_INVALID_ARG, "event is NULL");
  CB_CUDA(cudaStreamWaitEvent(S(stream), static_cast<cudaEvent_t>(event), 0));
  return CB_OK;
}

int64_t cb_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void cb_shutdown(void) {
  reset_mem_caches();
  reset_gemm_tc_caches();
  reset_attn_tc_caches();
  ProfState& P = g_prof;
  bool failed = false;
  for (cudaEvent_t e : P.ev) failed = cudaEventDestroy(e) != cudaSuccess || failed;
  if (failed) cudaGetLastError();   // clears the errors of the destroys just made
  P.ev.clear();
  P.rec.clear();
  P.on = false;
  if (P.spans) g_span_taken.store(false);
  P.spans = false;
  P.cap = 0;
  g_cur_span = nullptr;
}

int cb_profile_begin(int32_t max_records) {
  if (max_records < 1) return fail(CB_ERR_INVALID_ARG, "max_records < 1");
  ProfState& P = g_prof;
  if (P.spans) {   // leaving span mode: the slot buffer is free for other threads
    P.spans = false;
    g_cur_span = nullptr;
    g_span_taken.store(false);
  }
  while ((int)P.ev.size() < 2 * max_records) {
    cudaEvent_t e;
    CB_CUDA(cudaEventCreate(&e));
    P.ev.push_back(e);
  }
  P.rec.clear();
  P.rec.reserve(max_records);
  P.cap = max_records;
  P.on = true;
  return CB_OK;
}

int cb_profile_begin_spans(int32_t max_records) {
  if (max_records < 1 || max_records > kSpanMax) return fail(CB_ERR_INVALID_ARG, "max_records outside 1..%d", kSpanMax);
  ProfState& P = g_prof;
  if (!P.spans) {
    bool expected = false;
    if (!g_span_taken.compare_exchange_strong(expected, true))
      return fail(CB_ERR_INVALID_ARG, "span profiling is active on another thread");
  }
  P.spans = false;   // re-armed below once the buffer is reset
  void* addr = nullptr;
  const cudaError_t ea = cudaGetSymbolAddress(&addr, g_span_buf);
  if (ea != cudaSuccess) g_span_taken.store(false);
  CB_CUDA(ea);
  std::vector<unsigned long long> init(2 * (size_t)max_records, 0ull);
  for (int i = 0; i < max_records; ++i) init[2 * i] = ~0ull;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(addr, init.data(), init.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) g_span_taken.store(false);
  CB_CUDA(e);
  P.span_base = static_cast<unsigned long long*>(addr);
  P.rec.clear();
  P.rec.reserve(max_records);
  P.cap = max_records;
  P.spans = true;
  P.on = true;
  return CB_OK;
}

int cb_profile_end(cb_prof_record* out_host, int32_t max_records, int32_t* n_out_host) {
  ProfState& P = g_prof;
  P.on = false;
  const bool spans = P.spans;
  P.spans = false;
  g_cur_span = nullptr;
  if (spans) g_span_taken.store(false);
  if (!n_out_host) return fail(CB_ERR_INVALID_ARG, "n_out_host is NULL");
  const int n = std::min<int>((int)P.rec.size(), std::max(0, max_records));
  if (spans) {
    std::vector<unsigned long long> t(2 * P.rec.size() + 2, 0ull);
    CB_CUDA(cudaDeviceSynchronize());
    if (!P.rec.empty())
      CB_CUDA(cudaMemcpy(t.data(), P.span_base, 2 * P.rec.size() * sizeof(unsigned long long),
                         cudaMemcpyDeviceToHost));
    for (int i = 0; i < (int)P.rec.size(); ++i) {
      const unsigned long long a = t[2 * i], b = t[2 * i + 1];
      P.rec[i].ms = -1.f;
      P.rec[i].span_ms = (a != ~0ull && b >= a) ? (float)((double)(b - a) * 1e-6) : -1.f;
    }
  } else {
    for (int i = 0; i < (int)P.rec.size(); ++i) {
      CB_CUDA(cudaEventSynchronize(P.ev[2 * i + 1]));
      float ms = 0.f;
      CB_CUDA(cudaEventElapsedTime(&ms, P.ev[2 * i], P.ev[2 * i + 1]));
      P.rec[i].ms = ms;
      P.rec[i].span_ms = -1.f;
    }
  }
  if (out_host && n > 0) memcpy(out_host, P.rec.data(), sizeof(cb_prof_record) * n);
  *n_out_host = n;
  P.rec.clear();
  return CB_OK;
}

}  // extern "C"
