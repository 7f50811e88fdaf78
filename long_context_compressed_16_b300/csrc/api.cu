// Host side of the C ABI declared in include/csa.h: argument validation, workspace layout,
// RoPE tables and kernel orchestration.  Nothing here allocates device memory.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>

#include "common.cuh"

namespace {

std::atomic<uint64_t> g_launches{0};

#ifndef CSA_INDEX_FUSED_SELECT
#define CSA_INDEX_FUSED_SELECT 1   // 0: csa_index_topk always stores score rows and runs the selector kernels
#endif
#ifndef CSA_SCORE_CHUNK_MIB
#define CSA_SCORE_CHUNK_MIB 256
#endif
constexpr size_t kScoreChunkCap = size_t(CSA_SCORE_CHUNK_MIB) << 20;   // bytes of fp32 scores per top-k pass
#ifndef CSA_ATT_DECODE_SPLIT
#define CSA_ATT_DECODE_SPLIT 192                        // decode attention slots per split, bf16 rows
#endif
#ifndef CSA_ATT_DECODE_SPLIT_FP8
#define CSA_ATT_DECODE_SPLIT_FP8 128                    // the same for mixed FP8 rows
#endif
#ifndef CSA_ATT_DECODE_SPLIT_HCA
#define CSA_ATT_DECODE_SPLIT_HCA 512                    // dense HCA decode (every closed entry), bf16 rows
#endif

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline csa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

bool make_rope(int r, float theta, const float* inv_freq, csa::RopeParams* rp) {
  if (r < 0 || (r & 1) || r / 2 > csa::kMaxRopePairs) return false;
  std::memset(rp, 0, sizeof(*rp));
  rp->r = r;
  const long double two_pi = 2.0L * std::acos(-1.0L);
  const long double two64 = std::ldexp(1.0L, 64);
  for (int j = 0; j < r / 2; ++j) {
    const double f = inv_freq ? static_cast<double>(inv_freq[j])
                              : std::pow(static_cast<double>(theta), -2.0 * j / static_cast<double>(r));
    if (!std::isfinite(f)) return false;
    // the turn per position as a fraction of a revolution, mod 1, in 64-bit fixed point
    long double x = static_cast<long double>(f) / two_pi;
    x -= std::floor(x);
    x = std::floor(x * two64 + 0.5L);
    rp->phase[j] = x >= two64 ? 0ull : static_cast<unsigned long long>(x);
  }
  return true;
}

void count(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

// Compressor row widths: a power of two in [64, 1024], so an entry's d/8 threads form a
// power-of-two group for the RMSNorm reduction.
inline bool compress_width_ok(int w) { return w >= 64 && w <= 1024 && (w & (w - 1)) == 0; }

csa_status cache_desc_check(const csa_cache_desc* d) {
  if (!d) return CSA_ERR_INVALID_ARG;
  if (d->B < 0 || d->m < 1 || d->m > 256 || d->Wcap < 1 || d->N_cap < 0 || !(d->eps >= 0.f))
    return CSA_ERR_INVALID_ARG;
  if (!compress_width_ok(d->d)) return CSA_ERR_UNSUPPORTED;
  if (d->dI < 0) return CSA_ERR_INVALID_ARG;
  if (d->dI != 0 && (!compress_width_ok(d->dI) || !d->overlap)) return CSA_ERR_UNSUPPORTED;
  if (d->rope_dims < 0 || d->rope_dims > d->d || (d->rope_dims % 8) != 0 || d->rope_dims > 2 * csa::kMaxRopePairs)
    return CSA_ERR_UNSUPPORTED;
  if (d->index_flags & CSA_COMPRESS_ROPE) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

csa_status out_proj_check(const csa_out_proj_desc* d) {
  if (!d) return CSA_ERR_INVALID_ARG;
  if (d->T < 0 || d->n_heads < 1 || d->head_dim < 1 || d->groups < 1 || d->rank < 1 || d->d_out < 0)
    return CSA_ERR_INVALID_ARG;
  if (d->n_heads % d->groups != 0) return CSA_ERR_INVALID_ARG;
  const long long K = static_cast<long long>(d->n_heads / d->groups) * d->head_dim;
  if (K % 64 != 0 || d->rank % 64 != 0 || d->d_out % 64 != 0) return CSA_ERR_UNSUPPORTED;
  if (K > (1 << 20) || static_cast<long long>(d->groups) * d->rank > (1 << 20) || d->d_out > (1 << 20))
    return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

// Tail rings in the state buffer, each bf16 [B, R, width] on a 256-byte boundary:
// CSA: Ca, Cb, Za, Zb (width d) then Ca_I, Cb_I, Za_I, Zb_I (width dI); HCA: Ca, Za.
struct CacheLayout {
  size_t off[8];
  int width[8];
  int n, R;
  size_t total;
};

CacheLayout cache_layout(const csa_cache_desc* d) {
  CacheLayout L{};
  L.R = d->overlap ? 2 * d->m : d->m;
  L.n = d->overlap ? (d->dI > 0 ? 8 : 4) : 2;
  size_t at = 0;
  for (int s = 0; s < L.n; ++s) {
    L.width[s] = s < 4 ? d->d : d->dI;
    L.off[s] = at;
    const size_t bytes = static_cast<size_t>(d->B) * L.R * L.width[s] * 2;
    at += (bytes + 255) & ~static_cast<size_t>(255);
  }
  L.total = at;
  return L;
}

}  // namespace

namespace csa {
void note_launches(int n) { count(n); }
}  // namespace csa

namespace {

// ---------------------------------------------------------------- indexer chunking
struct IndexPlan {
  int G;             // queries per group
  long long groups;  // total groups
  long long chunk;   // groups per score + top-k pass
  size_t score_bytes;  // fp32 score rows of one chunk (rounded up to 256 bytes)
  size_t cand_bytes;   // two-stage top-k candidates of one chunk (0 for rows <= one slice)
  size_t q8_bytes;     // low-precision indexer: e4m3 query rows of one chunk (0 otherwise)
  size_t wp_bytes;     // low-precision indexer: scaled head weights of one chunk
  // fused selection (scores never stored): the score kernel selects each query's top k from
  // per-CTA candidate lists that take the place of the score rows in the workspace
  bool sel;
  size_t sel_bytes;
};

inline bool is_lowp(const csa_index_desc* d) { return d->key_fmt == CSA_FMT_FP8_ROWSCALE_LOWP; }
inline bool fp8_keys(const csa_index_desc* d) {
  return d->key_fmt == CSA_FMT_FP8_ROWSCALE || d->key_fmt == CSA_FMT_FP8_ROWSCALE_LOWP;
}

bool index_desc_ok(const csa_index_desc* d) {
  if (!d) return false;
  if (d->B < 0 || d->Tq < 0 || d->N < 0 || d->m < 1) return false;
  if (d->n_heads < 1 || d->n_heads > 64) return false;
  if (d->head_dim != 64 && d->head_dim != 128) return false;
  if (d->k < 1 || d->k > 2048) return false;
  if (d->key_fmt != CSA_FMT_BF16 && d->key_fmt != CSA_FMT_FP8_ROWSCALE && d->key_fmt != CSA_FMT_FP8_ROWSCALE_LOWP)
    return false;
  if (d->key_fmt == CSA_FMT_FP8_ROWSCALE_LOWP && d->head_dim != 128) return false;
  if (d->score_fmt != CSA_SCORE_FP32 && d->score_fmt != CSA_SCORE_BF16) return false;
  if (d->select_mode != CSA_SELECT_AUTO && d->select_mode != CSA_SELECT_FUSED && d->select_mode != CSA_SELECT_STORED)
    return false;
  return true;
}

inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

IndexPlan plan_index(const csa_index_desc* d) {
  IndexPlan p;
  p.G = csa::index_grouping(d->n_heads, d->Tq).G;
  const long long gpb = (d->Tq + p.G - 1) / p.G;
  p.groups = static_cast<long long>(d->B) * gpb;
  const size_t per_group_scores = static_cast<size_t>(p.G) * (d->N > 0 ? d->N : 1) * sizeof(float);
  long long cg = static_cast<long long>(kScoreChunkCap / per_group_scores);
  if (cg < 1) cg = 1;
  p.chunk = p.groups < cg ? p.groups : cg;
  if (p.chunk < 1) p.chunk = 1;
  p.score_bytes = round256(static_cast<size_t>(p.chunk) * per_group_scores);
  // candidate bytes of the largest selector launch: the slicing depends on the launch's query
  // count, and launches of 128 queries or more select in one stage, so the largest need is among
  // 1..128 queries
  size_t cand = 0;
  const long long q_total = static_cast<long long>(d->B) * d->Tq;
  const long long q_cap = static_cast<long long>(p.chunk) * p.G;
  const long long q_max = q_total < q_cap ? q_total : q_cap;
  for (long long q = 1; q <= q_max && q <= 128; ++q) {
    const size_t c = csa::topk_candidate_bytes(static_cast<int>(q), d->N, d->k);
    if (c > cand) cand = c;
  }
  p.cand_bytes = round256(cand);
  const size_t lowp_rows = is_lowp(d) ? static_cast<size_t>(p.chunk) * p.G * d->n_heads : 0;
  p.q8_bytes = round256(lowp_rows * 128);
  p.wp_bytes = round256(lowp_rows * sizeof(float));
  // the fused selection walks whole groups per CTA, so it needs enough groups to balance the
  // persistent grid; its lists take the place of the score rows (below about 28K entries per row
  // they are the smaller of the two)
  const csa::IndexGrouping gr = csa::index_grouping(d->n_heads, d->Tq);
  // (AUTO: only rows of at least 16 k entries, where it measured faster than storing the rows)
  p.sel = CSA_INDEX_FUSED_SELECT && d->select_mode != CSA_SELECT_STORED && d->N > 0 &&
          csa::index_select_supported(gr, d->head_dim, fp8_keys(d), is_lowp(d), d->N) &&
          p.groups >= 4LL * csa::index_select_ctas() &&
          (d->select_mode == CSA_SELECT_FUSED || static_cast<long long>(d->N) >= 16LL * d->k);
  p.sel_bytes = p.sel ? round256(csa::index_select_bytes(gr, d->N)) : 0;
  return p;
}

// Workspace after the status word: the score rows (unless the caller stores them) and the two-
// stage selector's candidates, or the fused selection's lists, whichever is larger; then the
// low-precision indexer's query rows and weights.
size_t index_region_a(const IndexPlan& p, bool score_out) {
  const size_t unfused = (score_out ? 0 : p.score_bytes) + p.cand_bytes;
  const size_t fused = (p.sel && !score_out) ? p.sel_bytes : 0;
  return unfused > fused ? unfused : fused;
}

// ---------------------------------------------------------------- attention planning
bool attend_desc_ok(const csa_attend_desc* d, bool csa_mode) {
  if (!d) return false;
  if (d->B < 0 || d->Tq < 0 || d->N < 0) return false;
  if (d->d != 128 && d->d != 512) return false;
  if (d->H < 16 || d->H > 128 || (d->H % 16) != 0) return false;
  if (d->rope_dims < 0 || d->rope_dims > d->d || d->rope_dims > 2 * csa::kMaxRopePairs || (d->rope_dims & 1))
    return false;
  if (csa_mode && (d->k < 1 || d->k > 65536)) return false;
  if (!csa_mode && d->m < 1) return false;
  if (d->window < 0 || d->window > d->Wcap || (d->window > 0 && d->Wcap < 1)) return false;
  if (d->kv_fmt != CSA_FMT_BF16 && d->kv_fmt != CSA_FMT_FP8_MIXED) return false;
  if (d->kv_fmt == CSA_FMT_FP8_MIXED && d->d != 512) return false;
  if (!(d->scale >= 0.f) || !(d->eps >= 0.f)) return false;
  return true;
}

struct AttendPlan {
  int n_slots, split_slots, n_splits;
  size_t partial_bytes;
};

AttendPlan plan_attend(const csa_attend_desc* d, bool csa_mode) {
  AttendPlan p;
  p.n_slots = (csa_mode ? d->k : d->N) + d->window;
  if (p.n_slots < 1) p.n_slots = 1;
  // Decode (one query per sequence) splits the slot range in fixed pieces merged by a second
  // kernel: 192 slots (three 64-row chunks) for bf16 rows (64 heads per CTA), 128 slots (four
  // 32-row chunks) for the FP8 rows (16 heads per CTA, so four CTAs share a split's rows), and
  // 512 slots for dense HCA decode, whose rows run to N + window (measured at 1M context, batch
  // 8: 512 -> 59 us, 192 -> 91 us, 384 -> 83 us, 832 -> 77 us).  The split size depends on the
  // call and the row format only, never on the batch.  Prefill keeps one split per query.
  const int dec_split = d->kv_fmt == CSA_FMT_FP8_MIXED ? CSA_ATT_DECODE_SPLIT_FP8
                        : csa_mode                         ? CSA_ATT_DECODE_SPLIT
                                                           : CSA_ATT_DECODE_SPLIT_HCA;
  p.split_slots = (d->Tq == 1) ? dec_split : ((p.n_slots + 63) / 64) * 64;
  p.n_splits = (p.n_slots + p.split_slots - 1) / p.split_slots;
  if (p.n_splits < 1) p.n_splits = 1;
  p.partial_bytes = csa::attend_partial_bytes(d->B * d->Tq, d->H, d->d, p.n_splits);
  return p;
}

csa_status attend_common(const csa_attend_desc* d, bool csa_mode, const void* q, const void* kv,
                         const int32_t* idx, const void* win, const float* sink, const int32_t* q_pos,
                         void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!attend_desc_ok(d, csa_mode)) return CSA_ERR_INVALID_ARG;
  const long long Q = static_cast<long long>(d->B) * d->Tq;
  if (!ws) return CSA_ERR_WORKSPACE;
  const AttendPlan plan = plan_attend(d, csa_mode);
  if (plan.n_splits > 65535) return CSA_ERR_UNSUPPORTED;
  if (ws_bytes < csa::kStatusBytes + plan.partial_bytes) return CSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA_ERR_INVALID_ARG;
  if (Q == 0) return CSA_OK;
  if (Q > 2147483647LL) return CSA_ERR_UNSUPPORTED;
  if (!q || !sink || !q_pos || !out) return CSA_ERR_INVALID_ARG;
  if (!kv && (d->N > 0)) return CSA_ERR_INVALID_ARG;
  if (csa_mode && !idx) return CSA_ERR_INVALID_ARG;
  if (!win && d->window > 0) return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || (kv && !aligned16(kv)) || (win && !aligned16(win)) || !aligned16(out))
    return CSA_ERR_INVALID_ARG;
  if ((d->flags & CSA_ATTEND_WRITE_LSE) && !lse) return CSA_ERR_INVALID_ARG;

  csa::AttendArgs a{};
  a.q = q; a.kv = kv; a.idx = csa_mode ? idx : nullptr; a.win = win; a.sink = sink; a.q_pos = q_pos;
  a.out = out; a.lse = (d->flags & CSA_ATTEND_WRITE_LSE) ? lse : nullptr;
  a.status = static_cast<int32_t*>(ws);
  a.partial = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + csa::kStatusBytes);
  a.B = d->B; a.Tq = d->Tq; a.N = d->N; a.H = d->H; a.d = d->d; a.k = csa_mode ? d->k : 0;
  a.m = csa_mode ? 1 : d->m;
  a.Wcap = d->Wcap > 0 ? d->Wcap : 1; a.window = d->window;
  a.fp8 = d->kv_fmt == CSA_FMT_FP8_MIXED;
  a.q_norm_rope = (d->flags & CSA_ATTEND_Q_NORM_ROPE) != 0;
  a.out_unrotate = (d->flags & CSA_ATTEND_OUT_UNROTATE) != 0;
  a.scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(static_cast<float>(d->d));
  a.eps = d->eps;
  a.n_slots = plan.n_slots; a.split_slots = plan.split_slots; a.n_splits = plan.n_splits;
  if (!make_rope(d->rope_dims, d->rope_theta, d->inv_freq, &a.rp)) return CSA_ERR_INVALID_ARG;
  int launches = 0;
  const cudaError_t e = csa::launch_attend(a, stream, &launches);
  count(launches);
  if (e == cudaErrorInvalidValue) return CSA_ERR_UNSUPPORTED;
  return from_cuda(e);
}

}  // namespace

extern "C" {

csa_status csa_compress(const csa_compress_desc* d, const void* Ca, const void* Cb, const void* Za,
                        const void* Zb, const float* bias_a, const float* bias_b, const float* gamma,
                        void* out, csa_stream_t stream) {
  if (!d) return CSA_ERR_INVALID_ARG;
  if (d->B < 0 || d->T < 0 || d->m < 1 || d->m > 256) return CSA_ERR_INVALID_ARG;
  if (!compress_width_ok(d->d)) return CSA_ERR_UNSUPPORTED;
  if (d->rope_dims < 0 || d->rope_dims > d->d || (d->rope_dims % 8) != 0 ||
      d->rope_dims > 2 * csa::kMaxRopePairs)
    return CSA_ERR_UNSUPPORTED;
  if (d->out_fmt != CSA_FMT_BF16) return CSA_ERR_UNSUPPORTED;
  if (!(d->eps >= 0.f)) return CSA_ERR_INVALID_ARG;
  const int N = d->T / d->m;
  if (static_cast<long long>(d->B) * N == 0) return CSA_OK;
  if (!Ca || !Za || !out) return CSA_ERR_INVALID_ARG;
  if (d->overlap && (!Cb || !Zb)) return CSA_ERR_INVALID_ARG;
  if (!aligned16(Ca) || !aligned16(Za) || !aligned16(out) || (d->overlap && (!aligned16(Cb) || !aligned16(Zb))) ||
      (bias_a && !aligned16(bias_a)) || (bias_b && !aligned16(bias_b)) || (gamma && !aligned16(gamma)))
    return CSA_ERR_INVALID_ARG;
  csa::CompressArgs a{};
  a.Ca = Ca; a.Cb = d->overlap ? Cb : nullptr; a.Za = Za; a.Zb = d->overlap ? Zb : nullptr;
  a.bias_a = bias_a; a.bias_b = d->overlap ? bias_b : nullptr; a.gamma = gamma; a.out = out;
  a.B = d->B; a.T = d->T; a.d = d->d; a.m = d->m; a.N = N; a.overlap = d->overlap ? 1 : 0;
  a.norm = (d->flags & CSA_COMPRESS_NORM) != 0;
  a.rope = (d->flags & CSA_COMPRESS_ROPE) != 0 && d->rope_dims > 0;
  a.pos_shift = d->pos_shift;
  a.eps = d->eps;
  a.out_N = N;
  if (!make_rope(d->rope_dims, d->rope_theta, d->inv_freq, &a.rp)) return CSA_ERR_INVALID_ARG;
  int launches = 0;
  const cudaError_t e = csa::launch_compress(a, reinterpret_cast<cudaStream_t>(stream), &launches);
  count(launches);
  return from_cuda(e);
}

size_t csa_out_proj_workspace(const csa_out_proj_desc* d) {
  return out_proj_check(d) == CSA_OK ? csa::kStatusBytes : 0;
}

csa_status csa_out_proj(const csa_out_proj_desc* d, const void* O, const void* W_down, const void* W_proj, void* z,
                        void* y, void* ws, size_t ws_bytes, csa_stream_t stream_) {
  const csa_status st = out_proj_check(d);
  if (st != CSA_OK) return st;
  if (!ws || ws_bytes < csa::kStatusBytes) return CSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA_ERR_INVALID_ARG;
  if (d->T == 0) return CSA_OK;
  if (!O || !W_down || !z || !aligned16(O) || !aligned16(W_down) || !aligned16(z)) return CSA_ERR_INVALID_ARG;
  if (d->d_out > 0 && (!W_proj || !y || !aligned16(W_proj) || !aligned16(y))) return CSA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int32_t* status = static_cast<int32_t*>(ws);
  const int K = d->n_heads / d->groups * d->head_dim;
  int launches = 0;
  cudaError_t e = csa::launch_gemm_tn(O, W_down, z, d->T, d->rank, K, d->groups, status, stream, &launches);
  if (e == cudaSuccess && d->d_out > 0)
    e = csa::launch_gemm_tn(z, W_proj, y, d->T, d->d_out, d->groups * d->rank, 1, status, stream, &launches);
  count(launches);
  return from_cuda(e);
}

size_t csa_cache_state_bytes(const csa_cache_desc* d) {
  if (cache_desc_check(d) != CSA_OK) return 0;
  return cache_layout(d).total;
}

csa_status csa_cache_append(const csa_cache_desc* d, int64_t t0, int n, const csa_cache_rows* rows,
                            const csa_cache_params* params, const csa_cache_buffers* bufs, csa_stream_t stream_) {
  const csa_status st = cache_desc_check(d);
  if (st != CSA_OK) return st;
  if (t0 < 0 || n < 0 || t0 + n > INT32_MAX) return CSA_ERR_INVALID_ARG;
  const int T0 = static_cast<int>(t0);
  const int i_begin = T0 / d->m;
  const int i_end = (T0 + n) / d->m;
  if (i_end > d->N_cap) return CSA_ERR_INVALID_ARG;
  if (n == 0 || d->B == 0) return CSA_OK;
  if (!rows || !bufs) return CSA_ERR_INVALID_ARG;
  const bool idx = d->dI > 0;
  const void* in_main[4] = {rows->Ca, rows->Cb, rows->Za, rows->Zb};
  const void* in_idx[4] = {rows->Ca_I, rows->Cb_I, rows->Za_I, rows->Zb_I};
  for (int s = 0; s < 4; ++s) {
    const bool used = d->overlap || s == 0 || s == 2;
    if (used && (!in_main[s] || !aligned16(in_main[s]))) return CSA_ERR_INVALID_ARG;
    if (idx && (!in_idx[s] || !aligned16(in_idx[s]))) return CSA_ERR_INVALID_ARG;
  }
  if (!rows->win || !aligned16(rows->win) || !bufs->win || !aligned16(bufs->win) || !bufs->state ||
      !aligned16(bufs->state))
    return CSA_ERR_INVALID_ARG;
  if (i_end > i_begin && (!bufs->kv || !aligned16(bufs->kv) || (idx && (!bufs->kI || !aligned16(bufs->kI)))))
    return CSA_ERR_INVALID_ARG;
  const csa_cache_params none{};
  const csa_cache_params& p = params ? *params : none;
  const float* fptr[6] = {p.bias_a, p.bias_b, p.gamma, p.bias_a_I, p.bias_b_I, p.gamma_I};
  for (const float* f : fptr)
    if (f && !aligned16(f)) return CSA_ERR_INVALID_ARG;

  const CacheLayout L = cache_layout(d);
  char* state = static_cast<char*>(bufs->state);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int launches = 0;
  cudaError_t e = cudaSuccess;
  if (i_end > i_begin) {
    for (int part = 0; part < (idx ? 2 : 1) && e == cudaSuccess; ++part) {
      const void* const* in = part ? in_idx : in_main;
      const int s0 = part ? 4 : 0;     // first ring of this part in the layout
      csa::CompressArgs a{};
      a.Ca = in[0]; a.Za = in[2];
      a.Cb = d->overlap ? in[1] : nullptr; a.Zb = d->overlap ? in[3] : nullptr;
      a.bias_a = part ? p.bias_a_I : p.bias_a;
      a.bias_b = d->overlap ? (part ? p.bias_b_I : p.bias_b) : nullptr;
      a.gamma = part ? p.gamma_I : p.gamma;
      a.out = part ? bufs->kI : bufs->kv;
      a.B = d->B; a.T = n; a.d = part ? d->dI : d->d; a.m = d->m; a.N = i_end - i_begin;
      a.overlap = d->overlap ? 1 : 0;
      const unsigned fl = part ? d->index_flags : d->flags;
      a.norm = (fl & CSA_COMPRESS_NORM) != 0;
      a.rope = !part && (fl & CSA_COMPRESS_ROPE) != 0 && d->rope_dims > 0;
      a.eps = d->eps;
      a.t0 = T0; a.i_begin = i_begin; a.out_N = d->N_cap;
      a.ring.R = L.R;
      a.ring.Ca = state + L.off[s0 + 0];
      a.ring.Za = state + L.off[s0 + (d->overlap ? 2 : 1)];
      a.ring.Cb = d->overlap ? state + L.off[s0 + 1] : nullptr;
      a.ring.Zb = d->overlap ? state + L.off[s0 + 3] : nullptr;
      if (!make_rope(part ? 0 : d->rope_dims, d->rope_theta, d->inv_freq, &a.rp)) return CSA_ERR_INVALID_ARG;
      e = csa::launch_compress(a, stream, &launches);
    }
  }
  if (e == cudaSuccess) {
    csa::RingArgs r{};
    r.B = d->B; r.t0 = T0; r.n = n;
    const void* srcs[8];
    int ns = 0;
    if (d->overlap) {
      for (int s = 0; s < 4; ++s) srcs[ns++] = in_main[s];
      if (idx)
        for (int s = 0; s < 4; ++s) srcs[ns++] = in_idx[s];
    } else {
      srcs[ns++] = in_main[0];
      srcs[ns++] = in_main[2];
    }
    for (int s = 0; s < ns; ++s) r.job[s] = csa::RingJob{srcs[s], state + L.off[s], L.width[s], L.R};
    r.job[ns] = csa::RingJob{rows->win, bufs->win, d->d, d->Wcap};
    r.n_jobs = ns + 1;
    e = csa::launch_ring_rows(r, stream, &launches);
  }
  count(launches);
  return from_cuda(e);
}

size_t csa_index_topk_workspace(const csa_index_desc* d) {
  if (!index_desc_ok(d)) return 0;
  const IndexPlan p = plan_index(d);
  return csa::kStatusBytes + index_region_a(p, false) + p.q8_bytes + p.wp_bytes;
}

csa_status csa_index_topk(const csa_index_desc* d, const void* qI, const float* w, const void* kI,
                          const float* kI_scale, const int32_t* q_pos, int32_t* idx_out, float* score_out,
                          void* ws, size_t ws_bytes, csa_stream_t stream_) {
  if (!index_desc_ok(d)) return CSA_ERR_INVALID_ARG;
  if (d->N > 262144) return CSA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const IndexPlan plan = plan_index(d);
  if (!ws) return CSA_ERR_WORKSPACE;
  if (ws_bytes < csa::kStatusBytes + index_region_a(plan, score_out != nullptr) + plan.q8_bytes + plan.wp_bytes)
    return CSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA_ERR_INVALID_ARG;
  const long long Q = static_cast<long long>(d->B) * d->Tq;
  if (Q == 0) return CSA_OK;
  if (!qI || !w || !q_pos || !idx_out || (!kI && d->N > 0)) return CSA_ERR_INVALID_ARG;
  const bool fp8 = fp8_keys(d);
  const bool lowp = is_lowp(d);
  if (fp8 && !kI_scale && d->N > 0) return CSA_ERR_INVALID_ARG;
  if (!aligned16(qI) || (kI && !aligned16(kI))) return CSA_ERR_INVALID_ARG;

  csa::IndexArgs ia{};
  ia.qI = qI; ia.w = w; ia.kI = kI; ia.kI_scale = kI_scale; ia.q_pos = q_pos;
  ia.B = d->B; ia.Tq = d->Tq; ia.N = d->N; ia.nI = d->n_heads; ia.dI = d->head_dim; ia.m = d->m;
  ia.fp8 = fp8 ? 1 : 0;
  ia.bf16_scores = d->score_fmt == CSA_SCORE_BF16 ? 1 : 0;
  ia.status = static_cast<int32_t*>(ws);
  const csa::IndexGrouping grouping = csa::index_grouping(d->n_heads, d->Tq);
  csa::TopkArgs ta{};
  ta.q_pos = q_pos; ta.idx_out = idx_out; ta.status = static_cast<int32_t*>(ws);
  ta.Tq = d->Tq; ta.N = d->N; ta.k = d->k; ta.m = d->m;
  ta.key_shift = d->score_fmt == CSA_SCORE_BF16 ? 16 : 0;

  const long long gpb = (d->Tq + plan.G - 1) / plan.G;
  unsigned char* wsb = static_cast<unsigned char*>(ws);
  unsigned char* after_scores = wsb + csa::kStatusBytes + (score_out ? 0 : plan.score_bytes);
  void* cand = plan.cand_bytes ? after_scores : nullptr;
  unsigned char* q8 = wsb + csa::kStatusBytes + index_region_a(plan, score_out != nullptr);   // low-precision query rows
  float* wp = reinterpret_cast<float*>(q8 + plan.q8_bytes);
  ia.lowp = lowp ? 1 : 0;
  int launches = 0;
  cudaError_t e = cudaSuccess;
  if (d->N == 0) {
    // nothing visible anywhere: the selector only pads
    ta.scores = nullptr; ta.q_begin = 0; ta.q_count = static_cast<int>(Q); ta.score_row_offset = 0;
    e = csa::launch_topk(ta, cand, stream, &launches);
    count(launches);
    return from_cuda(e);
  }
  if (plan.sel && !score_out) {
    // scores and selection in one kernel: the candidate lists sit where the score rows would
    ia.idx_out = idx_out;
    ia.k = d->k;
    ia.cand = reinterpret_cast<unsigned long long*>(wsb + csa::kStatusBytes);
    ia.cand_cap = csa::index_select_cap(d->N);
    ia.cand_ctas = csa::index_select_ctas();
    ia.score_row_offset = 0;
    // one launch over every group; the low-precision indexer quantises its queries per chunk
    const long long sstep = lowp ? plan.chunk : plan.groups;
    for (long long g0 = 0; g0 < plan.groups && e == cudaSuccess; g0 += sstep) {
      const long long g1 = (g0 + sstep < plan.groups) ? g0 + sstep : plan.groups;
      ia.q_begin = static_cast<int>(g0);
      ia.q_count = static_cast<int>(g1 - g0);
      if (lowp) {
        const long long q_first = (g0 / gpb) * d->Tq + (g0 % gpb) * plan.G;
        const long long gl = g1 - 1;
        const long long q_last = (gl / gpb) * d->Tq + (gl % gpb) * plan.G +
                                 ((d->Tq - (gl % gpb) * plan.G) < plan.G ? (d->Tq - (gl % gpb) * plan.G) : plan.G);
        const long long row0 = q_first * d->n_heads;
        e = csa::launch_quant_q(qI, w, q8, wp, row0, (q_last - q_first) * d->n_heads, stream, &launches);
        if (e != cudaSuccess) break;
        ia.qI = q8 - row0 * 128;
        ia.w = wp - row0;
      }
      e = csa::launch_index_select(ia, grouping, stream, &launches);
    }
    count(launches);
    if (e == cudaErrorInvalidValue) return CSA_ERR_UNSUPPORTED;
    return from_cuda(e);
  }
  const long long step = plan.chunk;
  for (long long g0 = 0; g0 < plan.groups && e == cudaSuccess; g0 += step) {
    const long long g1 = (g0 + step < plan.groups) ? g0 + step : plan.groups;
    const long long q_first = (g0 / gpb) * d->Tq + (g0 % gpb) * plan.G;
    const long long gl = g1 - 1;
    const long long q_last = (gl / gpb) * d->Tq + (gl % gpb) * plan.G +
                             ((d->Tq - (gl % gpb) * plan.G) < plan.G ? (d->Tq - (gl % gpb) * plan.G) : plan.G);
    float* scores = score_out ? score_out : reinterpret_cast<float*>(wsb + csa::kStatusBytes);
    ia.scores = scores;
    ia.q_begin = static_cast<int>(g0);
    ia.q_count = static_cast<int>(g1 - g0);
    ia.score_row_offset = score_out ? 0 : static_cast<int>(q_first);
    if (lowp) {
      // this chunk's query rows, quantised into the workspace; the score kernel addresses them by
      // global query index, so its base pointers step back by the chunk's first row
      const long long row0 = q_first * d->n_heads;
      e = csa::launch_quant_q(qI, w, q8, wp, row0, (q_last - q_first) * d->n_heads, stream, &launches);
      if (e != cudaSuccess) break;
      ia.qI = q8 - row0 * 128;
      ia.w = wp - row0;
    }
    e = csa::launch_index_score_groups(ia, grouping, score_out ? 1 : 0, stream, &launches);
    if (e != cudaSuccess) break;
    ta.scores = scores;
    ta.q_begin = static_cast<int>(q_first);
    ta.q_count = static_cast<int>(q_last - q_first);
    ta.score_row_offset = ia.score_row_offset;
    e = csa::launch_topk(ta, cand, stream, &launches);
  }
  count(launches);
  if (e == cudaErrorInvalidValue) return CSA_ERR_UNSUPPORTED;
  return from_cuda(e);
}

// low-precision indexer: e4m3 query rows and scaled weights of all B*Tq queries
size_t lowp_all_bytes(const csa_index_desc* d) {
  if (!is_lowp(d)) return 0;
  const size_t rows = static_cast<size_t>(d->B) * d->Tq * d->n_heads;
  return round256(rows * 128) + round256(rows * sizeof(float));
}

size_t csa_index_score_workspace(const csa_index_desc* d) {
  if (!index_desc_ok(d)) return 0;
  return csa::kStatusBytes + lowp_all_bytes(d);
}

csa_status csa_index_score(const csa_index_desc* d, const void* qI, const float* w, const void* kI,
                           const float* kI_scale, const int32_t* q_pos, float* score_out, void* ws,
                           size_t ws_bytes, csa_stream_t stream_) {
  if (!index_desc_ok(d)) return CSA_ERR_INVALID_ARG;
  if (d->N > 262144) return CSA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!ws) return CSA_ERR_WORKSPACE;
  if (ws_bytes < csa::kStatusBytes + lowp_all_bytes(d)) return CSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA_ERR_INVALID_ARG;
  const long long Q = static_cast<long long>(d->B) * d->Tq;
  if (Q == 0 || d->N == 0) return CSA_OK;
  if (!qI || !w || !q_pos || !kI || !score_out) return CSA_ERR_INVALID_ARG;
  const bool fp8 = fp8_keys(d);
  if (fp8 && !kI_scale) return CSA_ERR_INVALID_ARG;
  if (!aligned16(qI) || !aligned16(kI)) return CSA_ERR_INVALID_ARG;
  const IndexPlan plan = plan_index(d);
  if (plan.groups > 2147483647LL) return CSA_ERR_UNSUPPORTED;
  csa::IndexArgs ia{};
  ia.qI = qI; ia.w = w; ia.kI = kI; ia.kI_scale = kI_scale; ia.q_pos = q_pos;
  ia.B = d->B; ia.Tq = d->Tq; ia.N = d->N; ia.nI = d->n_heads; ia.dI = d->head_dim; ia.m = d->m;
  ia.fp8 = fp8 ? 1 : 0;
  ia.bf16_scores = d->score_fmt == CSA_SCORE_BF16 ? 1 : 0;
  ia.status = static_cast<int32_t*>(ws);
  ia.scores = score_out;
  ia.q_begin = 0;
  ia.q_count = static_cast<int>(plan.groups);
  ia.score_row_offset = 0;
  int launches = 0;
  cudaError_t e = cudaSuccess;
  if (is_lowp(d)) {
    const long long rows = Q * d->n_heads;
    unsigned char* q8 = static_cast<unsigned char*>(ws) + csa::kStatusBytes;
    float* wp = reinterpret_cast<float*>(q8 + round256(static_cast<size_t>(rows) * 128));
    e = csa::launch_quant_q(qI, w, q8, wp, 0, rows, stream, &launches);
    ia.qI = q8;
    ia.w = wp;
    ia.lowp = 1;
  }
  if (e == cudaSuccess)
    e = csa::launch_index_score_groups(ia, csa::index_grouping(d->n_heads, d->Tq), 0, stream, &launches);
  count(launches);
  if (e == cudaErrorInvalidValue) return CSA_ERR_UNSUPPORTED;
  return from_cuda(e);
}

size_t csa_topk_workspace(const csa_index_desc* d) {
  if (!index_desc_ok(d)) return 0;
  const long long Q = static_cast<long long>(d->B) * d->Tq;
  if (Q > 2147483647LL) return 0;
  return csa::kStatusBytes + round256(csa::topk_candidate_bytes(static_cast<int>(Q), d->N, d->k));
}

csa_status csa_topk(const csa_index_desc* d, const float* scores, const int32_t* q_pos, int32_t* idx_out,
                    void* ws, size_t ws_bytes, csa_stream_t stream_) {
  if (!index_desc_ok(d)) return CSA_ERR_INVALID_ARG;
  if (d->N > 262144) return CSA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!ws) return CSA_ERR_WORKSPACE;
  const long long Q = static_cast<long long>(d->B) * d->Tq;
  if (Q > 2147483647LL) return CSA_ERR_UNSUPPORTED;
  const size_t cand = round256(csa::topk_candidate_bytes(static_cast<int>(Q), d->N, d->k));
  if (ws_bytes < csa::kStatusBytes + cand) return CSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA_ERR_INVALID_ARG;
  if (Q == 0) return CSA_OK;
  if (!q_pos || !idx_out || (!scores && d->N > 0)) return CSA_ERR_INVALID_ARG;
  csa::TopkArgs ta{};
  ta.scores = scores; ta.q_pos = q_pos; ta.idx_out = idx_out; ta.status = static_cast<int32_t*>(ws);
  ta.Tq = d->Tq; ta.N = d->N; ta.k = d->k; ta.m = d->m;
  ta.key_shift = d->score_fmt == CSA_SCORE_BF16 ? 16 : 0;
  ta.q_begin = 0; ta.q_count = static_cast<int>(Q); ta.score_row_offset = 0;
  int launches = 0;
  const cudaError_t e =
      csa::launch_topk(ta, cand ? static_cast<unsigned char*>(ws) + csa::kStatusBytes : nullptr, stream, &launches);
  count(launches);
  if (e == cudaErrorInvalidValue) return CSA_ERR_UNSUPPORTED;
  return from_cuda(e);
}

size_t csa_attend_workspace(const csa_attend_desc* d) {
  if (!attend_desc_ok(d, true)) return 0;
  return csa::kStatusBytes + plan_attend(d, true).partial_bytes;
}

size_t hca_attend_workspace(const csa_attend_desc* d) {
  if (!attend_desc_ok(d, false)) return 0;
  return csa::kStatusBytes + plan_attend(d, false).partial_bytes;
}

csa_status csa_attend(const csa_attend_desc* d, const void* q, const void* kv, const int32_t* idx,
                      const void* win, const float* sink, const int32_t* q_pos, void* out, float* lse,
                      void* ws, size_t ws_bytes, csa_stream_t stream) {
  return attend_common(d, true, q, kv, idx, win, sink, q_pos, out, lse, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

csa_status hca_attend(const csa_attend_desc* d, const void* q, const void* kv, const void* win,
                      const float* sink, const int32_t* q_pos, void* out, float* lse, void* ws,
                      size_t ws_bytes, csa_stream_t stream) {
  return attend_common(d, false, q, kv, nullptr, win, sink, q_pos, out, lse, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

csa_status csa_read_device_status(const void* ws, csa_stream_t stream, int32_t* detail) {
  if (!ws) return CSA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
  int32_t h[2] = {0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  if (detail) *detail = h[1];
  if (h[0] == 0) return CSA_OK;
  return h[0] == CSA_ERR_TIMEOUT ? CSA_ERR_TIMEOUT : CSA_ERR_DEVICE_CHECK;
}

csa_status csa_clear_device_status(void* ws, csa_stream_t stream) {
  if (!ws) return CSA_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, 8, reinterpret_cast<cudaStream_t>(stream)));
}

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_DEVICE_CHECK: return "device-side range check failed";
    case CSA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

uint64_t csa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
