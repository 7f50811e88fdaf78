// Internal helpers shared by the library's kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "../../include/csa.h"

namespace csa {

constexpr int kMaxRopePairs = 64;   // rope_dims <= 128

// RoPE frequencies, computed on the host and passed by value.  Pair j turns by inv_freq_j radians
// per position; phase[j] is that turn as a 64-bit binary fraction of a revolution,
// round(inv_freq_j / (2 pi) * 2^64) mod 2^64, so the angle of an integer position reduces modulo
// 2 pi exactly in integer arithmetic (no FP64 on the device).
struct RopeParams {
  int r;                    // rotated dims (even), the last r dims of each vector
  unsigned long long phase[kMaxRopePairs];
};

// Status word at the start of every workspace: {code, detail, pad, pad}.
constexpr size_t kStatusBytes = 256;

// Adds to the library's count of kernel launches (csa_launch_count).
void note_launches(int n);

// Order-preserving 32-bit key of an fp32 score (unsigned comparison of keys = comparison of the
// scores); -0 and +0 map to the same key, so equal scores tie by entry index.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Closed compressed blocks visible to position t: s < floor((t+1)/m), clipped to [0, N].
__host__ __device__ __forceinline__ int n_visible(int t, int m, int N) {
  const long long v = (static_cast<long long>(t) + 1) / m;
  return v <= 0 ? 0 : (v >= N ? N : static_cast<int>(v));
}

// Programmatic dependent launch.  Every kernel is launched with programmatic stream
// serialization (launch_k), so its CTAs may be scheduled while the previous kernel on the stream
// is still finishing; grid_dep_wait() then blocks until that kernel has completed and its memory
// writes are visible.  Each kernel calls grid_dep_wait() before its first global-memory access
// (read or write), and grid_dep_launch() right after it: the next kernel's CTAs may then take
// SM resources as this kernel's CTAs retire, which hides the launch gap between them.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ void report_error(int32_t* status, int32_t code, int32_t detail) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// cos/sin of pos * inv_freq.  The product and its reduction modulo 2*pi run in double so that
// positions up to 2^20 and beyond keep full fp32 accuracy in the angle; the reduced angle lies in
// [-pi, pi], where the hardware sine/cosine (__sincosf, absolute error about 2^-21) is far more
// accurate than the bf16 values it rotates and needs no general-range reduction.
// cos and sin of the RoPE angle pos * inv_freq: pos * phase mod 2^64 is the angle's fraction of a
// revolution (to 2^-64 per unit of pos); its top 32 bits, read as a signed fraction, give the angle
// reduced to [-pi, pi) for the fast sine and cosine.
__device__ __forceinline__ void rope_cos_sin(long long pos, unsigned long long phase, float& c, float& s) {
  const unsigned long long turn = static_cast<unsigned long long>(pos) * phase;
  const float ang = __fmul_rn(static_cast<float>(static_cast<int>(turn >> 32)), 1.46291807926715968e-9f);  // 2 pi / 2^32
  __sincosf(ang, &s, &c);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// e4m3 pair -> f16 pair, exact (every e4m3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint16_t v) {
  uint32_t h2;
  asm("{cvt.rn.f16x2.e4m3x2 %0, %1;}" : "=r"(h2) : "h"(v));
  return h2;
}

// e4m3 pair -> two floats (exact) via the hardware f16x2 conversion.
__device__ __forceinline__ void e4m3x2_to_float2(uint16_t v, float& lo, float& hi) {
  uint32_t h2;
  asm("{cvt.rn.f16x2.e4m3x2 %0, %1;}" : "=r"(h2) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(hh);
  lo = f.x;
  hi = f.y;
}

// ------------------------------------------------------------------ warp-level MMA (bf16)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ------------------------------------------------------------------ cp.async

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const int n = valid ? 16 : 0;   // src-size 0 => the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
               :: "r"(smem_u32(smem)), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N)); }

}  // namespace csa

// ------------------------------------------------------------------ launchers (internal)
namespace csa {

// Rows of tokens before the chunk (cache append): stream rows of token u at slot u mod R of
// [B, R, d] rings.  Unused (R = 0) when the chunk starts at token 0.
struct CompressRing {
  const void *Ca, *Cb, *Za, *Zb;
  int R;
};

struct CompressArgs {
  const void *Ca, *Cb, *Za, *Zb;   // the chunk's rows: tokens t0 .. t0+T-1, [B, T, d]
  const float *bias_a, *bias_b, *gamma;
  void* out;                       // [B, out_N, d]: entry i at row i
  int B, T, d, m, N, overlap, norm, rope;
  int pos_shift;
  float eps;
  RopeParams rp;
  int t0;                          // first token of the chunk (0 for a whole-sequence call)
  int i_begin;                     // entries i_begin .. i_begin+N-1 are computed
  int out_N;
  CompressRing ring;
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s, int* launches);

// Row scatter into rings (cache append): job j copies rows of tokens [lo, t0+n) of src
// [B, n, w] to dst [B, R, w] slot u mod R, lo = max(t0, t0+n-R).
struct RingJob {
  const void* src;
  void* dst;
  int w, R;
};
constexpr int kMaxRingJobs = 9;
struct RingArgs {
  RingJob job[kMaxRingJobs];
  int n_jobs, B, t0, n;
};
cudaError_t launch_ring_rows(const RingArgs& a, cudaStream_t s, int* launches);

// C[m][u][n] = sum_k A[m][u][k] B[u][n][k] (bf16 in, fp32 accumulate, bf16 out); A [M][G][K],
// B [G][N][K], C [M][G][N]; K and N multiples of 64.
cudaError_t launch_gemm_tn(const void* A, const void* B, void* C, int M, int N, int K, int G, int32_t* status,
                           cudaStream_t s, int* launches);
int gemm_tn_tile_n(int M, int N, int K, int G);

struct IndexArgs {
  const void* qI;
  const float* w;
  const void* kI;
  const float* kI_scale;
  const int32_t* q_pos;
  float* scores;            // score rows of N floats
  int32_t* status;          // workspace status word (bounded-wait timeouts)
  int B, Tq, N, nI, dI, m, fp8;
  int lowp;                 // qI is the e4m3 query (q8) and w the scaled weights: FP8 tensor cores
  int bf16_scores;          // round each score to bf16 (RNE) before it is stored
  int q_begin, q_count;     // range of query GROUPS (G consecutive queries of one sequence)
  int score_row_offset;     // flattened query q (= b*Tq + i) owns score row q - score_row_offset
  // fused selection (launch_index_select): the top-k rows, k, and the candidate lists (two
  // buffers of G lists of cand_cap (key, entry) slots per CTA, for cand_ctas CTAs; a list is four
  // sub-lists of cand_cap / 4 slots)
  int32_t* idx_out;
  unsigned long long* cand;
  int cand_cap, cand_ctas, k;
};

// How the indexer packs queries into one tensor-core N dimension: heads padded to NHP (a power
// of two >= 16), G consecutive queries of one sequence per group, NCOL = G * NHP <= 256 columns.
struct IndexGrouping {
  int NHP, G, NCOL;
};
inline IndexGrouping index_grouping(int nI, int Tq) {
  IndexGrouping g;
  int nhp = 16;
  while (nhp < nI) nhp <<= 1;
  int G = 1;
  while (G < Tq && G * nhp < 256) G <<= 1;
  g.NHP = nhp;
  g.G = G;
  g.NCOL = G * nhp;
  return g;
}

// Scores for the query groups [q_begin, q_begin + q_count).  fill_invisible: also write -inf
// for every s in [N_vis, N) so that the rows are complete.
// Low-precision indexer query: rows [row0, row0 + rows) of qI ([.., 128] bf16) and w -> q8
// ([rows, 128] e4m3) and wp ([rows] fp32), both counted from row0.
cudaError_t launch_quant_q(const void* qI, const float* w, void* q8, float* wp, long long row0, long long rows,
                           cudaStream_t s, int* launches);
cudaError_t launch_index_score_groups(const IndexArgs& a, const IndexGrouping& gr, int fill_invisible,
                                      cudaStream_t s, int* launches);
// Scores and top-k in one kernel (the selection fused into the score kernel's epilogue): only for
// groupings of 4 queries x 64 heads (256 MMA columns), rows of at most 32768 entries, bf16 keys
// or the low-precision indexer.  index_select_supported says whether a call of this shape takes it;
// index_select_bytes is the candidate-list workspace it needs on the current device.
bool index_select_supported(const IndexGrouping& gr, int dI, int fp8, int lowp, int N);
size_t index_select_bytes(const IndexGrouping& gr, int N);
int index_select_cap(int N);
int index_select_ctas();
cudaError_t launch_index_select(const IndexArgs& a, const IndexGrouping& gr, cudaStream_t s, int* launches);

struct TopkArgs {
  const float* scores;
  const int32_t* q_pos;
  int32_t* idx_out;
  int32_t* status;
  int Tq, N, k, m;
  int q_begin, q_count;
  int score_row_offset;
  int key_shift;            // 16 for scores rounded to bf16 (16-bit order keys), else 0
};
// Rows longer than one selection slice are selected in two stages; the first writes
// topk_candidate_bytes(Q, N, k) bytes of (key, index) candidates for a launch over Q queries to
// cand_ws (8-byte aligned), which may be null when that size is 0.
int topk_slices(int Q, int N, int k);
size_t topk_candidate_bytes(int Q, int N, int k);
cudaError_t launch_topk(const TopkArgs& a, void* cand_ws, cudaStream_t s, int* launches);

struct AttendArgs {
  const void* q;
  const void* kv;
  const int32_t* idx;       // nullptr => dense (HCA)
  const void* win;
  const float* sink;
  const int32_t* q_pos;
  void* out;
  float* lse;
  float* partial;           // workspace for split partials
  int32_t* status;
  int B, Tq, N, H, d, k, m, Wcap, window, fp8;
  int q_norm_rope, out_unrotate;
  float scale, eps;
  int n_slots;              // slots per query (k + window, or N + window)
  int split_slots;          // slots per split (multiple of the chunk size)
  int n_splits;
  int cluster_merge;        // splits of a query merged inside a thread-block cluster (tensor-core kernel)
  RopeParams rp;
};
size_t attend_partial_bytes(int Q, int H, int d, int n_splits);
// Split merge (second kernel) for n_splits > 1.
cudaError_t launch_attend_combine(const AttendArgs& a, cudaStream_t s, int* launches);


cudaError_t launch_attend(const AttendArgs& a, cudaStream_t s, int* launches);
// The tensor-core kernel for 512-dim bf16 rows and 64-head groups (attend_tc.cu).
bool attend_tc_supported(const AttendArgs& a);
cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s, int* launches);



}  // namespace csa
