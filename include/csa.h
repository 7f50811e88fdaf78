/*
 * csa.h -- C ABI of the B300 (sm_103a) library for DeepSeek-V4 hybrid compressed attention.
 *
 * The method (as explained on "DeepSeek V4 模型技术大全", wineandchord.com, chapter "Hybrid
 * Attention", and "DeepSeek-V4 技术解析", chang-wenbin.github.io, section 2.1):
 *   CSA  compress every m = 4 tokens into one shared K=V entry (softmax-gated, overlapped over
 *        2m rows), RMSNorm it and rotate its last 64 dims; score every closed entry with the
 *        lightning indexer; keep the top-k per query; attend over those entries plus an
 *        uncompressed 128-token window with a per-head sink logit.
 *   HCA  compress every m' = 128 tokens (single stream) and attend densely over all closed
 *        entries plus the same window and sink.
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, contiguous, row-major with
 *     the last dimension fastest, and 16-byte aligned.  "bf16" is IEEE bfloat16, "e4m3" is OCP
 *     FP8 E4M3.  Host pointers appear only where a comment says HOST.
 *   - The library allocates no memory and keeps no global mutable state: it is re-entrant and
 *     thread-safe.  Scratch memory is a caller-supplied workspace whose size the matching
 *     *_workspace() query returns.  Two documented exceptions: the launch counter read by
 *     csa_launch_count (instrumentation), and the fixed scratch array of
 *     csa_index_topk_noalloc.
 *   - Every call only enqueues kernels on `stream` and returns; nothing synchronises.
 *   - Invalid or unsupported descriptors are rejected before any launch.  A failed launch
 *     returns CSA_ERR_CUDA.  Device-detected problems (an index out of range, a bounded wait
 *     that gave up) never trap: the kernel skips the access or returns, and records the first
 *     problem in the status word at the start of the workspace, which csa_read_device_status()
 *     returns.  The status word is sticky: calls never reset it, so it holds the first problem
 *     since it was last cleared (csa_clear_device_status).  A workspace must start with its
 *     first 8 bytes zero (clear it once, or allocate it zero-filled).  Keeping the reset out of
 *     the calls keeps a step's kernels back to back on the stream.
 *   - Positions are explicit: q_pos[b][i] is the 0-based token index t of query i of sequence
 *     b.  For decode, t is the index of the new token (the context length).
 */
#ifndef CSA_B300_H
#define CSA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* csa_stream_t;

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  CSA_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
  CSA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than *_workspace() */
  CSA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  CSA_ERR_DEVICE_CHECK = 5,  /* a kernel found an out-of-range index (see status word) */
  CSA_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up (see status word) */
} csa_status;

/* Storage formats of compressed entries and indexer keys. */
typedef enum {
  CSA_FMT_BF16 = 0,
  /* Mixed-precision cache row (the pages: RoPE dims stay BF16, the rest FP8), d = 512 only:
   * 608 bytes = [0,448) e4m3 codes of dims 0..447 | [448,576) bf16 dims 448..511 |
   * [576,604) seven fp32 scales, one per 64-dim block of the e4m3 part | [604,608) padding.
   * value = code * scale. */
  CSA_FMT_FP8_MIXED = 1,
  /* Indexer keys: e4m3 codes [.., dI] plus one fp32 scale per row; value = code * scale. */
  CSA_FMT_FP8_ROWSCALE = 2,
  /* Low-precision indexer (the pages' FP4/FP8 indexer, "DeepSeek-V4 技术报告深度解读" 5.4): keys
   * as CSA_FMT_FP8_ROWSCALE, and the query is quantised too, per (query, head) row of head_dim
   * 128: scale = amax/448 in fp32 (1 for an all-zero row), codes = e4m3 round-to-nearest-even,
   * saturating, of q/scale computed in fp32.  The contraction runs on the FP8 tensor cores; the
   * scores are those of the dequantised query against the dequantised keys (fp32 sums), so they
   * differ from CSA_FMT_FP8_ROWSCALE's by the query quantisation only.  head_dim must be 128. */
  CSA_FMT_FP8_ROWSCALE_LOWP = 3
} csa_format;

#define CSA_FP8_MIXED_ROW_BYTES 608

/* ---------------------------------------------------------------------------------------------
 * csa_compress -- token-level compressor (CSA overlapped or HCA single-stream).
 *
 * Source: "DeepSeek V4 模型技术大全", CSA path, the Softmax_row and C^Comp equations (overlapped
 * 2m rows with biases B^a, B^b), and the HCA path, its S / C^Comp equations (m' rows, bias B);
 * component table rows "query / KV RMSNorm" and "partial RoPE" (RMSNorm eps 1e-6, RoPE on the
 * last 64 dims, compressed-branch base 160000).
 *
 * For entry i in [0, N), N = floor(T/m), channel c:
 *   rows  = a-stream rows m*i .. m*i+m-1 with logits Za + bias_a[row - m*i]
 *           plus, when overlap and i >= 1, b-stream rows m*(i-1) .. m*i-1 with Zb + bias_b[..]
 *   out_i = sum_rows softmax_rows(logit)[c] * C[row][c]
 * then, if flags has CSA_COMPRESS_NORM: out_i = out_i / sqrt(mean(out_i^2) + eps) * gamma,
 * and if CSA_COMPRESS_ROPE: dims [d-r, d) rotated on adjacent pairs (2j, 2j+1) by angle
 * (m*i + pos_shift) * inv_freq_j.
 *
 * Ca, Za: bf16 [B, T, d].  Cb, Zb: bf16 [B, T, d] when overlap = 1, else ignored (may be NULL).
 * bias_a, bias_b: fp32 [m, d] or NULL (zero).  gamma: fp32 [d] or NULL (one).
 * out: bf16 [B, N, d].
 * Supported: d a power of two in [64, 1024]; 1 <= m <= 256; rope_dims even and <= d;
 * out_fmt CSA_FMT_BF16.
 * ------------------------------------------------------------------------------------------- */
enum { CSA_COMPRESS_NORM = 1u, CSA_COMPRESS_ROPE = 2u };

typedef struct {
  int B, T, d, m;
  int overlap;             /* 1: CSA (Cb, Zb used, block i-1 overlaps); 0: HCA single stream */
  int rope_dims;           /* r; 0 = no rotation */
  float rope_theta;        /* base used when inv_freq is NULL (160000 on the compressed branch) */
  const float* inv_freq;   /* HOST pointer to r/2 finite values (e.g. a YaRN table) or
                              NULL: inv_freq_j = theta^(-2j/r); a non-finite value is
                              CSA_ERR_INVALID_ARG */
  int pos_shift;           /* entry i sits at position m*i + pos_shift */
  float eps;               /* RMSNorm epsilon (1e-6) */
  unsigned flags;          /* CSA_COMPRESS_NORM | CSA_COMPRESS_ROPE */
  csa_format out_fmt;      /* CSA_FMT_BF16 */
} csa_compress_desc;

csa_status csa_compress(const csa_compress_desc* desc, const void* Ca, const void* Cb,
                        const void* Za, const void* Zb, const float* bias_a, const float* bias_b,
                        const float* gamma, void* out, csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * csa_index_topk -- lightning-indexer scores and per-query top-k selection.
 *
 * Source: "DeepSeek V4 模型技术大全", CSA path, the I_{t,s} and TopK equations:
 *   I_{t,s} = sum_h w_{t,h} * ReLU(q^I_{t,h} . K^I_s)  for s < floor((t+1)/m)
 *   idx_t   = TopK_k { I_{t,s} }
 * Ties go to the smaller s.  When fewer than k entries are visible, all are returned and the
 * row is padded with -1.  Output order inside a row: the selected entries in increasing s,
 * then the -1 padding.  The result depends only on the query's own inputs (batch-invariant)
 * and is deterministic.
 *
 * qI: bf16 [B, Tq, n_heads, head_dim].  w: fp32 [B, Tq, n_heads].
 * kI: bf16 [B, N, head_dim] (key_fmt CSA_FMT_BF16) or e4m3 [B, N, head_dim] with
 *     kI_scale fp32 [B, N] (CSA_FMT_FP8_ROWSCALE, CSA_FMT_FP8_ROWSCALE_LOWP).
 * q_pos: int32 [B, Tq].  idx_out: int32 [B, Tq, k].
 * score_out: fp32 [B, Tq, N] or NULL; when given, visible scores are written there and
 *     invisible ones are -inf.
 * workspace: device buffer of at least csa_index_topk_workspace(desc) bytes.
 * Supported: head_dim 64 or 128; 1 <= n_heads <= 64; 1 <= k <= 2048; N <= 262144
 * (larger N returns CSA_ERR_UNSUPPORTED).
 *
 * score_fmt CSA_SCORE_BF16 ("DeepSeek-V4 技术报告深度解读" 5.4 and the indexer QK-path table row
 * of "DeepSeek V4 模型技术大全": index scores in BF16 instead of FP32, for a faster top-k
 * selector): every score is rounded to bf16 (round to nearest even) after the head sum and the
 * FP8 row scale; the stored values (score_out, workspace rows) are those rounded values in fp32,
 * and the top-k selects on them with the same rule (ties, which rounding makes frequent, go to
 * the smaller s).  CSA_SCORE_FP32 (0, the default of a zeroed descriptor) keeps fp32 scores.
 *
 * select_mode: where the top-k selection runs (the result is the same bit for bit):
 *   CSA_SELECT_AUTO (0, the default): fused into the score kernel when the call qualifies (below)
 *     and its rows are long, N >= 16 k (there it is faster: 65536-token prefill, N = 16384,
 *     k = 512: 7.8 ms against 9.1 ms for the stored path); the stored path otherwise.
 *   CSA_SELECT_FUSED: fused whenever the call qualifies.
 *   CSA_SELECT_STORED: score rows stored in the workspace (in chunks of at most 256 MiB) and
 *     selected by the top-k kernels.
 * The fused selection keeps, per query, the entries that can still be among its top k (above a
 * running lower bound of the k-th score) and selects from those; the score rows are never
 * stored.  It qualifies when score_out is NULL, groups of 4 queries x 64 indexer heads fill the
 * tensor-core tile (n_heads in 33..64, Tq >= 4), the keys are bf16 or the low-precision indexer's,
 * N <= 32768, and the batch holds at least 4 groups per SM of the device.
 * ------------------------------------------------------------------------------------------- */
enum { CSA_SCORE_FP32 = 0, CSA_SCORE_BF16 = 1 };
enum { CSA_SELECT_AUTO = 0, CSA_SELECT_FUSED = 1, CSA_SELECT_STORED = 2 };

typedef struct {
  int B, Tq, N, n_heads, head_dim, k, m;
  csa_format key_fmt;      /* CSA_FMT_BF16, CSA_FMT_FP8_ROWSCALE or CSA_FMT_FP8_ROWSCALE_LOWP */
  int score_fmt;           /* CSA_SCORE_FP32 (0) or CSA_SCORE_BF16 */
  int select_mode;         /* CSA_SELECT_AUTO (0), CSA_SELECT_FUSED or CSA_SELECT_STORED */
} csa_index_desc;

size_t csa_index_topk_workspace(const csa_index_desc* desc);

csa_status csa_index_topk(const csa_index_desc* desc, const void* qI, const float* w,
                          const void* kI, const float* kI_scale, const int32_t* q_pos,
                          int32_t* idx_out, float* score_out, void* workspace, size_t ws_bytes,
                          csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * csa_index_score / csa_topk -- the two halves of csa_index_topk as separate calls.
 *
 * Same sources and conventions as csa_index_topk.  csa_index_score writes the visible scores
 * I_{t,s}, s < floor((t+1)/m), into score_out fp32 [B, Tq, N] and leaves the rest of each row
 * untouched; its workspace needs only the status header (csa_index_score_workspace).
 * csa_topk reads scores fp32
 * [B, Tq, N] (only the entries s < floor((t+1)/m) of each row, so the others may hold anything)
 * and writes idx_out exactly as csa_index_topk would for those scores; workspace:
 * csa_topk_workspace(desc) bytes.  csa_index_score followed by csa_topk on the same stream gives
 * the same idx_out as csa_index_topk, bit for bit.  Both reject what csa_index_topk rejects;
 * csa_topk ignores qI / head settings of the descriptor except for validation.
 * ------------------------------------------------------------------------------------------- */
size_t csa_index_score_workspace(const csa_index_desc* desc);

csa_status csa_index_score(const csa_index_desc* desc, const void* qI, const float* w,
                           const void* kI, const float* kI_scale, const int32_t* q_pos,
                           float* score_out, void* workspace, size_t ws_bytes, csa_stream_t stream);

size_t csa_topk_workspace(const csa_index_desc* desc);

csa_status csa_topk(const csa_index_desc* desc, const float* scores, const int32_t* q_pos,
                    int32_t* idx_out, void* workspace, size_t ws_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * csa_index_topk_noalloc -- csa_index_topk for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a library convenience.  Some callers cannot call
 * cudaMalloc when they need a selection, e.g. code running inside a host callback or an
 * allocator hook, or a plug-in whose host hands it only input and output buffers.  This call
 * computes exactly what csa_index_topk computes (same arguments, same results, bit for bit) but
 * takes no workspace: its scratch is one fixed array of CSA_NOALLOC_SCRATCH_BYTES in device
 * memory, declared by the library, which every GPU that loads the library keeps until the
 * process exits.  The call allocates nothing and frees nothing.
 *
 * Limits and behaviour:
 *   - Requests whose csa_index_topk_workspace() exceeds CSA_NOALLOC_SCRATCH_BYTES return
 *     CSA_ERR_UNSUPPORTED before any CUDA call (decode at N = 262144 fits up to B = 7; a
 *     prefill chunk fits while Tq * N * 4 bytes, rounded up to 4-query groups, stays under it).
 *   - The first call in a CUDA context looks up the array's device address
 *     (cudaGetSymbolAddress, with the calling thread's current device and context) and caches
 *     it under the context's unique ID (cuCtxGetId); make that first call before any stream
 *     capture.  A caller's own context, or the primary context created again after
 *     cudaDeviceReset, gets a lookup of its own.
 *   - Every call on a device shares the one array and it keeps the last call's contents: calls
 *     that may overlap on the GPU (other streams, other threads) race and must be serialised by
 *     the caller.  Each call zeroes the array's status word on `stream` (an 8-byte
 *     cudaMemsetAsync) before its kernels.  The caller cannot read that word, so this call
 *     cannot report device-detected problems (an index out of range, a bounded wait that gave
 *     up); a caller that needs them uses csa_index_topk with its own workspace.
 * Errors are otherwise those of csa_index_topk.
 * ------------------------------------------------------------------------------------------- */
#define CSA_NOALLOC_SCRATCH_BYTES (8u << 20)

csa_status csa_index_topk_noalloc(const csa_index_desc* desc, const void* qI, const float* w,
                                  const void* kI, const float* kI_scale, const int32_t* q_pos,
                                  int32_t* idx_out, float* score_out, csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * csa_attend / hca_attend -- shared K=V multi-query attention with SWA window and sink.
 *
 * Source: "DeepSeek V4 模型技术大全", component table rows "Shared K=V MQA", "query / KV RMSNorm",
 * "partial RoPE", "attention sink" (p = exp(z) / (exp(a_h) + sum exp(z))), "SWA"
 * (W_t = {t-127 .. t}), the HCA visibility set j < floor((t+1)/m'), and the implementation
 * note that the core-attention output gets a reverse rotation.
 *
 * Per query (b, i) at position t = q_pos[b][i], per head h:
 *   q_hat = RoPE_t(RMSNorm(q[b,i,h]))               (if CSA_ATTEND_Q_NORM_ROPE; unit weight)
 *   keys  = csa_attend: entries idx[b,i,0..k-1] (entries equal to -1 are skipped)
 *           hca_attend: every entry j < min(N, floor((t+1)/m))
 *           plus window rows win[b, u mod Wcap] for u in [max(0, t-window+1), t]
 *   z_j   = scale * q_hat . key_j
 *   out   = sum_j exp(z_j) key_j / (exp(sink[h]) + sum_j exp(z_j))
 *   out[d-r:] rotated by -t                          (if CSA_ATTEND_OUT_UNROTATE)
 *   lse   = log(exp(sink[h]) + sum_j exp(z_j))       (if CSA_ATTEND_WRITE_LSE)
 *
 * q: bf16 [B, Tq, H, d].  kv: bf16 [B, N, d] or FP8_MIXED rows [B, N, 608 bytes].
 * idx: int32 [B, Tq, k] (csa_attend only).  win: bf16 [B, Wcap, d]; the caller keeps every
 * window position of every query of the call in a distinct live slot (decode: a 128-slot ring;
 * prefill from position 0: Wcap >= T).  sink: fp32 [H].  q_pos: int32 [B, Tq].
 * out: bf16 [B, Tq, H, d].  lse: fp32 [B, Tq, H] or NULL.
 * An idx entry outside [-1, N) is skipped and reported through the status word.
 * Supported: d in {128, 512}; H % 16 == 0 and <= 128; kv_fmt FP8_MIXED needs d = 512;
 * rope_dims even, <= d; window <= Wcap.
 * ------------------------------------------------------------------------------------------- */
enum { CSA_ATTEND_Q_NORM_ROPE = 1u, CSA_ATTEND_OUT_UNROTATE = 2u, CSA_ATTEND_WRITE_LSE = 4u };

typedef struct {
  int B, Tq, N, H, d;
  int rope_dims;
  int k;                   /* csa_attend: columns of idx; ignored by hca_attend */
  int m;                   /* compression ratio (hca_attend visibility; csa_attend ignores it) */
  int Wcap, window;        /* ring capacity and window length (128) */
  float scale;             /* 0 => 1/sqrt(d) */
  float rope_theta;        /* base used when inv_freq is NULL */
  const float* inv_freq;   /* HOST pointer to rope_dims/2 finite values or NULL */
  float eps;               /* RMSNorm epsilon for q */
  csa_format kv_fmt;       /* CSA_FMT_BF16 or CSA_FMT_FP8_MIXED */
  unsigned flags;          /* CSA_ATTEND_* */
} csa_attend_desc;

/* Workspace bytes for csa_attend / hca_attend with this descriptor (0 if it is invalid).  The two
 * differ: a dense HCA query visits up to N + window rows, a CSA query k + window. */
size_t csa_attend_workspace(const csa_attend_desc* desc);
size_t hca_attend_workspace(const csa_attend_desc* desc);

csa_status csa_attend(const csa_attend_desc* desc, const void* q, const void* kv,
                      const int32_t* idx, const void* win, const float* sink,
                      const int32_t* q_pos, void* out, float* lse, void* workspace,
                      size_t ws_bytes, csa_stream_t stream);

csa_status hca_attend(const csa_attend_desc* desc, const void* q, const void* kv,
                      const void* win, const float* sink, const int32_t* q_pos, void* out,
                      float* lse, void* workspace, size_t ws_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * csa_cache_append -- hybrid KV cache maintenance for one attention layer of B sequences.
 *
 * Source: "DeepSeek V4 模型技术大全", the hybrid KV cache passage (C_state = the SWA window's last
 * n_win rows and the compressors' unclosed tails; C_classical = the closed CSA entries, indexer
 * keys and HCA entries; prefix reuse at lcm(4, 128) = 128-token boundaries, the tail recomputed)
 * and the CSA / HCA compressor equations quoted for csa_compress.
 *
 * Appends tokens t0 .. t0+n-1 (n = 1 is one decode step; t0 = 0 with the whole prompt fills the
 * cache after prefill).  Tokens 0 .. t0-1 must have been appended before with the same buffers.
 *   - Every entry i whose block closes inside the chunk, i.e. m*(i+1)-1 in [t0, t0+n), is
 *     compressed exactly as csa_compress would compute entry i of the whole sequence (same
 *     arithmetic, RoPE position m*i) and written to kv[b, i] (and the indexer key to kI[b, i]).
 *     Rows of blocks that began before t0 come from the tail rings in `state`.
 *   - Window row of token u goes to win[b, u mod Wcap] for u in [max(t0, t0+n-Wcap), t0+n).
 *   - The tail rings keep the last R stream rows (R = 2m with overlap, else m).
 * Entries compress in a first kernel; the rings and the window are written in a second one
 * ordered after it on `stream`, so a chunk may overwrite the slots it reads.
 *
 * CSA layer: overlap = 1, m = 4, rows Ca, Cb, Za, Zb (and the indexer streams when dI > 0).
 * HCA layer: overlap = 0, m = 128, rows Ca (the C stream) and Za (its gate logits Z).
 * rows->*: bf16 [B, n, d] (the *_I streams [B, n, dI]); rows->win: bf16 [B, n, d], the tokens'
 *     window rows as csa_attend reads them.
 * params->*: as csa_compress's bias_a, bias_b ([m, width] fp32) and gamma ([width] fp32); NULL
 *     = zero biases / unit gamma.
 * bufs->kv: bf16 [B, N_cap, d]; bufs->kI: bf16 [B, N_cap, dI] (dI > 0); bufs->win: bf16
 *     [B, Wcap, d]; bufs->state: csa_cache_state_bytes(desc) bytes, zero or as left by the
 *     previous append (opaque; a copy of it and of win taken at token t restores the cache to t).
 * Requires (t0+n)/m <= N_cap, t0 + n < 2^31.  Widths as csa_compress (d, dI powers of two in
 * [64, 1024]).  Invalid arguments return CSA_ERR_INVALID_ARG / CSA_ERR_UNSUPPORTED before any
 * launch; n = 0 or B = 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
  int B;                   /* sequences that advance together */
  int d;                   /* entry and window row width */
  int dI;                  /* indexer key width; 0 = no indexer stream (HCA layers) */
  int m;                   /* compression ratio */
  int overlap;             /* 1: CSA (two streams, block i-1 overlaps); 0: HCA */
  int Wcap;                /* window ring slots */
  int N_cap;               /* entries the kv / kI buffers hold per sequence */
  int rope_dims;           /* RoPE on the main entries, as csa_compress */
  float rope_theta;
  const float* inv_freq;   /* HOST pointer to rope_dims/2 finite values or NULL */
  float eps;
  unsigned flags;          /* CSA_COMPRESS_* for the main entries */
  unsigned index_flags;    /* CSA_COMPRESS_* for the indexer keys (rotation not supported) */
} csa_cache_desc;

typedef struct {
  const void *Ca, *Cb, *Za, *Zb;
  const void *Ca_I, *Cb_I, *Za_I, *Zb_I;
  const void* win;
} csa_cache_rows;

typedef struct {
  const float *bias_a, *bias_b, *gamma;
  const float *bias_a_I, *bias_b_I, *gamma_I;
} csa_cache_params;

typedef struct {
  void* kv;
  void* kI;
  void* win;
  void* state;
} csa_cache_buffers;

/* Bytes of the opaque tail state for this descriptor (0 if it is invalid). */
size_t csa_cache_state_bytes(const csa_cache_desc* desc);

csa_status csa_cache_append(const csa_cache_desc* desc, int64_t t0, int n, const csa_cache_rows* rows,
                            const csa_cache_params* params, const csa_cache_buffers* bufs,
                            csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * csa_out_proj -- grouped output projection of the attention output.
 *
 * Source: "DeepSeek V4 模型技术大全", the grouped output projection equations of the CSA path and
 * its component-table row (Flash: n_h = 64, d_h = 512, g = 8, r_o = 1024, hidden size 4096):
 *   O = Concat(o^(1) .. o^(n_h)) split into g groups O^[u] of n_h/g consecutive heads,
 *   z^[u] = O^[u] W_down^[u]   (W_down^[u] of (n_h/g) d_h x r_o),
 *   y = Proj(Concat_u z^[u])   (Proj: a linear map g r_o -> d_out).
 * Products accumulate in fp32 on the tensor cores; z is stored in bf16 and y is computed from
 * that bf16 z.
 *
 * O: bf16 [T, n_heads, head_dim] (the attention output, T = B x Tq).
 * W_down: bf16 [groups, rank, K], K = (n_heads/groups) x head_dim: row n of group u holds
 *     column n of W_down^[u] (the matrix stored transposed, K contiguous).
 * W_proj: bf16 [d_out, groups x rank] (Proj's matrix stored the same way); unused if d_out = 0.
 * z: bf16 [T, groups x rank] output.  y: bf16 [T, d_out] output (d_out > 0).
 * workspace: at least csa_out_proj_workspace(desc) bytes (the status word), first 8 bytes zero.
 * Supported: groups divides n_heads; K, rank and d_out multiples of 64; T < 2^31.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
  int T;                   /* tokens */
  int n_heads, head_dim;
  int groups;              /* g */
  int rank;                /* r_o */
  int d_out;               /* width of y; 0 = compute z only */
} csa_out_proj_desc;

size_t csa_out_proj_workspace(const csa_out_proj_desc* desc);

csa_status csa_out_proj(const csa_out_proj_desc* desc, const void* O, const void* W_down, const void* W_proj,
                        void* z, void* y, void* workspace, size_t ws_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Status helpers.
 * csa_read_device_status: waits for `stream`, reads the status word at the start of a
 * workspace that a previous call used, returns CSA_OK, CSA_ERR_DEVICE_CHECK (a range check
 * failed) or CSA_ERR_TIMEOUT (a bounded device-side wait gave up), and (if
 * detail != NULL, HOST pointer) stores the first offending value.  csa_clear_device_status
 * enqueues a reset of that word.  csa_status_string never returns NULL.
 * ------------------------------------------------------------------------------------------- */
csa_status csa_read_device_status(const void* workspace, csa_stream_t stream, int32_t* detail);
csa_status csa_clear_device_status(void* workspace, csa_stream_t stream);
const char* csa_status_string(csa_status status);

/* Number of kernel launches the library has enqueued in this process (all calls, all threads;
 * an atomic counter kept for instrumentation, not part of any result). */
uint64_t csa_launch_count(void);

/* ---------------------------------------------------------------------------------------------
 * csa_selftest_bounded_wait -- exercises the library's failure path on purpose.
 *
 * No counterpart in the pages: a diagnostic of the library itself.  Every wait inside the
 * library's kernels is bounded; a wait that is never satisfied gives up after its limit, writes
 * CSA_ERR_TIMEOUT to the workspace status word and the kernel returns, leaving the CUDA context
 * usable.  This call launches one small kernel whose wait nothing can complete (an mbarrier no
 * thread arrives on), with the given limit, so a caller can check that path end to end:
 * afterwards csa_read_device_status returns CSA_ERR_TIMEOUT and the detail holds the time the
 * wait took, in microseconds.
 * workspace: at least 256 bytes, 16-byte aligned (its status word is the only thing written).
 * limit_ns: 1000 .. 2000000000.  Returns CSA_ERR_INVALID_ARG / CSA_ERR_WORKSPACE for bad
 * arguments, CSA_ERR_CUDA if the launch fails, else CSA_OK (the timeout itself is reported
 * through the status word).
 * ------------------------------------------------------------------------------------------- */
csa_status csa_selftest_bounded_wait(void* workspace, size_t ws_bytes, int64_t limit_ns, csa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA_B300_H */
