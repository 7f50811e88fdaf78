// Shared K=V multi-query attention on the 5th-generation tensor cores, for 512-dim bf16 rows and
// 64 query heads per CTA ("DeepSeek V4 模型技术大全", component table rows Shared K=V MQA,
// query/KV RMSNorm, partial RoPE, attention sink, SWA; the HCA visibility set; the
// reverse-rotation note).  Same slots, splits and partial format as the warp-MMA kernel in
// attend.cu, which keeps the other shapes (d = 128, the FP8 cache).
//
// Per CTA: one query, 64 heads, one split of the slot range, 64 rows per chunk, warp-specialised
// so that the gather of chunk c+2, the products of chunks c and c+1 and the softmax of chunk c
// overlap:
//   loader warps (2)      row pointers from the idx row, cp.async of the chunk's rows straight into
//                         the 128-byte swizzled operand layout (two chunk buffers)
//   MMA warp (1 thread)   S^T(c) = K q_hat^T   M = 128 (the chunk's 64 rows are TMEM lanes 0..63),
//                                              N = 64 heads, K = 512, fp32 in TMEM (two buffers)
//                         O^T += V^T P^T(c)    M = 128 dims (4 tiles), N = 64 heads, K = 64 rows;
//                                              V^T is the chunk's rows through an MN-major descriptor
//   softmax warps (4)     one thread per (row, 32 heads): per-head chunk maximum by a warp
//                         butterfly; a per-head reference maximum that moves only when a chunk
//                         exceeds it by more than 2^8; p = exp2(z - ref) rounded to bf16 into P^T
//                         (K-major, 128-byte swizzle); per-thread running sums of the rounded p
//   correction warps (4)  the query block (RMSNorm, RoPE) before the loop; rescale of O^T in TMEM
//                         when a reference moved; the epilogue (sink, normaliser, reverse
//                         rotation, output or split partials)
// Every wait is bounded (CSA_ERR_TIMEOUT in the status word, never a hang).
#include "common.cuh"
#include "tc.cuh"

namespace csa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int D = 512;
constexpr int HG = 64;                        // heads per CTA (MMA N)
constexpr int CK = 64;                        // rows per chunk
constexpr int NREG = D / 64;                  // 128-byte column regions of a row
constexpr float kRescaleLog2 = 8.f;           // a head's reference maximum moves only past 2^8
constexpr uint64_t kWaitNs = 200000000ull;    // 0.2 s: every wait here normally ends in microseconds

// warp roles
constexpr int NT = 11 * 32;
constexpr int kLoad0 = 6, kNLoad = 2;         // loader warps 6, 7
constexpr int kMmaWarp = 10;
// softmax warps 4, 5 (heads 0..31) and 8, 9 (heads 32..63): TMEM lane quarters 0 and 1 = rows 0..63
__device__ __forceinline__ bool is_softmax_warp(int w) { return w == 4 || w == 5 || w == 8 || w == 9; }

constexpr int Q_REGION = HG * 128;            // 64 heads x 64 dims (bf16)
constexpr int KV_REGION = 2 * CK * 128;       // two buffers x 64 rows x 64 dims
constexpr int PT_BYTES = HG * 128;            // P^T of one chunk: 64 heads x 64 rows
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + NREG * Q_REGION;
constexpr int KV_PAD = CK * 128;              // the M = 128 read of buffer 1 runs 64 rows past region 7
constexpr int OFF_PT = OFF_KV + NREG * KV_REGION + KV_PAD;
constexpr int OFF_MISC = OFF_PT + 2 * PT_BYTES;
constexpr int MISC_BYTES = 4096;
constexpr int SMEM = 1024 + OFF_MISC + MISC_BYTES;
constexpr int TMEM_COLS = 512;                // S^T at columns 0 / 64, O^T tiles at 128 + 64 mt
static_assert(SMEM <= 232448, "shared memory budget");

// misc area: byte offsets
constexpr int M_ROWPTR = 0;                   // [2][CK] row pointers (8 B)
constexpr int M_ROPE = 1024;                  // [kMaxRopePairs] float2
constexpr int M_REF = 1536;                   // [HG] reference maximum (log2 domain)
constexpr int M_FAC = M_REF + HG * 4;         // [2][HG] factor of chunk c (buffer c & 1)
constexpr int M_FIN = M_FAC + 2 * HG * 4;     // [HG] epilogue factor
constexpr int M_LSUM = M_FIN + HG * 4;        // [HG]
constexpr int M_RED = M_LSUM + HG * 4;        // [2][HG]
constexpr int M_FLAG = M_RED + 2 * HG * 4;    // [2][2] rescale needed (chunk buffer, head half); [4] skip
constexpr int M_BARS = M_FLAG + 32;           // mbarriers
constexpr int NBARS = 13;
constexpr int M_TMEM = M_BARS + NBARS * 8;
constexpr int M_ABORT = M_TMEM + 4;
static_assert(M_BARS % 8 == 0 && M_ABORT + 4 <= MISC_BYTES, "misc layout");

// Butterfly over 32 values per lane: afterwards v[0] of lane L holds the reduction over the 32
// lanes of value L (max when MAX, else sum).
template <bool MAX>
__device__ __forceinline__ void butterfly32(float* v, int lane) {
#pragma unroll
  for (int o = 16, nc = 32; o >= 1; o >>= 1, nc >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < nc / 2) {
        const float send = up ? v[i] : v[i + nc / 2];
        const float keep = up ? v[i + nc / 2] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
      }
    }
  }
}

__global__ void __launch_bounds__(NT, 1) k_attend_tc(const AttendArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (tc::sptr(smem_raw) & 1023u)) & 1023u);
  unsigned char* qs = sm + OFF_Q;
  unsigned char* kvs = sm + OFF_KV;
  unsigned char* pts = sm + OFF_PT;
  unsigned char* misc = sm + OFF_MISC;
  const unsigned char** rowptr = reinterpret_cast<const unsigned char**>(misc + M_ROWPTR);
  float2* rope = reinterpret_cast<float2*>(misc + M_ROPE);
  float* ref = reinterpret_cast<float*>(misc + M_REF);
  float* facb = reinterpret_cast<float*>(misc + M_FAC);
  float* fin = reinterpret_cast<float*>(misc + M_FIN);
  float* lsum = reinterpret_cast<float*>(misc + M_LSUM);
  float* red = reinterpret_cast<float*>(misc + M_RED);
  int* flag = reinterpret_cast<int*>(misc + M_FLAG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + M_BARS);
  uint64_t* q_ready = bars + 0;       // correction warps wrote q_hat (128 arrivals)
  uint64_t* kv_full = bars + 1;       // [2] a chunk's rows landed (loader threads)
  uint64_t* kv_empty = bars + 3;      // [2] PV of the chunk in that buffer completed (commit)
  uint64_t* s_full = bars + 5;        // [2] S of the chunk in that buffer completed (commit)
  uint64_t* p_full = bars + 7;        // [2] P^T and factors of the chunk written (softmax threads)
  uint64_t* c_done = bars + 9;        // [2] O^T rescaled for the chunk (correction threads)
  uint64_t* sm_done = bars + 11;      // softmax wrote the final sums / factors (softmax threads)
  uint64_t* drain = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + M_ABORT);
  grid_dep_wait();
  grid_dep_launch();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long qi = blockIdx.x;
  const int h0 = blockIdx.y * HG;
  const int split = blockIdx.z;
  const int t = a.q_pos[qi];
  const int b = static_cast<int>(qi / a.Tq);
  const int nvis = n_visible(t, a.m, a.N);
  const int Kq = (a.idx == nullptr) ? nvis : a.k;
  const int nslots = Kq + a.window;
  const int s_begin = split * a.split_slots;
  const int s_end = min(nslots, s_begin + a.split_slots);
  const int nch = s_end > s_begin ? (s_end - s_begin + CK - 1) / CK : 0;
  const float sl2 = a.scale * kLog2e;

  if ((tc::sptr(sm) & 1023u) != 0u) {               // the swizzled operands need 1024-byte alignment
    if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2000);
    return;
  }
  if (tid == 0) {
    // a wait of this call already gave up: later CTAs do no work instead of waiting in turn (the
    // decision is thread 0's, shared through shared memory, so the whole CTA takes it)
    flag[4] = (*reinterpret_cast<volatile int32_t*>(a.status) == CSA_ERR_TIMEOUT) ? 1 : 0;
    tc::mbar_init(q_ready, 128);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&kv_full[i], kNLoad * 32);
      tc::mbar_init(&kv_empty[i], 1);
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], 128);
      tc::mbar_init(&c_done[i], 128);
    }
    tc::mbar_init(sm_done, 128);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid < a.rp.r / 2) {
    float cs, sn;
    rope_cos_sin(static_cast<double>(t), a.rp.inv_freq[tid], cs, sn);
    rope[tid] = make_float2(cs, sn);
  }
  if (tid < HG) {
    ref[tid] = -INFINITY;
    lsum[tid] = 0.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = flag[4] != 0;
  auto fail = [&](int where) {
    *abort_flag = 1;
    report_error(a.status, CSA_ERR_TIMEOUT, where);
  };
  auto wait = [&](uint64_t* bar, int use, int where) {   // the phase of the use-th completion
    const bool ok = tc::mbar_wait(bar, static_cast<uint32_t>(use & 1), abort_flag, kWaitNs);
    if (!ok) fail(where);
    return ok;
  };

  bool issued = false;
  if (!skip && warp >= kLoad0 && warp < kLoad0 + kNLoad) {
    // ------------------------------------------------------------ loader warps
    const int lt = tid - kLoad0 * 32;                    // 0..63: one row each for the pointers
    const unsigned char* kvb = static_cast<const unsigned char*>(a.kv);
    const unsigned char* winb = static_cast<const unsigned char*>(a.win);
    const unsigned char* dummy = static_cast<const unsigned char*>(a.q);   // source of zero-size copies
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      const int s = s_begin + c * CK + lt;
      const int raw = (s < s_end && s < Kq && a.idx != nullptr) ? a.idx[qi * a.k + s] : 0;
      if (c >= 2) wait(&kv_empty[buf], (c - 2) >> 1, 41);   // PV of chunk c-2 has read this buffer
      const unsigned char* p = nullptr;
      if (s < s_end) {
        if (s < Kq) {
          const int e = (a.idx == nullptr) ? s : raw;
          if (e >= 0 && e < a.N) {
            p = kvb + (static_cast<size_t>(b) * a.N + e) * (D * 2);
          } else if (e != -1) {
            report_error(a.status, CSA_ERR_DEVICE_CHECK, e);
          }
        } else {
          const int jw = s - Kq;
          const int u = t - a.window + 1 + jw;
          if (jw < a.window && u >= 0) p = winb + (static_cast<size_t>(b) * a.Wcap + u % a.Wcap) * (D * 2);
        }
      }
      rowptr[buf * CK + lt] = p;
      tc::named_bar_sync(2, kNLoad * 32);
#pragma unroll 4
      for (int i = lt; i < CK * 64; i += kNLoad * 32) {
        const int j = i >> 6, cc = i & 63;
        const unsigned char* rp = rowptr[buf * CK + j];
        const int row = buf * CK + j;
        unsigned char* dst = kvs + (cc >> 3) * KV_REGION + row * 128 + (((cc & 7) ^ (row & 7)) << 4);
        cp_async16(dst, rp ? rp + cc * 16 : dummy, rp != nullptr);
      }
      cp_async_commit();
      cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&kv_full[buf]);
    }
  } else if (!skip && warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (lane 0 only)
    if (lane == 0) {
      constexpr uint32_t idS = tc::umma_idesc_bf16(128, HG, 0, 0);
      constexpr uint32_t idPV = tc::umma_idesc_bf16(128, HG, 1, 0);
      const uint32_t kva = tc::sptr(kvs), qa = tc::sptr(qs), pa = tc::sptr(pts);
      auto issue_s = [&](int c) {
        const int buf = c & 1;
#pragma unroll 8
        for (int k = 0; k < D / 16; ++k) {
          const int r = k >> 2, off = (k & 3) * 32;
          const uint64_t ad = tc::umma_desc_sw128(kva + r * KV_REGION + buf * CK * 128 + off);
          const uint64_t bd = tc::umma_desc_sw128(qa + r * Q_REGION + off);
          tc::umma_bf16(tmem + buf * HG, ad, bd, idS, k > 0 ? 1u : 0u);
        }
        tc::umma_commit(&s_full[buf]);
        issued = true;
      };
      bool ok = nch == 0 || (wait(q_ready, 0, 42) && wait(&kv_full[0], 0, 43));
      if (ok && nch > 0) {
        tc::tc_fence_after();
        issue_s(0);
      }
      for (int c = 0; ok && c < nch; ++c) {
        const int buf = c & 1;
        if (c + 1 < nch) {
          if (!wait(&kv_full[(c + 1) & 1], (c + 1) >> 1, 44)) break;
          tc::tc_fence_after();
          issue_s(c + 1);
        }
        if (!wait(&p_full[buf], c >> 1, 45) || !wait(&c_done[buf], c >> 1, 46)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int k = 0; k < CK / 16; ++k) {
            const uint64_t ad = tc::umma_desc_sw128_mn(kva + (2 * mt) * KV_REGION + (buf * CK + 16 * k) * 128,
                                                       KV_REGION, 1024);
            const uint64_t bd = tc::umma_desc_sw128(pa + buf * PT_BYTES + k * 32);
            tc::umma_bf16(tmem + 2 * HG + mt * HG, ad, bd, idPV, (c > 0 || k > 0) ? 1u : 0u);
          }
        }
        tc::umma_commit(&kv_empty[buf]);
      }
      if (issued) {                                      // all MMAs done before TMEM is released
        tc::umma_commit(drain);
        if (!tc::mbar_wait(drain, 0, nullptr, kWaitNs)) report_error(a.status, CSA_ERR_TIMEOUT, 47);
      }
    }
    __syncwarp();
  } else if (!skip && is_softmax_warp(warp)) {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;                        // 0 or 1: rows 32*quarter + lane
    const int hh = warp >= 8 ? 1 : 0;                    // heads 32*hh + i
    const int j = quarter * 32 + lane;
    float ps[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) ps[i] = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      wait(&s_full[buf], c >> 1, 48);
      wait(&kv_full[buf], c >> 1, 53);                  // the loaders' row pointers of chunk c
      tc::tc_fence_after();
      float z[32];
      tc::tmem_ld32_wait(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * HG + hh * 32, z);
      const bool valid = rowptr[buf * CK + j] != nullptr;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        z[i] = valid ? z[i] * sl2 : -INFINITY;
        v[i] = z[i];
      }
      butterfly32<true>(v, lane);
      red[quarter * HG + hh * 32 + lane] = v[0];
      tc::named_bar_sync(1, 128);
      if (quarter == 0) {                                // one thread per head updates its reference
        const int h = hh * 32 + lane;
        const float cm = fmaxf(red[h], red[HG + h]);
        const float rold = ref[h];
        float f = 1.f;
        bool need = false;
        if (cm > rold + kRescaleLog2 || (rold == -INFINITY && cm > -INFINITY)) {
          f = (rold == -INFINITY) ? 0.f : exp2f(rold - cm);
          need = c > 0 && rold > -INFINITY;              // O^T holds terms scaled by rold
          ref[h] = cm;
        }
        facb[buf * HG + h] = f;
        const bool any = __any_sync(0xffffffffu, need);
        if (lane == 0) flag[buf * 2 + hh] = any ? 1 : 0;
      }
      tc::named_bar_sync(1, 128);
      // p = exp2(z - ref) rounded to bf16 into P^T[h][j]; running sums of the rounded values
      unsigned char* pt = pts + buf * PT_BYTES;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int h = hh * 32 + i;
        const float r = ref[h];
        const float p = exp2f(z[i] - (r == -INFINITY ? 0.f : r));
        const __nv_bfloat16 pb = __float2bfloat16_rn(p);
        ps[i] = fmaf(ps[i], facb[buf * HG + h], __bfloat162float(pb));
        *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + (((j >> 3) ^ (h & 7)) << 4) + (j & 7) * 2) = pb;
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&p_full[buf]);
    }
    // final sums over the 64 rows-threads of each head, then the epilogue factors
    butterfly32<false>(ps, lane);
    red[quarter * HG + hh * 32 + lane] = ps[0];
    tc::named_bar_sync(1, 128);
    if (quarter == 0) {
      const int h = hh * 32 + lane;
      const float ls = red[h] + red[HG + h];
      const float r = ref[h];
      const int hg = h0 + h;
      if (a.n_splits == 1) {
        const float a2 = a.sink[hg] * kLog2e;
        const float M = fmaxf(r, a2);
        const float f = (r == -INFINITY) ? 0.f : exp2f(r - M);
        const float L = ls * f + exp2f(a2 - M);
        fin[h] = f / L;
        if (a.lse != nullptr) a.lse[qi * a.H + hg] = (M + log2f(L)) * kLn2;
      } else {
        const int Q = a.B * a.Tq;
        float* pml = a.partial + static_cast<size_t>(Q) * a.n_splits * a.H * D;
        const size_t rowi = (static_cast<size_t>(qi) * a.n_splits + split) * a.H + hg;
        pml[rowi * 2 + 0] = r;
        pml[rowi * 2 + 1] = ls;
      }
    }
    tc::mbar_arrive(sm_done);
  } else if (!skip && warp < 4) {
    // ------------------------------------------------------------ correction warps (lane quarter = warp)
    {
      // q_hat = RoPE_t(RMSNorm(q)) as bf16 into the K-major swizzled B operand of S: warp w prepares
      // heads 16w..16w+15; lane L owns dims 16L..16L+15 (two 16-byte chunks of region L/4)
      const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(a.q);
      const int region = lane >> 2, ch0 = (lane & 3) * 2;
#pragma unroll 2
      for (int i = 0; i < HG / 4; ++i) {
        const int hl = warp * (HG / 4) + i;
        const uint4* src =
            reinterpret_cast<const uint4*>(qsrc + ((qi * a.H) + h0 + hl) * static_cast<long long>(D) + lane * 16);
        const uint4 u0 = src[0], u1 = src[1];
        float v[16] = {bf16lo(u0.x), bf16hi(u0.x), bf16lo(u0.y), bf16hi(u0.y), bf16lo(u0.z), bf16hi(u0.z),
                       bf16lo(u0.w), bf16hi(u0.w), bf16lo(u1.x), bf16hi(u1.x), bf16lo(u1.y), bf16hi(u1.y),
                       bf16lo(u1.z), bf16hi(u1.z), bf16lo(u1.w), bf16hi(u1.w)};
        if (a.q_norm_rope) {
          float ss = 0.f;
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) ss = fmaf(v[cc], v[cc], ss);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + a.eps);
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) v[cc] *= inv;
#pragma unroll
          for (int cc = 0; cc < 16; cc += 2) {
            const int ch = lane * 16 + cc;
            if (ch >= D - a.rp.r) {
              const float2 cssn = rope[(ch - (D - a.rp.r)) >> 1];
              const float x0 = v[cc], x1 = v[cc + 1];
              v[cc] = x0 * cssn.x - x1 * cssn.y;
              v[cc + 1] = x0 * cssn.y + x1 * cssn.x;
            }
          }
        }
        unsigned char* row = qs + region * Q_REGION + hl * 128;
        *reinterpret_cast<uint4*>(row + ((ch0 ^ (hl & 7)) << 4)) = make_uint4(
            pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        *reinterpret_cast<uint4*>(row + (((ch0 + 1) ^ (hl & 7)) << 4)) =
            make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                       pack_bf16x2(v[14], v[15]));
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(q_ready);
    }
    const int quarter = warp;
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      wait(&p_full[buf], c >> 1, 49);
      if (flag[buf * 2] | flag[buf * 2 + 1]) {
        // a reference moved: O^T (lanes of this quarter, all heads) times the chunk's factors, once
        // the PV of chunk c-1 has landed
        wait(&kv_empty[(c - 1) & 1], (c - 1) >> 1, 50);
        tc::tc_fence_after();
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
          const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 2 * HG + mt * HG;
          float o[64];
          tc::tmem_ld64_wait(ta, o);
#pragma unroll
          for (int h = 0; h < 64; ++h) o[h] *= facb[buf * HG + h];
          tc::tmem_st64_wait(ta, o);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&c_done[buf]);
    }
    // ---------------- epilogue: O^T out of TMEM, normalised (one split) or as a partial
    const bool have = nch > 0;
    if (have) wait(&kv_empty[(nch - 1) & 1], (nch - 1) >> 1, 51);
    wait(sm_done, 0, 52);
    tc::tc_fence_after();
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      const int d = mt * 128 + quarter * 32 + lane;
      float o[64];
      if (have) {
        tc::tmem_ld64_wait(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 2 * HG + mt * HG, o);
      } else {
#pragma unroll
        for (int h = 0; h < 64; ++h) o[h] = 0.f;
      }
      if (a.n_splits == 1) {
        __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
        const bool rot = a.out_unrotate && d >= D - a.rp.r;      // warp-uniform (32-dim groups)
        float cs = 1.f, sn = 0.f;
        if (rot) {                                                 // rotation by -t
          const float2 cssn = rope[(d - (D - a.rp.r)) >> 1];
          cs = cssn.x;
          sn = -cssn.y;
        }
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          float x = o[h] * fin[h];
          if (rot) {
            const float y = __shfl_xor_sync(0xffffffffu, x, 1);
            x = (lane & 1) ? (y * sn + x * cs) : (x * cs - y * sn);
          }
          outp[(qi * a.H + h0 + h) * static_cast<long long>(D) + d] = __float2bfloat16_rn(x);
        }
      } else {
        float* po = a.partial;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          const size_t rowi = (static_cast<size_t>(qi) * a.n_splits + split) * a.H + h0 + h;
          po[rowi * D + d] = o[h];
        }
      }
    }
  }

  // ---------------- teardown: every MMA complete (the MMA thread drained) before TMEM is released
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool attend_tc_supported(const AttendArgs& a) {
  return a.d == D && !a.fp8 && a.H % HG == 0 && a.rp.r % 64 == 0 && a.rp.r <= D;
}

cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s, int* launches) {
  cudaError_t e = cudaFuncSetAttribute(k_attend_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  const int Q = a.B * a.Tq;
  e = launch_k(k_attend_tc, dim3(Q, a.H / HG, a.n_splits), dim3(NT), static_cast<size_t>(SMEM), s, a);
  ++*launches;
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attend_combine(a, s, launches);
}

}  // namespace csa
