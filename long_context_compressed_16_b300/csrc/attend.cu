// Shared K=V multi-query attention over the selected (CSA) or all closed (HCA) compressed entries
// plus the uncompressed SWA window, with a per-head sink logit and the reverse rotation of the
// output's RoPE dims ("DeepSeek V4 模型技术大全", component table rows Shared K=V MQA, query/KV
// RMSNorm, partial RoPE, attention sink, SWA; the HCA visibility set; the reverse-rotation note).
//
// Per query the candidate rows are laid out as "slots": [0, K_q) entry slots (the idx row, or
// entries 0..N_vis-1 for HCA) followed by `window` window slots (positions t-window+1 .. t).
// A CTA owns one query, a group of 16*NG heads and one split of the slot range.  Rows are
// gathered CK at a time with cp.async into a double-buffered shared-memory tile; the heads x keys
// logits and the heads x d output run on the tensor
// cores; the softmax is online in the log2 domain and the sink joins the normaliser at the end.
// bf16 rows: the query enters the logits exactly.  q_hat = inv * RoPE_t(q) (inv the RMSNorm
// factor), so the unrotated dims are the query's own bf16 bits, the rotated dims a bf16 hi + lo
// pair (the lo block spans the last r rounded up to 16 dims, zero where nothing is rotated), and
// inv multiplies the fp32 logit.  The FP8 rows use an fp16 hi + lo split of q_hat instead.
// Split boundaries sit at fixed multiples of the split size in slot space, never depending on
// the batch, and splits are merged by a second kernel in fixed order (batch-invariant decode).
#include "common.cuh"

namespace csa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int NG, bool FP8>
struct AttnCfg {
  // keys per chunk: fixed per row format (never per head grouping), so the rounding of the
  // probabilities, which follows the chunked running maximum, is identical for any batch size
  static constexpr int CK = FP8 ? 32 : 64;
  static constexpr int NKT = CK / 32;                         // n8 key tiles per warp (S phase)
  static constexpr int HG = 16 * NG;                          // heads per CTA
  static constexpr int THREADS = 128 * NG;
  static constexpr int QS = D + 8;                            // padded smem row strides (bf16)
  static constexpr int LS = 128 + 8;                          // lo block of the rotated dims (r <= 128)
  static constexpr int KS = D + 8;
  static constexpr int PS = CK + 8;
  static constexpr int ROWB = FP8 ? CSA_FP8_MIXED_ROW_BYTES : D * 2;   // global row bytes
  // FP8 rows: 8 blocks of 64 dims (7 e4m3 blocks with their own scale + the bf16 RoPE block).
  // That path multiplies in fp16: e4m3 codes and the bf16 parts are exact in fp16, the query is
  // split into fp16 hi + lo, and block scales are applied in fp32.
  static constexpr int NB = FP8 ? D / 64 : 1;
  static constexpr int QPARTS = FP8 ? 2 : 1;
  static constexpr size_t q_off = 0;
  static constexpr size_t lo_off = q_off + size_t(QPARTS) * HG * QS * 2;
  static constexpr size_t inv_off = lo_off + (FP8 ? 0 : size_t(HG) * LS * 2);
  static constexpr size_t k_off = inv_off + (FP8 ? 0 : size_t(HG) * 4);
  static constexpr size_t st_off = k_off + size_t(2) * CK * KS * 2;
  static constexpr size_t p_off = st_off + (FP8 ? size_t(2) * CK * ROWB : 0);
  static constexpr size_t sc_off = p_off + size_t(NB) * HG * PS * 2;
  static constexpr size_t red_off = sc_off + (FP8 ? size_t(2) * CK * NB * 4 : 0);
  static constexpr size_t lsum_off = red_off + size_t(HG) * 4 * 4;
  static constexpr size_t ptr_off = lsum_off + size_t(HG) * 4 * 4;
  static constexpr size_t rope_off = ptr_off + size_t(3) * CK * 8;   // float2 [kMaxRopePairs]
  static constexpr size_t smem = rope_off + size_t(kMaxRopePairs) * 8;
  static_assert(!FP8 || (NG == 1 && D == 512), "the FP8 cache path runs 16 heads per CTA, d = 512");
};

// The idx value of slot s (its only global read), loaded ahead of slot_row.
__device__ __forceinline__ int slot_raw(const AttendArgs& a, long long qi, int Kq, int s) {
  return (s < Kq && a.idx != nullptr) ? a.idx[qi * a.k + s] : 0;
}

__device__ __forceinline__ int slot_row(const AttendArgs& a, int t, int Kq, int s, int raw, bool& win_row,
                                        int32_t* status) {
  // returns the row index (entry index or ring slot) or -1 when the slot holds nothing
  if (s < Kq) {
    win_row = false;
    if (a.idx == nullptr) return s;
    const int e = raw;
    if (e == -1) return -1;
    if (e < -1 || e >= a.N) {
      report_error(status, CSA_ERR_DEVICE_CHECK, e);
      return -1;
    }
    return e;
  }
  const int j = s - Kq;
  if (j >= a.window) return -1;
  win_row = true;
  const int u = t - a.window + 1 + j;
  if (u < 0) return -1;
  return u % a.Wcap;
}

template <int D, int NG, bool FP8>
__global__ void __launch_bounds__(AttnCfg<D, NG, FP8>::THREADS, 1) k_attend(AttendArgs a) {
  using C = AttnCfg<D, NG, FP8>;
  constexpr int CK = C::CK, NKT = C::NKT, HG = C::HG, QS = C::QS, KS = C::KS, PS = C::PS;
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem + C::q_off);
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem + C::k_off);
  unsigned char* St = smem + C::st_off;
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + C::p_off);
  float* bscale = reinterpret_cast<float*>(smem + C::sc_off);      // FP8: [2][CK][NB] row block scales
  float* redmax = reinterpret_cast<float*>(smem + C::red_off);
  float* lsum = reinterpret_cast<float*>(smem + C::lsum_off);
  const unsigned char** rowptr = reinterpret_cast<const unsigned char**>(smem + C::ptr_off);
  float2* rope_tab = reinterpret_cast<float2*>(smem + C::rope_off);   // (cos, sin) of t * inv_freq_j
  __nv_bfloat16* Qlo = reinterpret_cast<__nv_bfloat16*>(smem + C::lo_off);   // bf16 rows: [HG][LS]
  float* qinv = reinterpret_cast<float*>(smem + C::inv_off);                 // bf16 rows: [HG]
  grid_dep_wait();
  grid_dep_launch();

  const int tid = threadIdx.x, lane = tid & 31, wall = tid >> 5;
  const int g = wall >> 2, wq = wall & 3;
  const int split = blockIdx.z;
  const int h0 = blockIdx.y * HG;
  const long long qi = blockIdx.x;
  const int b = static_cast<int>(qi / a.Tq);
  const int t = a.q_pos[qi];
  const int nvis = n_visible(t, a.m, a.N);
  const int Kq = (a.idx == nullptr) ? nvis : a.k;
  const int nslots = Kq + a.window;
  const int s_begin = split * a.split_slots;
  const int s_end = min(nslots, s_begin + a.split_slots);
  const int nchunks = s_end > s_begin ? (s_end - s_begin + CK - 1) / CK : 0;

  const unsigned char* kvb = static_cast<const unsigned char*>(a.kv);
  const unsigned char* winb = static_cast<const unsigned char*>(a.win);
  const unsigned char* dummy = static_cast<const unsigned char*>(a.q);   // source of zero-size copies

  // Row pointers of chunk c live in rowptr[(c % 3) * CK ...]: the idx values of chunk c + 2 are
  // loaded at the top of chunk c's iteration and turned into pointers after its QK^T product,
  // so their latency hides behind that product instead of stalling the next gather.
  auto load_raw = [&](int c) -> int {
    const int s = s_begin + c * CK + tid;
    return (tid < CK && s < s_end) ? slot_raw(a, qi, Kq, s) : 0;
  };
  auto compute_ptrs = [&](int c, int buf, int raw) {
    if (tid < CK) {
      const int s = s_begin + c * CK + tid;
      const unsigned char* p = nullptr;
      if (s < s_end) {
        bool isw = false;
        const int r = slot_row(a, t, Kq, s, raw, isw, a.status);
        if (r >= 0) {
          p = isw ? winb + (static_cast<size_t>(b) * a.Wcap + r) * (D * 2)
                  : kvb + (static_cast<size_t>(b) * a.N + r) * C::ROWB;
          if (FP8 && isw) p = reinterpret_cast<const unsigned char*>(reinterpret_cast<uintptr_t>(p) | 1u);
        }
      }
      rowptr[buf * CK + tid] = p;
    }
  };
  // cp.async of chunk rows into Ks (bf16) or the FP8 staging area (window rows go straight to Ks)
  auto issue_loads = [&](int buf, int pbuf) {
    constexpr int CPR = D * 2 / 16;
    for (int c = tid; c < CK * CPR; c += C::THREADS) {
      const int r = c / CPR, q = c % CPR;
      const unsigned char* p = rowptr[pbuf * CK + r];
      __nv_bfloat16* kd = Ks + (buf * CK + r) * KS + q * 8;
      if (!FP8) {
        cp_async16(kd, p ? p + q * 16 : dummy, p != nullptr);
      } else {
        const bool isw = (reinterpret_cast<uintptr_t>(p) & 1u) != 0;
        const unsigned char* pw = reinterpret_cast<const unsigned char*>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(1));
        if (isw) {
          cp_async16(kd, pw + q * 16, true);
        } else if (q < C::ROWB / 16) {
          cp_async16(St + (buf * CK + r) * C::ROWB + q * 16, p ? p + q * 16 : dummy, p != nullptr);
        }
      }
    }
  };

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  constexpr int NO = D / 32;          // n8 tiles of output dims per warp (D/4 dims)
  float oacc[NO][4];
#pragma unroll
  for (int i = 0; i < NO; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) oacc[i][c] = 0.f;
  const float sl2 = a.scale * kLog2e;

  // the first chunk's row gather is in flight while the query block is prepared
  if (nchunks > 0) {
    const int raw0 = load_raw(0);
    const int raw1 = nchunks > 1 ? load_raw(1) : 0;
    compute_ptrs(0, 0, raw0);
    if (nchunks > 1) compute_ptrs(1, 1, raw1);
    __syncthreads();
    issue_loads(0, 0);
    cp_async_commit();
  }

  // ---------------- prologue: the query block in shared memory (bf16 rows: raw q, the rotated
  // dims as hi + lo, inv per head; FP8 rows: q_hat = RoPE_t(RMSNorm(q)) as fp16 hi + lo).  The
  // query's rotation angles are shared by all heads: one (cos, sin) table per CTA.
  const int r16 = (a.q_norm_rope && !FP8) ? ((a.rp.r + 15) & ~15) : 0;   // dims of the lo block
  if (tid < a.rp.r / 2) {
    float cs, sn;
    rope_cos_sin(t, a.rp.phase[tid], cs, sn);
    rope_tab[tid] = make_float2(cs, sn);
  }
  __syncthreads();
  {
    constexpr int E = D / 32;   // elements per lane
    const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(a.q);
    for (int hl = wall; hl < HG; hl += 4 * NG) {
      const __nv_bfloat16* src = qsrc + ((qi * a.H) + h0 + hl) * static_cast<long long>(D) + lane * E;
      float v[E];
      if constexpr (E >= 8) {
#pragma unroll
        for (int c = 0; c < E; c += 8) {
          const uint4 u = *reinterpret_cast<const uint4*>(src + c);
          v[c + 0] = bf16lo(u.x); v[c + 1] = bf16hi(u.x);
          v[c + 2] = bf16lo(u.y); v[c + 3] = bf16hi(u.y);
          v[c + 4] = bf16lo(u.z); v[c + 5] = bf16hi(u.z);
          v[c + 6] = bf16lo(u.w); v[c + 7] = bf16hi(u.w);
        }
      } else {
        static_assert(E == 4, "d must be 128 or 512");
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        v[0] = bf16lo(u.x); v[1] = bf16hi(u.x);
        v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
      }
      if (a.q_norm_rope) {
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) ss = fmaf(v[c], v[c], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + a.eps);
        if constexpr (FP8) {
#pragma unroll
          for (int c = 0; c < E; ++c) v[c] *= inv;
        } else if (lane == 0) {
          qinv[hl] = inv;
        }
        const int cbase = lane * E;
        if (cbase + E > D - a.rp.r) {
#pragma unroll
          for (int c = 0; c < E; c += 2) {
            const int ch = cbase + c;
            if (ch >= D - a.rp.r) {
              const float2 cssn = rope_tab[(ch - (D - a.rp.r)) >> 1];
              const float cs = cssn.x, sn = cssn.y;
              const float x0 = v[c], x1 = v[c + 1];
              v[c] = x0 * cs - x1 * sn;
              v[c + 1] = x0 * sn + x1 * cs;
            }
          }
        }
      }
      if constexpr (!FP8) {
        if (!a.q_norm_rope && lane == 0) qinv[hl] = 1.f;
        // lo half of the last r16 dims (zero where the dim is not rotated: raw q is exact in bf16)
        const int cbase = lane * E;
        if (r16 > 0 && cbase + E > D - r16) {
#pragma unroll
          for (int c = 0; c < E; ++c) {
            const int ch = cbase + c;
            if (ch >= D - r16) {
              const float hi = __bfloat162float(__float2bfloat16_rn(v[c]));
              Qlo[hl * C::LS + (ch - (D - r16))] = __float2bfloat16_rn(v[c] - hi);
            }
          }
        }
      }
      __nv_bfloat16* dst = Qs + hl * QS + lane * E;
      if constexpr (FP8) {
#pragma unroll
        for (int c = 0; c < E; c += 8) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int p2 = 0; p2 < 4; ++p2) {
            const float x0 = v[c + 2 * p2], x1 = v[c + 2 * p2 + 1];
            hw[p2] = pack_half2(x0, x1);
            const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hw[p2]));
            lw[p2] = pack_half2(x0 - hf.x, x1 - hf.y);        // residual: hi + lo ~ 22 significant bits
          }
          *reinterpret_cast<uint4*>(dst + c) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(dst + HG * QS + c) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      } else if constexpr (E >= 8) {
#pragma unroll
        for (int c = 0; c < E; c += 8) {
          uint4 u;
          u.x = pack_bf16x2(v[c + 0], v[c + 1]);
          u.y = pack_bf16x2(v[c + 2], v[c + 3]);
          u.z = pack_bf16x2(v[c + 4], v[c + 5]);
          u.w = pack_bf16x2(v[c + 6], v[c + 7]);
          *reinterpret_cast<uint4*>(dst + c) = u;
        }
      } else {
        uint2 u;
        u.x = pack_bf16x2(v[0], v[1]);
        u.y = pack_bf16x2(v[2], v[3]);
        *reinterpret_cast<uint2*>(dst) = u;
      }
    }
  }

  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const int pb = c % 3;
    const int raw_next = c + 2 < nchunks ? load_raw(c + 2) : 0;
    __syncthreads();                                   // (A)
    if (c + 1 < nchunks) {
      issue_loads(buf ^ 1, (c + 1) % 3);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();                                   // (B)
    if (FP8) {
      // fp16 tile: entry rows take their e4m3 codes (exact) and the bf16 RoPE block; window rows,
      // cp.async'ed as bf16, are converted in place; block scales go to shared memory (window
      // rows and the RoPE block use scale 1)
      for (int idx = tid; idx < CK * (D / 8); idx += C::THREADS) {
        const int r = idx / (D / 8), p8 = idx % (D / 8);
        const unsigned char* p = rowptr[pb * CK + r];
        const bool isw = (reinterpret_cast<uintptr_t>(p) & 1u) != 0;
        const unsigned char* row = St + (buf * CK + r) * C::ROWB;
        if ((p8 & 7) == 0) {
          const int blk = p8 >> 3;
          float sc = 1.f;
          if (!isw && blk < 7) sc = (p != nullptr) ? *reinterpret_cast<const float*>(row + 576 + blk * 4) : 0.f;
          bscale[(buf * CK + r) * C::NB + blk] = sc;
        }
        __nv_bfloat16* kd = Ks + (buf * CK + r) * KS + p8 * 8;
        uint4 src;
        if (isw || p8 >= 56) {
          src = isw ? *reinterpret_cast<const uint4*>(kd)
                    : *reinterpret_cast<const uint4*>(row + 448 + (p8 - 56) * 16);
          src = make_uint4(pack_half2(bf16lo(src.x), bf16hi(src.x)), pack_half2(bf16lo(src.y), bf16hi(src.y)),
                           pack_half2(bf16lo(src.z), bf16hi(src.z)), pack_half2(bf16lo(src.w), bf16hi(src.w)));
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(row + p8 * 8);
          src = make_uint4(e4m3x2_to_half2(static_cast<uint16_t>(v.x & 0xFFFF)), e4m3x2_to_half2(static_cast<uint16_t>(v.x >> 16)),
                           e4m3x2_to_half2(static_cast<uint16_t>(v.y & 0xFFFF)), e4m3x2_to_half2(static_cast<uint16_t>(v.y >> 16)));
        }
        *reinterpret_cast<uint4*>(kd) = src;
      }
      __syncthreads();                                 // (B')
    }
    const __nv_bfloat16* Kb = Ks + buf * CK * KS;

    // ---- S = Q K^T for heads [16g, 16g+16) x keys [wq*8*NKT, +8*NKT)
    float sacc[NKT][4];
#pragma unroll
    for (int n = 0; n < NKT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[n][e] = 0.f;
    if constexpr (!FP8) {
#pragma unroll 4
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4];
        ldmatrix_x4(af[0], af[1], af[2], af[3],
                    smem_u32(Qs + (16 * g + (lane & 15)) * QS + ks * 16 + (lane >> 4) * 8));
        if (NKT == 2) {
          uint32_t b0, b1, b2, b3;
          const int key = wq * 16 + (lane >> 4) * 8 + (lane & 7);
          ldmatrix_x4(b0, b1, b2, b3, smem_u32(Kb + key * KS + ks * 16 + ((lane >> 3) & 1) * 8));
          const uint32_t bb0[2] = {b0, b1}, bb1[2] = {b2, b3};
          mma_bf16_16816(sacc[0], af, bb0);
          mma_bf16_16816(sacc[NKT - 1], af, bb1);
        } else {
          uint32_t b0, b1;
          const int key = wq * 8 + (lane & 7);
          ldmatrix_x2(b0, b1, smem_u32(Kb + key * KS + ks * 16 + ((lane >> 3) & 1) * 8));
          const uint32_t bb0[2] = {b0, b1};
          mma_bf16_16816(sacc[0], af, bb0);
        }
      }
      // lo half of the rotated dims against the keys' last r16 dims
      for (int kl = 0; kl < r16 / 16; ++kl) {
        const int kd = D - r16 + kl * 16;
        uint32_t af[4];
        ldmatrix_x4(af[0], af[1], af[2], af[3],
                    smem_u32(Qlo + (16 * g + (lane & 15)) * C::LS + kl * 16 + (lane >> 4) * 8));
        if (NKT == 2) {
          uint32_t b0, b1, b2, b3;
          const int key = wq * 16 + (lane >> 4) * 8 + (lane & 7);
          ldmatrix_x4(b0, b1, b2, b3, smem_u32(Kb + key * KS + kd + ((lane >> 3) & 1) * 8));
          const uint32_t bb0[2] = {b0, b1}, bb1[2] = {b2, b3};
          mma_bf16_16816(sacc[0], af, bb0);
          mma_bf16_16816(sacc[NKT - 1], af, bb1);
        } else {
          uint32_t b0, b1;
          const int key = wq * 8 + (lane & 7);
          ldmatrix_x2(b0, b1, smem_u32(Kb + key * KS + kd + ((lane >> 3) & 1) * 8));
          const uint32_t bb0[2] = {b0, b1};
          mma_bf16_16816(sacc[0], af, bb0);
        }
      }
    } else {
      // z = sum_b scale_{j,b} * (q_hat_b . code_{j,b}), q_hat = hi + lo (fp16), each block in fp32
      const float* scb = bscale + buf * CK * C::NB;
      const int kc0 = wq * 8 + 2 * (lane & 3);
#pragma unroll 1
      for (int blk = 0; blk < C::NB; ++blk) {
        float pacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int ks = blk * 4 + kq;
          uint32_t ah[4], al[4];
          ldmatrix_x4(ah[0], ah[1], ah[2], ah[3],
                      smem_u32(Qs + (lane & 15) * QS + ks * 16 + (lane >> 4) * 8));
          ldmatrix_x4(al[0], al[1], al[2], al[3],
                      smem_u32(Qs + HG * QS + (lane & 15) * QS + ks * 16 + (lane >> 4) * 8));
          uint32_t b0, b1;
          const int key = wq * 8 + (lane & 7);
          ldmatrix_x2(b0, b1, smem_u32(Kb + key * KS + ks * 16 + ((lane >> 3) & 1) * 8));
          const uint32_t bb0[2] = {b0, b1};
          mma_f16_16816(pacc, ah, bb0);
          mma_f16_16816(pacc, al, bb0);
        }
        const float s0 = scb[kc0 * C::NB + blk], s1 = scb[(kc0 + 1) * C::NB + blk];
        sacc[0][0] = fmaf(pacc[0], s0, sacc[0][0]);
        sacc[0][1] = fmaf(pacc[1], s1, sacc[0][1]);
        sacc[0][2] = fmaf(pacc[2], s0, sacc[0][2]);
        sacc[0][3] = fmaf(pacc[3], s1, sacc[0][3]);
      }
    }
    // chunk c + 2's pointers: rowptr[(c + 2) % 3] last served chunk c - 1, finished before (A)
    if (c + 2 < nchunks) compute_ptrs(c + 2, (c + 2) % 3, raw_next);
    // ---- mask, scale to log2 domain (bf16 rows: times the head's RMSNorm factor), row max over
    // this warp's keys
    float rsc[2] = {sl2, sl2};
    if constexpr (!FP8) {
      rsc[0] = sl2 * qinv[16 * g + (lane >> 2)];
      rsc[1] = sl2 * qinv[16 * g + (lane >> 2) + 8];
    }
    float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < NKT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = wq * 8 * NKT + n * 8 + 2 * (lane & 3) + (e & 1);
        const bool ok = rowptr[pb * CK + key] != nullptr;
        const float v = ok ? sacc[n][e] * rsc[e >> 1] : -INFINITY;
        sacc[n][e] = v;
        cmax[e >> 1] = fmaxf(cmax[e >> 1], v);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      cmax[r] = fmaxf(cmax[r], __shfl_xor_sync(0xffffffffu, cmax[r], 1));
      cmax[r] = fmaxf(cmax[r], __shfl_xor_sync(0xffffffffu, cmax[r], 2));
    }
    if ((lane & 3) == 0) {
      redmax[(16 * g + (lane >> 2)) * 4 + wq] = cmax[0];
      redmax[(16 * g + (lane >> 2) + 8) * 4 + wq] = cmax[1];
    }
    __syncthreads();                                   // (C)
    float alpha[2], muse[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float* rm = redmax + (16 * g + (lane >> 2) + 8 * r) * 4;
      const float mc = fmaxf(fmaxf(rm[0], rm[1]), fmaxf(rm[2], rm[3]));
      const float mn = fmaxf(m_run[r], mc);
      muse[r] = (mn == -INFINITY) ? 0.f : mn;
      alpha[r] = exp2f(m_run[r] - muse[r]);
      m_run[r] = mn;
    }
    // ---- P = exp2(s - m), partial row sums, P (bf16) to shared memory
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < NKT; ++n) {
      const float p0 = exp2f(sacc[n][0] - muse[0]);
      const float p1 = exp2f(sacc[n][1] - muse[0]);
      const float p2 = exp2f(sacc[n][2] - muse[1]);
      const float p3 = exp2f(sacc[n][3] - muse[1]);
      psum[0] += p0 + p1;
      psum[1] += p2 + p3;
      const int key = wq * 8 * NKT + n * 8 + 2 * (lane & 3);
      const int hr = 16 * g + (lane >> 2);
      if constexpr (!FP8) {
        *reinterpret_cast<uint32_t*>(Ps + hr * PS + key) = pack_bf16x2(p0, p1);
        *reinterpret_cast<uint32_t*>(Ps + (hr + 8) * PS + key) = pack_bf16x2(p2, p3);
      } else {
        const float* scb = bscale + buf * CK * C::NB;
#pragma unroll
        for (int blk = 0; blk < C::NB; ++blk) {
          const float s0 = scb[key * C::NB + blk], s1 = scb[(key + 1) * C::NB + blk];
          __nv_bfloat16* pb = Ps + blk * HG * PS;
          // p * scale * 2^8 stays in fp16's normal range; the 2^-8 is taken back after the loop
          *reinterpret_cast<uint32_t*>(pb + hr * PS + key) = pack_half2(p0 * s0 * 256.f, p1 * s1 * 256.f);
          *reinterpret_cast<uint32_t*>(pb + (hr + 8) * PS + key) = pack_half2(p2 * s0 * 256.f, p3 * s1 * 256.f);
        }
      }
    }
    l_run[0] = l_run[0] * alpha[0] + psum[0];
    l_run[1] = l_run[1] * alpha[1] + psum[1];
#pragma unroll
    for (int i = 0; i < NO; ++i) {
      oacc[i][0] *= alpha[0]; oacc[i][1] *= alpha[0];
      oacc[i][2] *= alpha[1]; oacc[i][3] *= alpha[1];
    }
    __syncthreads();                                   // (D)
    // ---- O += P V for heads [16g,16g+16) x dims [wq*D/4, +D/4)
#pragma unroll
    for (int kk = 0; kk < CK / 16; ++kk) {
      uint32_t pa[4], pb2[4] = {0u, 0u, 0u, 0u};
      const __nv_bfloat16* P0 = FP8 ? Ps + (wq * 2) * HG * PS : Ps;
      ldmatrix_x4(pa[0], pa[1], pa[2], pa[3],
                  smem_u32(P0 + (16 * g + (lane & 15)) * PS + kk * 16 + (lane >> 4) * 8));
      if constexpr (FP8) {
        const __nv_bfloat16* P1 = Ps + (wq * 2 + 1) * HG * PS;
        ldmatrix_x4(pb2[0], pb2[1], pb2[2], pb2[3],
                    smem_u32(P1 + (16 * g + (lane & 15)) * PS + kk * 16 + (lane >> 4) * 8));
      }
#pragma unroll
      for (int np = 0; np < NO / 2; ++np) {
        uint32_t v0, v1, v2, v3;
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int dim = wq * (D / 4) + np * 16 + (lane >> 4) * 8;
        ldmatrix_x4_trans(v0, v1, v2, v3, smem_u32(Kb + key * KS + dim));
        const uint32_t vb0[2] = {v0, v1}, vb1[2] = {v2, v3};
        if constexpr (FP8) {
          const uint32_t* A = (np >= NO / 4) ? pb2 : pa;   // dims of the warp's second block
          mma_f16_16816(oacc[2 * np], A, vb0);
          mma_f16_16816(oacc[2 * np + 1], A, vb1);
        } else {
          mma_bf16_16816(oacc[2 * np], pa, vb0);
          mma_bf16_16816(oacc[2 * np + 1], pa, vb1);
        }
      }
    }
  }
  if constexpr (FP8) {
#pragma unroll
    for (int i = 0; i < NO; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) oacc[i][c] *= (1.0f / 256.0f);
  }

  // ---------------- epilogue: total row sums, sink, normalise / write partials
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  __syncthreads();
  if ((lane & 3) == 0) {
    lsum[(16 * g + (lane >> 2)) * 4 + wq] = l_run[0];
    lsum[(16 * g + (lane >> 2) + 8) * 4 + wq] = l_run[1];
  }
  __syncthreads();
  float ltot[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float* ls = lsum + (16 * g + (lane >> 2) + 8 * r) * 4;
    ltot[r] = (ls[0] + ls[1]) + (ls[2] + ls[3]);
  }
  const int Q = a.B * a.Tq;
  if (a.n_splits == 1) {
    float fac[2], linv[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = h0 + 16 * g + (lane >> 2) + 8 * r;
      const float a2 = a.sink[h] * kLog2e;
      const float M = fmaxf(m_run[r], a2);
      fac[r] = (m_run[r] == -INFINITY) ? 0.f : exp2f(m_run[r] - M);
      const float L = ltot[r] * fac[r] + exp2f(a2 - M);
      linv[r] = 1.0f / L;
      if (a.lse != nullptr && wq == 0 && (lane & 3) == 0) a.lse[qi * a.H + h] = (M + log2f(L)) * kLn2;
    }
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
    for (int i = 0; i < NO; ++i) {
      const int dim = wq * (D / 4) + i * 8 + 2 * (lane & 3);
      float cs = 1.f, sn = 0.f;
      const bool rot = a.out_unrotate && dim >= D - a.rp.r;
      if (rot) {                      // rotation by -t: (cos, -sin) of the query's angles
        const float2 cssn = rope_tab[(dim - (D - a.rp.r)) >> 1];
        cs = cssn.x;
        sn = -cssn.y;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int h = h0 + 16 * g + (lane >> 2) + 8 * r;
        float x0 = oacc[i][2 * r] * fac[r] * linv[r];
        float x1 = oacc[i][2 * r + 1] * fac[r] * linv[r];
        if (rot) {
          const float y0 = x0 * cs - x1 * sn, y1 = x0 * sn + x1 * cs;
          x0 = y0; x1 = y1;
        }
        *reinterpret_cast<uint32_t*>(outp + (qi * a.H + h) * static_cast<long long>(D) + dim) =
            pack_bf16x2(x0, x1);
      }
    }
  } else {
    // partial: O (relative to m_run, log2 domain) and (m, l) per (query, split, head)
    float* po = a.partial;
    float* pml = a.partial + static_cast<size_t>(Q) * a.n_splits * a.H * D;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = h0 + 16 * g + (lane >> 2) + 8 * r;
      const size_t rowi = (static_cast<size_t>(qi) * a.n_splits + split) * a.H + h;
      if (wq == 0 && (lane & 3) == 0) {
        pml[rowi * 2 + 0] = m_run[r];
        pml[rowi * 2 + 1] = ltot[r];
      }
#pragma unroll
      for (int i = 0; i < NO; ++i) {
        const int dim = wq * (D / 4) + i * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(po + rowi * D + dim) = make_float2(oacc[i][2 * r], oacc[i][2 * r + 1]);
      }
    }
  }
}

// Merge split partials: out = sum_s O_s 2^(m_s - M) / (sum_s l_s 2^(m_s - M) + 2^(a_h - M)),
// M = max(a_h, max_s m_s), in fixed split order.  One CTA per (query, pair of heads), 128 threads
// per head: the two heads' merge factors and the query's rotation table are computed once in
// shared memory, then each thread merges dim pairs of its head.
constexpr int kCombineHeads = 2;

template <int D>
__global__ void __launch_bounds__(128 * kCombineHeads) k_attend_combine(AttendArgs a) {
  extern __shared__ float csm[];
  grid_dep_wait();
  grid_dep_launch();
  const long long qi = blockIdx.x;
  const int h0 = blockIdx.y * kCombineHeads;
  const int S = a.n_splits, H = a.H;
  const int Q = a.B * a.Tq;
  float* fac = csm;                                                               // [2][S]
  float2* tab = reinterpret_cast<float2*>(csm + ((kCombineHeads * S + 1) & ~1));  // [r/2]
  const float* po = a.partial;
  const float* pml = a.partial + static_cast<size_t>(Q) * S * H * D;
  const int t = a.q_pos[qi];
  const int tid = threadIdx.x;
  if (tid < a.rp.r / 2) {
    float cs, sn;
    rope_cos_sin(t, a.rp.phase[tid], cs, sn);
    tab[tid] = make_float2(cs, -sn);                                              // rotation by -t
  }
  if (tid < kCombineHeads) {
    const int h = h0 + tid;
    const float a2 = a.sink[h] * kLog2e;
    float M = a2;
    for (int s = 0; s < S; ++s) M = fmaxf(M, pml[((qi * S + s) * H + h) * 2]);
    float L = exp2f(a2 - M);
    for (int s = 0; s < S; ++s) {
      const size_t ri = (static_cast<size_t>(qi) * S + s) * H + h;
      const float ms = pml[ri * 2];
      if (ms != -INFINITY) L = fmaf(pml[ri * 2 + 1], exp2f(ms - M), L);
    }
    const float linv = 1.0f / L;
    for (int s = 0; s < S; ++s) {
      const float ms = pml[((qi * S + s) * H + h) * 2];
      fac[tid * S + s] = (ms == -INFINITY) ? 0.f : exp2f(ms - M) * linv;
    }
    if (a.lse != nullptr) a.lse[qi * H + h] = (M + log2f(L)) * kLn2;
  }
  __syncthreads();
  const int hl = tid / 128;
  const int h = h0 + hl;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
  for (int pr = tid % 128; pr < D / 2; pr += 128) {
    const int dim = pr * 2;
    float x0 = 0.f, x1 = 0.f;
    for (int s = 0; s < S; ++s) {
      const float f = fac[hl * S + s];         // 0 for a split without rows (its partial is zeros)
      const float2 v = *reinterpret_cast<const float2*>(po + ((static_cast<size_t>(qi) * S + s) * H + h) * D + dim);
      x0 = fmaf(v.x, f, x0);
      x1 = fmaf(v.y, f, x1);
    }
    if (a.out_unrotate && dim >= D - a.rp.r) {
      const float2 cssn = tab[(dim - (D - a.rp.r)) >> 1];
      const float y0 = x0 * cssn.x - x1 * cssn.y, y1 = x0 * cssn.y + x1 * cssn.x;
      x0 = y0; x1 = y1;
    }
    *reinterpret_cast<uint32_t*>(outp + (qi * H + h) * static_cast<long long>(D) + dim) = pack_bf16x2(x0, x1);
  }
}

template <int D, int NG, bool FP8>
cudaError_t launch_t(const AttendArgs& a, cudaStream_t s, int* launches) {
  using C = AttnCfg<D, NG, FP8>;
  cudaError_t e = cudaFuncSetAttribute(k_attend<D, NG, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::smem));
  if (e != cudaSuccess) return e;
  const int Q = a.B * a.Tq;
  dim3 grid(Q, a.H / C::HG, a.n_splits);
  e = launch_k(k_attend<D, NG, FP8>, grid, dim3(C::THREADS), C::smem, s, a);
  ++*launches;
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attend_combine(a, s, launches);
}

template <int D>
cudaError_t launch_combine_t(const AttendArgs& a, cudaStream_t s, int* launches) {
  const int Q = a.B * a.Tq;
  const size_t csmem =
      (static_cast<size_t>((kCombineHeads * a.n_splits + 1) & ~1) + 2 * kMaxRopePairs) * sizeof(float);
  if (csmem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_attend_combine<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(csmem));
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch_k(k_attend_combine<D>, dim3(Q, a.H / kCombineHeads), dim3(128 * kCombineHeads), csmem,
                                 s, a);
  ++*launches;
  return e;
}

}  // namespace

cudaError_t launch_attend_combine(const AttendArgs& a, cudaStream_t s, int* launches) {
  if (a.n_splits <= 1 || a.B * a.Tq == 0) return cudaSuccess;
  if (a.d == 512) return launch_combine_t<512>(a, s, launches);
  if (a.d == 128) return launch_combine_t<128>(a, s, launches);
  return cudaErrorInvalidValue;
}

size_t attend_partial_bytes(int Q, int H, int d, int n_splits) {
  if (n_splits <= 1) return 0;
  return static_cast<size_t>(Q) * n_splits * H * (d + 2) * sizeof(float);
}

cudaError_t launch_attend(const AttendArgs& a, cudaStream_t s, int* launches) {
  const int Q = a.B * a.Tq;
  if (Q == 0) return cudaSuccess;
#ifndef CSA_ATT_WARP_MMA_ONLY
  if (attend_tc_supported(a)) return launch_attend_tc(a, s, launches);
#endif
  // 64 heads per CTA (each gathered row read once) when that still gives work to at least half
  // of the SMs, otherwise 16 heads per CTA; the numerics are identical
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool wide = (a.H % 64 == 0) && (2LL * Q * a.n_splits * (a.H / 64) >= sms);
  if (a.d == 512) {
    if (a.fp8) return launch_t<512, 1, true>(a, s, launches);
    return wide ? launch_t<512, 4, false>(a, s, launches) : launch_t<512, 1, false>(a, s, launches);
  }
  if (a.d == 128 && !a.fp8) {
    return wide ? launch_t<128, 4, false>(a, s, launches) : launch_t<128, 1, false>(a, s, launches);
  }
  return cudaErrorInvalidValue;
}

}  // namespace csa
