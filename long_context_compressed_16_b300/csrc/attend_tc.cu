// Shared K=V multi-query attention on the 5th-generation tensor cores, for 512-dim bf16 rows
// and 64 query heads per CTA ("DeepSeek V4 模型技术大全", component table rows Shared K=V MQA,
// query/KV RMSNorm, partial RoPE, attention sink, SWA; the HCA visibility set; the
// reverse-rotation note).  Same slots, splits and partial format as the warp-MMA kernel in
// attend.cu, which keeps the other shapes (d = 128, the FP8 cache).
//
// Per CTA: one query, 64 heads, one split of the slot range, processed 64 rows at a time.
//   S^T = K q_hat^T   tcgen05.mma M = 128 rows (64 valid), N = 64 heads, K = 512, fp32 in TMEM:
//                     one TMEM lane per row, so the rows of a chunk are TMEM lanes 0..63
//   softmax           four warps, one thread per (row, half of the heads): exp2 against a per-head
//                     reference maximum that is set exactly (warp butterfly) from the first rows
//                     and afterwards only moves when a logit exceeds it by more than 2^8 (the O
//                     accumulator is then rescaled in TMEM); P^T is written to shared memory as
//                     bf16 and the per-head row sums are read back from it, so the normaliser
//                     uses exactly the probabilities the PV product uses
//   O^T += V^T P^T    tcgen05.mma M = 128 dims (4 tiles), N = 64 heads, K = 64 rows; V^T is the
//                     same shared-memory rows read through an MN-major descriptor (K = V)
// Rows are gathered by one loader warp with TMA tile::gather4 (four rows per instruction; the
// rare group of four that mixes cache entries and window rows uses cp.async) into two 64-row
// buffers laid out in the 128-byte swizzle, so the next chunk's gather overlaps the current
// chunk's math.  One thread
// issues all MMAs; eight warps prepare the query block and read the accumulator out.  Waits are
// bounded (CSA_ERR_TIMEOUT, never a hang).
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
constexpr float kRescaleLog2 = 8.f;           // move a head's reference maximum only past 2^8

constexpr int Q_REGION = HG * 128;            // 64 heads x 64 dims (bf16)
constexpr int Q_BYTES = NREG * Q_REGION;      // 64 KB
constexpr int KV_REGION = 2 * CK * 128;       // two buffers x 64 rows x 64 dims
constexpr int KV_BYTES = NREG * KV_REGION;    // 128 KB
constexpr int PT_BYTES = HG * 128;            // P^T of one chunk: 64 heads x 64 rows
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + Q_BYTES;
constexpr int OFF_PT = OFF_KV + KV_BYTES;     // two P^T buffers (also cover the S over-read)
constexpr int OFF_MISC = OFF_PT + 2 * PT_BYTES;
constexpr int kMaxSlots = 2304;               // rows of one split whose indices are staged
constexpr int MISC_BYTES = kMaxSlots * 4 + 2560;
constexpr int SMEM = 1024 + OFF_MISC + MISC_BYTES;
constexpr int NTHREADS = 320;                 // warps 0-7 compute (0,1,4,5 softmax), 8 MMA, 9 loader
constexpr int NLOAD = 32;                     // loader threads (one warp issuing TMA gathers)
constexpr int MMA_WARP = 8;
constexpr int LOADER_WARP0 = 9;
constexpr int TMEM_COLS = 512;                // S^T x2 at columns 0, 64; O^T tiles at 128 + 64*mt
constexpr int kWinFlag = 1 << 30;             // row index of a window slot (ring slot | flag)
static_assert(SMEM <= 232448, "shared memory budget");

struct Misc {
  int* rowidx;                    // [kMaxSlots] entry index, window slot | kWinFlag, or -1
  float2* rope;                   // [kMaxRopePairs] (cos, sin) of t * inv_freq_j
  float* Rref;                    // [HG] reference maximum (log2 domain)
  float* Lsum;                    // [HG] sum of exp2(z - Rref)
  float* Fac;                     // [HG] rescale factor of this chunk
  float* norm;                    // [HG]
  float* red;                     // [2][HG]
  int* flags;                     // [8]
  uint64_t* bars;                 // [13]
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

__device__ __forceinline__ Misc carve_misc(unsigned char* base) {
  Misc m;
  m.rowidx = reinterpret_cast<int*>(base);
  unsigned char* r = base + kMaxSlots * 4;
  m.rope = reinterpret_cast<float2*>(r);                 // 512 B
  m.Rref = reinterpret_cast<float*>(r + 512);
  m.Lsum = m.Rref + HG;
  m.Fac = m.Lsum + HG;
  m.norm = m.Fac + HG;
  m.red = m.norm + HG;                                   // 2 * HG
  m.flags = reinterpret_cast<int*>(m.red + 2 * HG);      // r + 2048, 8 ints
  m.bars = reinterpret_cast<uint64_t*>(r + 2112);
  m.tmem_slot = reinterpret_cast<uint32_t*>(r + 2112 + 13 * 8);
  m.abort_flag = reinterpret_cast<volatile int*>(r + 2112 + 13 * 8 + 4);
  return m;
}

// q_hat = RoPE_t(RMSNorm(q)) in place for COUNT heads starting at head hl0 of the CTA.  The raw
// query block was loaded by TMA into the K-major 128-byte swizzled layout (the B operand of S):
// lane L of the warp owns dims 16L..16L+15 of a head, i.e. two 16-byte chunks of region L/4.
template <int COUNT>
__device__ __forceinline__ void norm_q_inplace(const AttendArgs& a, int hl0, const float2* rope, unsigned char* qs,
                                               int lane) {
  const int region = lane >> 2, ch0 = (lane & 3) * 2;
#pragma unroll 2
  for (int i = 0; i < COUNT; ++i) {
    const int hl = hl0 + i;
    unsigned char* row = qs + region * Q_REGION + hl * 128;
    uint4* p0 = reinterpret_cast<uint4*>(row + ((ch0 ^ (hl & 7)) << 4));
    uint4* p1 = reinterpret_cast<uint4*>(row + (((ch0 + 1) ^ (hl & 7)) << 4));
    const uint4 u0 = *p0, u1 = *p1;
    float v[16] = {bf16lo(u0.x), bf16hi(u0.x), bf16lo(u0.y), bf16hi(u0.y), bf16lo(u0.z), bf16hi(u0.z),
                   bf16lo(u0.w), bf16hi(u0.w), bf16lo(u1.x), bf16hi(u1.x), bf16lo(u1.y), bf16hi(u1.y),
                   bf16lo(u1.z), bf16hi(u1.z), bf16lo(u1.w), bf16hi(u1.w)};
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) ss = fmaf(v[c], v[c], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + a.eps);
#pragma unroll
    for (int c = 0; c < 16; ++c) v[c] *= inv;
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const int ch = lane * 16 + c;
      if (ch >= D - a.rp.r) {
        const float2 cssn = rope[(ch - (D - a.rp.r)) >> 1];
        const float x0 = v[c], x1 = v[c + 1];
        v[c] = x0 * cssn.x - x1 * cssn.y;
        v[c + 1] = x0 * cssn.y + x1 * cssn.x;
      }
    }
    *p0 = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    *p1 = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                     pack_bf16x2(v[14], v[15]));
  }
}

// Warp butterfly maximum over 32 values per lane: afterwards v[0] of lane L holds the maximum
// over the 32 lanes of column L.
__device__ __forceinline__ void butterfly_max32(float* v, int lane) {
#pragma unroll
  for (int o = 16, nc = 32; o >= 1; o >>= 1, nc >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < nc / 2) {
        const float send = up ? v[i] : v[i + nc / 2];
        const float keep = up ? v[i + nc / 2] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = fmaxf(keep, recv);
      }
    }
  }
}

__device__ __forceinline__ int slot_row_tc(const AttendArgs& a, long long qi, int t, int Kq, int s, bool& win_row) {
  if (s < Kq) {
    win_row = false;
    if (a.idx == nullptr) return s;
    const int e = a.idx[qi * a.k + s];
    if (e == -1) return -1;
    if (e < -1 || e >= a.N) {
      report_error(a.status, CSA_ERR_DEVICE_CHECK, e);
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

__global__ void __launch_bounds__(NTHREADS, 1) k_attend_tc(const AttendArgs a,
                                                            const __grid_constant__ CUtensorMap qmap,
                                                            const __grid_constant__ CUtensorMap kvmap,
                                                            const __grid_constant__ CUtensorMap winmap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (tc::sptr(smem_raw) & 1023u)) & 1023u);
  unsigned char* qs = sm + OFF_Q;
  unsigned char* kvs = sm + OFF_KV;
  unsigned char* pts = sm + OFF_PT;
  const Misc ms = carve_misc(sm + OFF_MISC);
  uint64_t* kv_full = ms.bars;        // [2] loader threads (128 arrivals)
  uint64_t* kv_empty = ms.bars + 2;   // [2] commit after PV
  uint64_t* s_full = ms.bars + 4;     // [2] commit after S
  uint64_t* p_full = ms.bars + 6;     // [2] softmax threads (128 arrivals)
  uint64_t* pv_done = ms.bars + 8;    // [2] commit after PV
  uint64_t* q_ready = ms.bars + 10;   // compute threads (256 arrivals)
  uint64_t* drain = ms.bars + 11;
  uint64_t* q_loaded = ms.bars + 12;  // TMA bytes of the raw query block

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

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&kv_full[i], NLOAD);
      tc::mbar_init(&kv_empty[i], 1);
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], 128);
      tc::mbar_init(&pv_done[i], 1);
    }
    tc::mbar_init(q_ready, 256);
    tc::mbar_init(drain, 1);
    tc::mbar_init(q_loaded, 1);
    *ms.abort_flag = 0;
    tc::fence_barrier_init();
    // raw query block: 64 heads x 512 dims as eight 64 x 64 boxes, straight into the operand layout
    tc::mbar_arrive_expect_tx(q_loaded, Q_BYTES);
    for (int r = 0; r < NREG; ++r)
      tc::tma_load_2d(qs + r * Q_REGION, &qmap, r * 64, static_cast<int>(qi * a.H + h0), q_loaded);
  }
  if (warp == MMA_WARP) {
    tc::tmem_alloc(ms.tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid < a.rp.r / 2) {
    float cs, sn;
    rope_cos_sin(static_cast<double>(t), a.rp.inv_freq[tid], cs, sn);
    ms.rope[tid] = make_float2(cs, sn);
  }
  if (tid < HG) {
    ms.Rref[tid] = -INFINITY;
    ms.Lsum[tid] = 0.f;
    ms.Fac[tid] = 1.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *ms.tmem_slot;
  auto fail = [&](int where) {
    *ms.abort_flag = 1;
    report_error(a.status, CSA_ERR_TIMEOUT, where);
  };

  if (warp == LOADER_WARP0) {
    // ------------------------------------------------------------ loader warp: row gather
    const unsigned char* kvb = static_cast<const unsigned char*>(a.kv);
    const unsigned char* winb = static_cast<const unsigned char*>(a.win);
    const unsigned char* dummy = static_cast<const unsigned char*>(a.q);
    // every row index of the split, once (one round of index loads for the whole split)
    for (int i = lane; i < nch * CK; i += NLOAD) {
      const int s = s_begin + i;
      int ri = -1;
      if (s < s_end) {
        bool isw = false;
        const int r = slot_row_tc(a, qi, t, Kq, s, isw);
        if (r >= 0) ri = isw ? (r | kWinFlag) : r;
      }
      ms.rowidx[i] = ri;
    }
    __syncwarp();
    // Groups of four rows: all cache entries (or empty) -> gather4 on the cache map; all window
    // rows (or empty) -> gather4 on the window map; an empty row reads a finite dummy row of the
    // same map (its probability is zero).  A group mixing both sources is copied with cp.async.
    const bool has_kv = a.N > 0;
    auto issue = [&](int c) {
      const int buf = c & 1;
      // classify the 16 groups of this chunk (lane g < 16 owns group g)
      int kind = 0;                                        // 0 cache gather, 1 window gather, 2 mixed
      int y[4] = {0, 0, 0, 0};
      if (lane < CK / 4) {
        bool any_kv = false, any_win = false;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ri = ms.rowidx[c * CK + lane * 4 + u];
          if (ri >= 0) {
            if (ri & kWinFlag) any_win = true; else any_kv = true;
          }
        }
        kind = (any_kv && any_win) ? 2 : ((any_win || !has_kv) ? 1 : 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ri = ms.rowidx[c * CK + lane * 4 + u];
          if (kind == 1) y[u] = b * a.Wcap + ((ri >= 0) ? (ri & (kWinFlag - 1)) : 0);
          else y[u] = b * a.N + ((ri >= 0) ? ri : 0);
        }
      }
      const unsigned tma_mask = __ballot_sync(0xffffffffu, lane < CK / 4 && kind != 2);
      const unsigned mixed_mask = __ballot_sync(0xffffffffu, lane < CK / 4 && kind == 2);
      if (lane == 0) tc::mbar_expect_tx(&kv_full[buf], __popc(tma_mask) * NREG * 4 * 128);
      __syncwarp();
      if (lane < CK / 4 && kind != 2) {
        const CUtensorMap* map = kind == 1 ? &winmap : &kvmap;
#pragma unroll
        for (int rg = 0; rg < NREG; ++rg)
          tc::tma_gather4(kvs + rg * KV_REGION + (buf * CK + lane * 4) * 128, map, rg * 64, y[0], y[1], y[2], y[3],
                          &kv_full[buf]);
      }
      // mixed groups: 4 rows x 64 chunks of 16 bytes each, spread over the warp
      for (unsigned m = mixed_mask; m != 0; m &= m - 1) {
        const int g = __ffs(m) - 1;
        for (int i = lane; i < 4 * 64; i += 32) {
          const int r = g * 4 + (i >> 6), cc = i & 63;
          const int ri = ms.rowidx[c * CK + r];
          const unsigned char* p = nullptr;
          if (ri >= 0)
            p = (ri & kWinFlag) ? winb + (static_cast<size_t>(b) * a.Wcap + (ri & (kWinFlag - 1))) * (D * 2)
                                : kvb + (static_cast<size_t>(b) * a.N + ri) * (D * 2);
          unsigned char* dst = kvs + (cc >> 3) * KV_REGION + (buf * CK + r) * 128 + (((cc & 7) ^ (r & 7)) << 4);
          cp_async16(dst, p ? p + cc * 16 : dummy, p != nullptr);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&kv_full[buf]);                      // 32 arrivals + the gathers' bytes
    };
    // chunk c is published as soon as its rows land: its buffer only waits for the PV of chunk
    // c - 2, never for a later step of the pipeline (the MMA warp issues S(c) before PV(c - 1)).
    // A timed-out wait still reaches the arrival (no thread leaves alone).
    for (int c = 0; c < nch; ++c) {
      if (c > 0 && !tc::mbar_wait(&kv_empty[c & 1], ((c >> 1) & 1) ^ 1, ms.abort_flag)) fail(21);
      issue(c);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer (lane 0 only)
    if (lane == 0) {
      constexpr uint32_t idS = tc::umma_idesc_bf16(128, HG, 0, 0);
      constexpr uint32_t idPV = tc::umma_idesc_bf16(128, HG, 1, 0);
      const uint32_t kva = tc::sptr(kvs), qa = tc::sptr(qs), pa = tc::sptr(pts);
      bool issued = false, ok = true;
      if (nch > 0 && !tc::mbar_wait(q_ready, 0, ms.abort_flag)) { fail(22); ok = false; }
      auto issue_s = [&](int c) -> bool {
        const int buf = c & 1;
        if (!tc::mbar_wait(&kv_full[buf], (c >> 1) & 1, ms.abort_flag)) return false;
        tc::tc_fence_after();
#pragma unroll 8
        for (int k = 0; k < D / 16; ++k) {
          const int r = k >> 2, off = (k & 3) * 32;
          const uint64_t ad = tc::umma_desc_sw128(kva + r * KV_REGION + buf * CK * 128 + off);
          const uint64_t bd = tc::umma_desc_sw128(qa + r * Q_REGION + off);
          tc::umma_bf16(tmem + buf * HG, ad, bd, idS, k > 0 ? 1u : 0u);
        }
        tc::umma_commit(&s_full[buf]);
        issued = true;
        return true;
      };
      if (ok && nch > 0 && !issue_s(0)) { fail(23); ok = false; }
      for (int c = 0; ok && c < nch; ++c) {
        const int buf = c & 1;
        if (c + 1 < nch && !issue_s(c + 1)) { fail(23); break; }
        if (!tc::mbar_wait(&p_full[buf], (c >> 1) & 1, ms.abort_flag)) { fail(24); break; }
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
        tc::umma_commit(&pv_done[buf]);
      }
      if (issued) {
        tc::umma_commit(drain);
        if (!tc::mbar_wait(drain, 0, nullptr)) report_error(a.status, CSA_ERR_TIMEOUT, 25);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps 0-7
    // quarter: TMEM lanes 32*quarter..; hh: which 32 heads (columns) this warp handles
    const int quarter = warp & 3, hh = warp >> 2;
    const bool softmax_warp = quarter < 2;                 // rows 0..63 of a chunk live in lanes 0..63
    const int sw = quarter * 2 + hh;                       // 0..3 among the softmax warps
    if (!tc::mbar_wait(q_loaded, 0, ms.abort_flag)) fail(20);
    if (a.q_norm_rope) norm_q_inplace<8>(a, warp * 8, ms.rope, qs, lane);
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(q_ready);

    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      if (softmax_warp) {
        const int j = quarter * 32 + lane;                 // row of the chunk = TMEM lane
        bool good = tc::mbar_wait(&s_full[buf], (c >> 1) & 1, ms.abort_flag);
        good = good && tc::mbar_wait(&kv_full[buf], (c >> 1) & 1, ms.abort_flag);
        if (!good) fail(26);
        float z[32];
        if (good) {
          tc::tc_fence_after();
          tc::tmem_ld32_wait(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * HG + hh * 32, z);
        }
        const bool valid = good && ms.rowidx[c * CK + j] >= 0;
        bool over = false;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          z[i] = valid ? z[i] * sl2 : -INFINITY;
          over |= z[i] > ms.Rref[hh * 32 + i] + kRescaleLog2;   // also true for the first valid rows
        }
        const bool wover = __any_sync(0xffffffffu, over);
        if (lane == 0) ms.flags[sw] = wover ? 1 : 0;
        tc::named_bar_sync(3, 128);
        const bool maxpass = (ms.flags[0] | ms.flags[1] | ms.flags[2] | ms.flags[3]) != 0;
        if (maxpass) {
          // exact per-head maximum of this chunk's rows; the reference moves only past 2^8
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = z[i];
          butterfly_max32(v, lane);
          ms.red[quarter * HG + hh * 32 + lane] = v[0];
          tc::named_bar_sync(3, 128);
          if (quarter == 0) {
            const int h = hh * 32 + lane;
            const float cm = fmaxf(ms.red[h], ms.red[HG + h]);
            const float rold = ms.Rref[h];
            float rnew = rold, f = 1.f;
            bool need = false;
            if (cm > -INFINITY) {
              if (rold == -INFINITY) {
                rnew = cm;                                 // first rows of this head: O and l are zero
              } else if (cm > rold + kRescaleLog2) {
                rnew = cm;
                f = exp2f(rold - rnew);
                need = true;
              }
            }
            ms.Rref[h] = rnew;
            ms.Fac[h] = f;
            const bool any = __any_sync(0xffffffffu, need);
            if (lane == 0) ms.flags[4 + hh] = any ? 1 : 0;
          }
          tc::named_bar_sync(3, 128);
        } else if (quarter == 0 && lane < 2) {
          ms.flags[4 + lane] = 0;
        }
        // probabilities against the reference, stored as bf16 P^T (the buffer was last read by
        // the PV of chunk c - 2)
        if (!tc::mbar_wait(&pv_done[buf], ((c >> 1) & 1) ^ 1, ms.abort_flag)) fail(28);
        unsigned char* pt = pts + buf * PT_BYTES;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = hh * 32 + i;
          const float pv = (z[i] == -INFINITY) ? 0.f : exp2f(z[i] - ms.Rref[h]);
          *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + ((((j >> 3) ^ (h & 7))) << 4) + (j & 7) * 2) =
              __float2bfloat16_rn(pv);
        }
        tc::tc_fence_before();
        tc::named_bar_sync(3, 128);                        // P^T of the chunk complete
        if (quarter == 0) {
          // per-head sum of the stored (bf16) probabilities: one thread per head reads its row of P^T
          const int h = hh * 32 + lane;
          const unsigned char* prow = pt + h * 128;
          float sum = 0.f;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 u = *reinterpret_cast<const uint4*>(prow + ((ch ^ (h & 7)) << 4));
            sum += (bf16lo(u.x) + bf16hi(u.x)) + (bf16lo(u.y) + bf16hi(u.y)) +
                   (bf16lo(u.z) + bf16hi(u.z)) + (bf16lo(u.w) + bf16hi(u.w));
          }
          ms.Lsum[h] = ms.Lsum[h] * (maxpass ? ms.Fac[h] : 1.f) + sum;
        }
      }
      tc::named_bar_sync(1, 256);                          // rescale decision visible to all eight warps
      if (ms.flags[4] | ms.flags[5]) {
        // a head's reference maximum moved: O^T columns are rescaled once PV(c-1) is done
        if (!tc::mbar_wait(&pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1, ms.abort_flag)) fail(29);
        tc::tc_fence_after();
        const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
        for (int mt = 0; mt < 4; ++mt) {
          float v[32];
          const uint32_t ta = tmem + lb + 2 * HG + mt * HG + hh * 32;
          tc::tmem_ld32_wait(ta, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= ms.Fac[hh * 32 + i];
          tc::tmem_st32_wait(ta, v);
        }
        tc::tc_fence_before();
      }
      tc::named_bar_sync(1, 256);
      if (softmax_warp) {
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&p_full[buf]);
      }
    }

    // ------------------------------------------------------------ epilogue
    if (nch > 0 && !tc::mbar_wait(&pv_done[(nch - 1) & 1], ((nch - 1) >> 1) & 1, ms.abort_flag)) fail(30);
    tc::tc_fence_after();
    const int Q = a.B * a.Tq;
    float* pml = a.partial + static_cast<size_t>(Q) * a.n_splits * a.H * D;
    if (tid < HG) {
      const int h = tid;
      const float R = ms.Rref[h], l = ms.Lsum[h];
      if (a.n_splits == 1) {
        const float a2 = a.sink[h0 + h] * kLog2e;
        const float M = fmaxf(R, a2);
        const float fo = (R == -INFINITY) ? 0.f : exp2f(R - M);
        const float den = l * fo + exp2f(a2 - M);
        ms.norm[h] = fo / den;
        if (a.lse != nullptr) a.lse[qi * a.H + h0 + h] = (M + log2f(den)) * kLn2;
      } else {
        const size_t ri = (static_cast<size_t>(qi) * a.n_splits + split) * a.H + h0 + h;
        pml[ri * 2 + 0] = R;
        pml[ri * 2 + 1] = l;
      }
    }
    tc::named_bar_sync(1, 256);
    // the accumulator is staged in shared memory that no MMA reads any more (all are complete):
    // bf16 output rows in the query block, fp32 partials in the row buffers; then one coalesced
    // 16-byte copy of the CTA's contiguous 64 heads x 512 dims
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const bool final_out = a.n_splits == 1;
    for (int mt = 0; mt < 4; ++mt) {
      const int dim = mt * 128 + quarter * 32 + lane;
      float v[32];
      if (nch > 0) {
        tc::tmem_ld32_wait(tmem + lb + 2 * HG + mt * HG + hh * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      if (final_out) {
        const bool rot = a.out_unrotate && dim >= D - a.rp.r;
        float2 cssn = make_float2(1.f, 0.f);
        if (rot) cssn = ms.rope[(dim - (D - a.rp.r)) >> 1];
        __nv_bfloat16* ostage = reinterpret_cast<__nv_bfloat16*>(qs);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = hh * 32 + i;
          const float x = v[i] * ms.norm[h];
          const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
          float y = x;
          // rotation by -t on the pair (2j, 2j+1): [x0 c + x1 s, -x0 s + x1 c]
          if (rot) y = (dim & 1) ? (x * cssn.x - partner * cssn.y) : (x * cssn.x + partner * cssn.y);
          ostage[h * D + dim] = __float2bfloat16_rn(y);
        }
      } else {
        float* pstage = reinterpret_cast<float*>(kvs);
#pragma unroll
        for (int i = 0; i < 32; ++i) pstage[(hh * 32 + i) * D + dim] = v[i];
      }
    }
    tc::named_bar_sync(1, 256);
    if (final_out) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (qi * a.H + h0) * static_cast<long long>(D));
      const uint4* src = reinterpret_cast<const uint4*>(qs);
      for (int i = tid; i < HG * D * 2 / 16; i += 256) dst[i] = src[i];
    } else {
      float4* dst = reinterpret_cast<float4*>(a.partial + ((static_cast<size_t>(qi) * a.n_splits + split) * a.H + h0) * D);
      const float4* src = reinterpret_cast<const float4*>(kvs);
      for (int i = tid; i < HG * D / 4; i += 256) dst[i] = src[i];
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == MMA_WARP) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool attend_tc_supported(const AttendArgs& a) {
  const long long staged = (static_cast<long long>(a.split_slots) + CK - 1) / CK * CK;
  return a.d == D && !a.fp8 && (a.H % HG) == 0 && a.rp.r <= 2 * kMaxRopePairs && a.rp.r <= D &&
         staged <= kMaxSlots;
}

cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s, int* launches) {
  const int Q = a.B * a.Tq;
  if (Q == 0) return cudaSuccess;
  // queries as rows of 512 bf16: box of 64 dims x 64 heads, 128-byte swizzle (the MMA layout)
  CUtensorMap qmap;
  const uint64_t dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Q) * a.H};
  const uint32_t box[2] = {64, HG};
  if (!tc::make_tensor_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, 2, dims, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // row gathers: cache rows and window rows, box of 64 dims x 1 row (tile::gather4)
  CUtensorMap kvmap, winmap;
  const uint32_t gbox[2] = {64, 1};
  const uint64_t wdims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.B) * (a.Wcap > 0 ? a.Wcap : 1)};
  if (a.win == nullptr ||
      !tc::make_tensor_map(&winmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.win, 2, wdims, gbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.N > 0) {
    const uint64_t kdims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.B) * a.N};
    if (!tc::make_tensor_map(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kv, 2, kdims, gbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    kvmap = winmap;                                        // never used when there are no entries
  }
  cudaError_t e = cudaFuncSetAttribute(k_attend_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  k_attend_tc<<<dim3(Q, a.H / HG, a.n_splits), NTHREADS, SMEM, s>>>(a, qmap, kvmap, winmap);
  ++*launches;
  e = cudaGetLastError();
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attend_combine(a, s, launches);
}

}  // namespace csa
