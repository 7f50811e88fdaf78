// Shared K=V multi-query attention on the 5th-generation tensor cores, for 512-dim bf16 rows and
// 64 query heads per CTA ("DeepSeek V4 模型技术大全", component table rows Shared K=V MQA,
// query/KV RMSNorm, partial RoPE, attention sink, SWA; the HCA visibility set; the
// reverse-rotation note).  Same slots, splits and partial format as the warp-MMA kernel in
// attend.cu, which keeps the other shapes (d = 128, the FP8 cache).
//
// Per CTA: one query, 64 heads, one split of the slot range, 64 rows per chunk.
//   S^T = K q_hat^T   tcgen05.mma M = 128 (the chunk's 64 rows are TMEM lanes 0..63), N = 64
//                     heads, K = 512, fp32 in TMEM, two buffers
//   softmax           four warps, one thread per (row, 32 heads): per-head chunk maximum by a
//                     warp butterfly, a per-head reference maximum that moves only when a chunk
//                     exceeds it by more than 2^8 (the O accumulator is then rescaled in TMEM);
//                     p = exp2(z - ref) rounded to bf16 into P^T (K-major, 128-byte swizzle); the
//                     row sums add the rounded values, so the normaliser uses exactly the
//                     probabilities of the PV product
//   O^T += V^T P^T    M = 128 dims (4 tiles), N = 64 heads, K = 64 rows; V^T is the chunk's rows
//                     read through an MN-major descriptor (K = V)
// Rows are gathered with cp.async by all 256 threads straight into the 128-byte swizzled operand
// layout, two chunk buffers, so chunk c+1's gather overlaps chunk c's products.  One thread
// issues the MMAs.  Every wait is bounded (CSA_ERR_TIMEOUT in the status word, never a hang).
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
constexpr int NT = 256;
constexpr float kRescaleLog2 = 8.f;           // a head's reference maximum moves only past 2^8
constexpr uint64_t kWaitNs = 200000000ull;    // 0.2 s: every wait here normally ends in microseconds

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

constexpr int kBarsOff = 3584 + 4 * 4;        // after rowptr, rope, ref/lsum/fac/fin, red, red2, flags
static_assert(kBarsOff % 8 == 0 && kBarsOff + 5 * 8 + 8 <= MISC_BYTES, "misc layout");

struct Misc {
  const unsigned char** rowptr;   // [2][CK]
  float2* rope;                   // [kMaxRopePairs]
  float* ref;                     // [HG] reference maximum (log2 domain)
  float* lsum;                    // [HG] sum of the rounded exp2(z - ref)
  float* fac;                     // [HG]
  float* fin;                     // [HG] epilogue factor
  float* red;                     // [2][HG]
  float* red2;                    // [2][HG]
  int* flags;                     // [4]
  uint64_t* bars;                 // [5]
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

__device__ __forceinline__ Misc carve(unsigned char* base) {
  Misc m;
  m.rowptr = reinterpret_cast<const unsigned char**>(base);                  // 1024 B
  m.rope = reinterpret_cast<float2*>(base + 1024);                           // 512 B
  m.ref = reinterpret_cast<float*>(base + 1536);
  m.lsum = m.ref + HG;
  m.fac = m.lsum + HG;
  m.fin = m.fac + HG;
  m.red = m.fin + HG;                                                        // base + 2560
  m.red2 = m.red + 2 * HG;                                                   // base + 3072
  m.flags = reinterpret_cast<int*>(m.red2 + 2 * HG);                         // base + 3584
  m.bars = reinterpret_cast<uint64_t*>(base + kBarsOff);
  m.tmem_slot = reinterpret_cast<uint32_t*>(base + kBarsOff + 5 * 8);
  m.abort_flag = reinterpret_cast<volatile int*>(base + kBarsOff + 5 * 8 + 4);
  return m;
}

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
  const Misc ms = carve(sm + OFF_MISC);
  uint64_t* s_full = ms.bars;         // [2] commit after S of the chunk in that buffer
  uint64_t* o_full = ms.bars + 2;     // [2] commit after PV of the chunk in that buffer
  uint64_t* drain = ms.bars + 4;
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
  const unsigned char* kvb = static_cast<const unsigned char*>(a.kv);
  const unsigned char* winb = static_cast<const unsigned char*>(a.win);
  const unsigned char* dummy = static_cast<const unsigned char*>(a.q);   // source of zero-size copies

  if ((tc::sptr(sm) & 1023u) != 0u) {               // the swizzled operands need 1024-byte alignment
    if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2000);
    return;
  }
  if (tid == 0) {
    // a wait of this call already gave up: later CTAs do no work instead of waiting in turn (the
    // decision is thread 0's, shared through shared memory, so the whole CTA takes it)
    ms.flags[1] = (*reinterpret_cast<volatile int32_t*>(a.status) == CSA_ERR_TIMEOUT) ? 1 : 0;
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&o_full[i], 1);
    }
    tc::mbar_init(drain, 1);
    *ms.abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(ms.tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid < a.rp.r / 2) {
    float cs, sn;
    rope_cos_sin(static_cast<double>(t), a.rp.inv_freq[tid], cs, sn);
    ms.rope[tid] = make_float2(cs, sn);
  }
  if (tid < HG) {
    ms.ref[tid] = -INFINITY;
    ms.lsum[tid] = 0.f;
  }
  if (tid == 0 || tid == 2 || tid == 3) ms.flags[tid] = 0;

  // row pointers of chunk c into rowptr[buf]: the idx value is loaded by load_raw (the only global
  // read) and turned into a pointer by set_ptr; threads 0..63 own one row each
  auto load_raw = [&](int c) -> int {
    const int s = s_begin + c * CK + (tid & (CK - 1));
    return (s < s_end && s < Kq && a.idx != nullptr) ? a.idx[qi * a.k + s] : 0;
  };
  auto set_ptr = [&](int c, int buf, int raw) {
    const int j = tid & (CK - 1);
    const int s = s_begin + c * CK + j;
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
    ms.rowptr[buf * CK + j] = p;
  };
  // cp.async of the chunk's 64 rows into buffer `buf`, 128-byte swizzled: 16 copies per thread
  auto gather = [&](int buf) {
#pragma unroll 4
    for (int i = tid; i < CK * 64; i += NT) {
      const int j = i >> 6, cc = i & 63;
      const unsigned char* p = ms.rowptr[buf * CK + j];
      const int row = buf * CK + j;
      unsigned char* dst = kvs + (cc >> 3) * KV_REGION + row * 128 + (((cc & 7) ^ (row & 7)) << 4);
      cp_async16(dst, p ? p + cc * 16 : dummy, p != nullptr);
    }
    cp_async_commit();
  };
  auto fail = [&](int where) {
    *ms.abort_flag = 1;
    report_error(a.status, CSA_ERR_TIMEOUT, where);
  };

  // ---------------- prologue: first two chunks' rows, the query block, then S of chunk 0
  {
    const int raw = (tid < CK) ? load_raw(0) : (tid < 2 * CK && nch > 1 ? load_raw(1) : 0);
    if (tid < CK && nch > 0) set_ptr(0, 0, raw);
    else if (tid >= CK && tid < 2 * CK && nch > 1) set_ptr(1, 1, raw);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *ms.tmem_slot;
  bool issued = false;
  if (ms.flags[1] == 0) {
  if (nch > 0) gather(0);

  // q_hat = RoPE_t(RMSNorm(q)) as bf16 into the K-major swizzled B operand of S: warp w prepares
  // heads 8w..8w+7; lane L owns dims 16L..16L+15 (two 16-byte chunks of region L/4)
  {
    const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(a.q);
    const int region = lane >> 2, ch0 = (lane & 3) * 2;
#pragma unroll 2
    for (int i = 0; i < HG / 8; ++i) {
      const int hl = warp * (HG / 8) + i;
      const uint4* src = reinterpret_cast<const uint4*>(qsrc + ((qi * a.H) + h0 + hl) * static_cast<long long>(D) + lane * 16);
      const uint4 u0 = src[0], u1 = src[1];
      float v[16] = {bf16lo(u0.x), bf16hi(u0.x), bf16lo(u0.y), bf16hi(u0.y), bf16lo(u0.z), bf16hi(u0.z),
                     bf16lo(u0.w), bf16hi(u0.w), bf16lo(u1.x), bf16hi(u1.x), bf16lo(u1.y), bf16hi(u1.y),
                     bf16lo(u1.z), bf16hi(u1.z), bf16lo(u1.w), bf16hi(u1.w)};
      if (a.q_norm_rope) {
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
            const float2 cssn = ms.rope[(ch - (D - a.rp.r)) >> 1];
            const float x0 = v[c], x1 = v[c + 1];
            v[c] = x0 * cssn.x - x1 * cssn.y;
            v[c + 1] = x0 * cssn.y + x1 * cssn.x;
          }
        }
      }
      unsigned char* row = qs + region * Q_REGION + hl * 128;
      *reinterpret_cast<uint4*>(row + ((ch0 ^ (hl & 7)) << 4)) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      *reinterpret_cast<uint4*>(row + (((ch0 + 1) ^ (hl & 7)) << 4)) =
          make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                     pack_bf16x2(v[14], v[15]));
    }
  }
  if (nch > 1) gather(1);
  if (nch > 1) cp_async_wait<1>(); else cp_async_wait<0>();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  constexpr uint32_t idS = tc::umma_idesc_bf16(128, HG, 0, 0);
  constexpr uint32_t idPV = tc::umma_idesc_bf16(128, HG, 1, 0);
  const uint32_t kva = tc::sptr(kvs), qa = tc::sptr(qs), pa = tc::sptr(pts);
  auto issue_s = [&](int c) {                           // thread 0
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
  auto issue_pv = [&](int c) {                          // thread 0
    const int buf = c & 1;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
      for (int k = 0; k < CK / 16; ++k) {
        const uint64_t ad = tc::umma_desc_sw128_mn(kva + (2 * mt) * KV_REGION + (buf * CK + 16 * k) * 128, KV_REGION, 1024);
        const uint64_t bd = tc::umma_desc_sw128(pa + buf * PT_BYTES + k * 32);
        tc::umma_bf16(tmem + 2 * HG + mt * HG, ad, bd, idPV, (c > 0 || k > 0) ? 1u : 0u);
      }
    }
    tc::umma_commit(&o_full[buf]);
    issued = true;
  };
  if (tid == 0 && nch > 0 && !*ms.abort_flag) issue_s(0);

  const bool smx = (warp & 3) < 2;                      // softmax warps: rows 0..63 = TMEM lanes 0..63
  const int quarter = warp & 3, hh = warp >> 2;         // softmax: rows 32*quarter + lane, heads 32*hh + i
  for (int c = 0; c < nch; ++c) {
    const int buf = c & 1;
    const uint32_t ph = static_cast<uint32_t>((c >> 1) & 1);
    const int raw_next = (tid < CK && c + 2 < nch) ? load_raw(c + 2) : 0;   // lands during this chunk
    // ---- softmax of chunk c
    const bool got = tc::mbar_wait(&s_full[buf], ph, ms.abort_flag, kWaitNs);
    if (!__all_sync(0xffffffffu, got) && lane == 0) fail(31);
    tc::tc_fence_after();
    float z[32];
    const int j = quarter * 32 + lane;
    if (smx) {
      tc::tmem_ld32_wait(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * HG + hh * 32, z);
      const bool valid = ms.rowptr[buf * CK + j] != nullptr;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        z[i] = valid ? z[i] * sl2 : -INFINITY;
        v[i] = z[i];
      }
      butterfly32<true>(v, lane);
      ms.red[quarter * HG + hh * 32 + lane] = v[0];
    }
    __syncthreads();
    if (tid < HG) {
      const float cm = fmaxf(ms.red[tid], ms.red[HG + tid]);
      const float rold = ms.ref[tid];
      float rnew = rold, f = 1.f;
      if (cm > rold + kRescaleLog2 || (rold == -INFINITY && cm > -INFINITY)) {
        rnew = cm;
        f = (rold == -INFINITY) ? 0.f : exp2f(rold - rnew);
        if (c > 0 && rold > -INFINITY) ms.flags[0] = 1;           // O holds terms scaled by rold
      }
      ms.ref[tid] = rnew;
      ms.fac[tid] = f;
      ms.lsum[tid] *= f;
    }
    __syncthreads();
    if (ms.flags[0]) {
      // rescale O^T columns of the moved heads: wait until the PV of chunk c-1 has landed
      const bool g2 = tc::mbar_wait(&o_full[(c - 1) & 1], static_cast<uint32_t>(((c - 1) >> 1) & 1), ms.abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, g2) && lane == 0) fail(32);
      tc::tc_fence_after();
#pragma unroll 1
      for (int mi = 0; mi < 2; ++mi) {
        const int mt = (warp >> 2) + 2 * mi;
        const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 2 * HG + mt * HG;
        float o[64];
        tc::tmem_ld64_wait(ta, o);
#pragma unroll
        for (int h = 0; h < 64; ++h) o[h] *= ms.fac[h];
        tc::tmem_st64_wait(ta, o);
      }
      tc::tc_fence_before();
      __syncthreads();
      tc::tc_fence_after();
      if (tid == 0) ms.flags[0] = 0;
    }
    if (smx) {
      // p = exp2(z - ref) rounded to bf16 into P^T[h][j]; row sums of the rounded values
      unsigned char* pt = pts + buf * PT_BYTES;
      float ps[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int h = hh * 32 + i;
        const float r = ms.ref[h];
        const float p = exp2f(z[i] - (r == -INFINITY ? 0.f : r));
        const __nv_bfloat16 pb = __float2bfloat16_rn(p);
        ps[i] = __bfloat162float(pb);
        *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + ((((j >> 3) ^ (h & 7))) << 4) + (j & 7) * 2) = pb;
      }
      butterfly32<false>(ps, lane);
      ms.red2[quarter * HG + hh * 32 + lane] = ps[0];
    }
    tc::fence_proxy_async_smem();
    if (c + 1 < nch) cp_async_wait<0>();                // chunk c+1's rows (this thread's copies)
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid < HG) ms.lsum[tid] += ms.red2[tid] + ms.red2[HG + tid];
    if (tid == 0 && !*ms.abort_flag) {
      if (c + 1 < nch) issue_s(c + 1);
      issue_pv(c);
    }
    // ---- rows of chunk c+2 into this buffer once the PV of chunk c has read it
    if (c + 2 < nch) {
      const bool g3 = tc::mbar_wait(&o_full[buf], ph, ms.abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, g3) && lane == 0) fail(33);
      if (tid < CK) set_ptr(c + 2, buf, raw_next);
      __syncthreads();
      gather(buf);
    }
  }

  // ---------------- epilogue: normaliser with the sink, O^T out of TMEM
  const bool have = nch > 0;
  if (have) {
    const int last = nch - 1;
    const bool g4 = tc::mbar_wait(&o_full[last & 1], static_cast<uint32_t>((last >> 1) & 1), ms.abort_flag, kWaitNs);
    if (!__all_sync(0xffffffffu, g4) && lane == 0) fail(34);
    tc::tc_fence_after();
  }
  const int Q = a.B * a.Tq;
  if (tid < HG) {
    const int h = h0 + tid;
    const float r = ms.ref[tid];
    if (a.n_splits == 1) {
      const float a2 = a.sink[h] * kLog2e;
      const float M = fmaxf(r, a2);
      const float f = (r == -INFINITY) ? 0.f : exp2f(r - M);
      const float L = ms.lsum[tid] * f + exp2f(a2 - M);
      ms.fin[tid] = f / L;
      if (a.lse != nullptr) a.lse[qi * a.H + h] = (M + log2f(L)) * kLn2;
    } else {
      float* pml = a.partial + static_cast<size_t>(Q) * a.n_splits * a.H * D;
      const size_t rowi = (static_cast<size_t>(qi) * a.n_splits + split) * a.H + h;
      pml[rowi * 2 + 0] = r;
      pml[rowi * 2 + 1] = ms.lsum[tid];
    }
  }
  __syncthreads();
#pragma unroll 1
  for (int mi = 0; mi < 2; ++mi) {
    const int mt = (warp >> 2) + 2 * mi;
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
      const bool rot = a.out_unrotate && d >= D - a.rp.r;          // warp-uniform (32-dim groups)
      float cs = 1.f, sn = 0.f;
      if (rot) {                                                     // rotation by -t
        const float2 cssn = ms.rope[(d - (D - a.rp.r)) >> 1];
        cs = cssn.x;
        sn = -cssn.y;
      }
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        float x = o[h] * ms.fin[h];
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

  }  // work of a CTA whose call had not timed out

  // ---------------- teardown: every MMA complete before tensor memory is released
  if (tid == 0 && issued) {
    tc::umma_commit(drain);
    if (!tc::mbar_wait(drain, 0, nullptr, kWaitNs)) report_error(a.status, CSA_ERR_TIMEOUT, 35);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
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
