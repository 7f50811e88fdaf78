// Shared K=V multi-query attention on the 5th-generation tensor cores for 512-dim bf16 rows, 64
// query heads per CTA ("DeepSeek V4 模型技术大全", component table rows Shared K=V MQA, query/KV
// RMSNorm, partial RoPE, attention sink, SWA; the HCA visibility set; the reverse-rotation note).
// Same slots, splits and partial format as the warp-MMA kernel in attend.cu, which keeps the other
// shapes (d = 128, the FP8 cache, head counts that are not a multiple of 64, other RoPE widths).
//
// Exact query path.  q_hat = RoPE_t(RMSNorm(q)) = inv * RoPE_t(q) with inv = 1/sqrt(mean(q^2)+eps),
// so q_hat . K = inv * (q[0, d-r) . K[0, d-r) + RoPE_t(q)[d-r, d) . K[d-r, d)).  The unrotated dims
// enter the product as the query's own bf16 bits (exact), the r rotated dims as a bf16 hi + lo pair
// (about 16 significant bits), and inv multiplies the fp32 logit.  No rounding of the normalised
// query stands between the inputs and the logits beyond the fp32 sums of the tensor cores.
//
// A CTA is persistent over work items (query, group of 64 heads, split of the slot range) and is
// warp-specialised around two 64-row chunk buffers:
//   loader warps (7)       row pointers from the idx row, then cp.async of the chunk's 4096 16-byte
//                          pieces straight into the 128-byte swizzled operand layout.  Gathering
//                          scattered rows is bound by how many warps issue copies (one warp needs
//                          ~9K cycles per 64 KB, sixteen ~2.3K), hence seven warps
//   MMA warp (1 thread)    S^T(c) = K q'^T   M = 128 (the chunk's 64 rows are TMEM lanes 0..63),
//                          N = 64 heads, K = 512 (+ 64 for the lo half of the rotated dims), fp32 in
//                          TMEM, two buffers
//                          O^T += V^T P^T(c) M = 128 dims (4 tiles), N = 64 heads, K = 64 rows;
//                          V^T is the chunk's rows through an MN-major descriptor
//                          S^T and PV are issued greedily in chunk order, each as soon as its inputs
//                          are ready, so one buffer's gather never holds back the other's products
//   softmax warps (8)      one thread per (row, 16 heads): per-head chunk maxima by a butterfly
//                          over the warp and a pair exchange; a per-head reference maximum that
//                          moves only when a chunk exceeds it by more than 2^8; p = exp2(z - ref)
//                          rounded to bf16 into P^T (K-major, swizzled); running sums of the
//                          unrounded p per thread
//   correction warps (4)   the query block of the next item (a TMA load of the raw q rows, inv per
//                          head, the rotated dims' hi / lo), the rescale of O^T in TMEM when a
//                          reference moved, and the epilogue (sink, normaliser, reverse rotation,
//                          bf16 output or split partials)
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
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: every wait here normally ends in microseconds

constexpr int QREG = HG * 128;                // one 64-dim region of the query block
constexpr int KVREG = 2 * CK * 128;           // one 64-dim region of both chunk buffers
constexpr int PTB = HG * 128;                 // P^T of one chunk: 64 heads x 64 rows, bf16
constexpr int OFF_Q = 0;                      // regions 0..7: the raw query (rotated dims: hi)
constexpr int OFF_QLO = OFF_Q + NREG * QREG;  // region 8: lo half of the rotated dims
constexpr int OFF_KV = OFF_QLO + QREG;
constexpr int OFF_PT = OFF_KV + NREG * KVREG; // also absorbs the M = 128 read of buffer 1 past region 7
constexpr int OFF_MISC = OFF_PT + 2 * PTB;
constexpr int M_ROWPTR = 0;                   // [2][CK] row pointers
constexpr int M_ROPE = 1024;                  // [2][32] (cos, sin) of t * inv_freq, by item parity
constexpr int M_CSCALE = M_ROPE + 512;        // [2][HG] log2-domain logit factor per head (scale * inv)
constexpr int M_REF = M_CSCALE + 512;         // [HG] reference maximum (log2 domain)
constexpr int M_FAC = M_REF + 256;            // [2][HG] factor of chunk buffer b
constexpr int M_RED = M_FAC + 512;            // [2][HG] pair exchange of the two row quarters
constexpr int M_FREF = M_RED + 512;           // [2][HG] final reference per item parity
constexpr int M_FL = M_FREF + 512;            // [2][HG] final sums per item parity
constexpr int M_EFAC = M_FL + 512;            // [HG] epilogue factor
constexpr int M_FLAG = M_EFAC + 256;          // [2][4] rescale needed (buffer, head quarter)
constexpr int M_BARS = M_FLAG + 32;
// Barriers used once per item come in pairs by item parity where a waiter could otherwise see
// two completions before it looks (items of one chunk let the producer run an item ahead).
enum {
  B_QTMA = 0, B_QREADY, B_QFREE = B_QREADY + 2, B_KVFULL, B_KVEMPTY = B_KVFULL + 2, B_SFULL = B_KVEMPTY + 2,
  B_PFULL = B_SFULL + 2, B_CDONE = B_PFULL + 2, B_OREADY = B_CDONE + 2, B_OFREE, B_SMDONE = B_OFREE + 1,
  B_DRAIN = B_SMDONE + 2, NBARS
};
constexpr int M_TMEM = M_BARS + NBARS * 8;
constexpr int M_ABORT = M_TMEM + 4;
constexpr int M_PML = (M_ABORT + 4 + 15) & ~15;   // [HG] (m, l) of this split (cluster merge)
constexpr int MISC_BYTES = M_PML + HG * 8;
constexpr int SMEM = 1024 + OFF_MISC + MISC_BYTES;
static_assert(M_BARS % 8 == 0 && M_ABORT + 4 <= MISC_BYTES, "misc layout");
static_assert(SMEM <= 232448, "shared memory budget");
constexpr int TMEM_COLS = 512;                // S^T at columns 0 / 64, O^T tiles at 128 + 64 mt

// warp roles (20 warps).  TMEM lane quarter = warp % 4.  softmax: warps 0,1,4,5,8,9,12,13 (lane
// quarters 0 and 1 = the chunk's 64 rows; head quarter = warp / 4); loaders: 2,3,6,7,10,11,14;
// MMA: 15; correction: 16..19 (lane quarters 0..3 = the dims of an O^T tile)
constexpr int NWARPS = 20;
constexpr int NT = NWARPS * 32;
constexpr int kMmaWarp = 15;
constexpr int kNLoad = 7 * 32;
constexpr int BAR_SOFTMAX = 1, BAR_CORR = 2, BAR_LOAD = 3;
__device__ __forceinline__ bool is_softmax_warp(int w) { return w < 16 && (w & 3) < 2; }
__device__ __forceinline__ bool is_loader_warp(int w) { return w < 15 && (w & 3) >= 2; }
__device__ __forceinline__ int loader_index(int w) { return (w >> 2) * 2 + (w & 1); }   // 0..6

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Four floats at the same shared-memory offset as p (16-byte aligned) in CTA `rank` of the cluster.
__device__ __forceinline__ float4 ld_peer4f(const float* p, uint32_t rank) {
  const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(ra));
  return v;
}
// Two floats at the same shared-memory offset as p (8-byte aligned) in CTA `rank` of the cluster.
__device__ __forceinline__ float2 ld_peer2(const float* p, uint32_t rank) {
  const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(ra));
  return v;
}

// Butterfly over 16 values per lane and the 32 lanes: afterwards v[0] of lane L (and of lane L^1)
// holds the reduction over all 32 lanes of value (L >> 1) & 15 (max when MAX, else sum).
template <bool MAX>
__device__ __forceinline__ void butterfly16(float* v, int lane) {
#pragma unroll
  for (int o = 16, nc = 16; o >= 2; o >>= 1, nc >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < nc / 2) {
        const float send = up ? v[i] : v[i + nc / 2];
        const float keep = up ? v[i + nc / 2] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
      }
    }
  }
  const float r = __shfl_xor_sync(0xffffffffu, v[0], 1);
  v[0] = MAX ? fmaxf(v[0], r) : v[0] + r;
}

struct Item {
  long long qi;
  int h0, split, t, b, Kq, s_begin, s_end, nch;
};

__device__ __forceinline__ Item item_at(const AttendArgs& a, long long it) {
  const long long per_q = static_cast<long long>(a.H / HG) * a.n_splits;
  Item r;
  r.qi = it / per_q;
  const int rem = static_cast<int>(it - r.qi * per_q);
  r.h0 = (rem / a.n_splits) * HG;
  r.split = rem % a.n_splits;
  r.b = static_cast<int>(r.qi / a.Tq);
  r.t = a.q_pos[r.qi];
  const int nvis = n_visible(r.t, a.m, a.N);
  r.Kq = (a.idx == nullptr) ? nvis : a.k;
  const int nslots = r.Kq + a.window;
  r.s_begin = r.split * a.split_slots;
  r.s_end = min(nslots, r.s_begin + a.split_slots);
  r.nch = r.s_end > r.s_begin ? (r.s_end - r.s_begin + CK - 1) / CK : 0;
  return r;
}

// The next item of this CTA after `it` that has rows (-1 if none).
__device__ __forceinline__ long long next_with_rows(const AttendArgs& a, long long it, long long items, Item& out) {
  for (long long j = it + gridDim.x; j < items; j += gridDim.x) {
    const Item r = item_at(a, j);
    if (r.nch > 0) {
      out = r;
      return j;
    }
  }
  return -1;
}

// Walks the chunks of this CTA's items with rows, in order: the item, its count n among items with
// rows, the chunk c within the item and the global chunk index g.
struct Cursor {
  long long it, n, g;
  Item I;
  int c;
  __device__ __forceinline__ void start(const AttendArgs& a, long long items) {
    it = next_with_rows(a, static_cast<long long>(blockIdx.x) - gridDim.x, items, I);
    n = 0;
    g = 0;
    c = 0;
  }
  __device__ __forceinline__ bool valid() const { return it >= 0; }
  __device__ __forceinline__ void advance(const AttendArgs& a, long long items) {
    ++g;
    if (++c < I.nch) return;
    c = 0;
    ++n;
    it = next_with_rows(a, it, items, I);
  }
};

__global__ void __launch_bounds__(NT, 1) k_attend_tc(const AttendArgs a, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (tc::sptr(smem_raw) & 1023u)) & 1023u);
  unsigned char* qs = sm + OFF_Q;
  unsigned char* kvs = sm + OFF_KV;
  unsigned char* pts = sm + OFF_PT;
  unsigned char* misc = sm + OFF_MISC;
  const unsigned char** rowptr = reinterpret_cast<const unsigned char**>(misc + M_ROWPTR);
  float2* rope = reinterpret_cast<float2*>(misc + M_ROPE);
  float* cscale = reinterpret_cast<float*>(misc + M_CSCALE);
  float* ref = reinterpret_cast<float*>(misc + M_REF);
  float* facb = reinterpret_cast<float*>(misc + M_FAC);
  float* red = reinterpret_cast<float*>(misc + M_RED);
  float* fref = reinterpret_cast<float*>(misc + M_FREF);
  float* fl = reinterpret_cast<float*>(misc + M_FL);
  float* efac = reinterpret_cast<float*>(misc + M_EFAC);
  volatile int* flag = reinterpret_cast<volatile int*>(misc + M_FLAG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + M_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + M_ABORT);
  grid_dep_wait();
  grid_dep_launch();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the swizzled operands need 1024-byte alignment; a CTA without it does no work (it still
  // reaches every block and cluster barrier, so no peer waits on it)
  const bool aligned = (tc::sptr(sm) & 1023u) == 0u;
  const long long items = aligned ? static_cast<long long>(a.B) * a.Tq * (a.H / HG) * a.n_splits : 0;
  const float sl2 = a.scale * kLog2e;
  const int n_lo = (a.q_norm_rope && a.rp.r > 0) ? 1 : 0;   // the rotated dims are region 7 (r = 64)

  if (!aligned && tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2000);
  if (tid == 0) {
    // a wait of this call already gave up: this CTA does no work instead of waiting in turn
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(a.status) == CSA_ERR_TIMEOUT) ? 1 : 0;
    for (int i = 0; i < NBARS; ++i) tc::mbar_init(&bars[i], i == B_OFREE ? 4u : 1u);
    tc::fence_barrier_init();
    tc::prefetch_tensormap(&qmap);
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid < HG) ref[tid] = -INFINITY;
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&](int where) {
    *abort_flag = 1;
    report_error(a.status, CSA_ERR_TIMEOUT, where);
  };
  auto wait = [&](int bi, long long use, int where) {   // the phase of the use-th completion
    const bool ok = tc::mbar_wait(&bars[bi], static_cast<uint32_t>(use & 1), abort_flag, kWaitNs);
    if (!ok) fail(where);
    return ok;
  };

  if (is_softmax_warp(warp)) {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 1;                        // rows 32 * quarter + lane
    const int hq = warp >> 2;                            // heads 16 * hq + i
    const int j = quarter * 32 + lane;
    const int sid = quarter * 32 + hq * 64 + lane;       // 0..255 within the softmax group
    float ps[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ps[i] = 0.f;
    Cursor cur;
    cur.start(a, items);
    while (cur.valid()) {
      const int par = static_cast<int>(cur.n & 1);
      const int c = cur.c;
      const long long g = cur.g;
      if (c == 0) wait(B_QREADY + par, cur.n >> 1, 60);   // this item's logit factors
      const int buf = static_cast<int>(g & 1);
      wait(B_SFULL + buf, g >> 1, 61);
      wait(B_KVFULL + buf, g >> 1, 62);                  // the loaders' row pointers of this chunk
      tc::tc_fence_after();
      float z[16], rr[16];
      tc::tmem_ld16_wait(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * HG + hq * 16, z);
      const bool valid = rowptr[buf * CK + j] != nullptr;
      {
        const float4* cs4 = reinterpret_cast<const float4*>(cscale + par * HG + hq * 16);
        const float4* rf4 = reinterpret_cast<const float4*>(ref + hq * 16);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 cv = cs4[q4], rv = rf4[q4];
          z[4 * q4 + 0] = valid ? z[4 * q4 + 0] * cv.x : -INFINITY;
          z[4 * q4 + 1] = valid ? z[4 * q4 + 1] * cv.y : -INFINITY;
          z[4 * q4 + 2] = valid ? z[4 * q4 + 2] * cv.z : -INFINITY;
          z[4 * q4 + 3] = valid ? z[4 * q4 + 3] * cv.w : -INFINITY;
          rr[4 * q4 + 0] = rv.x;
          rr[4 * q4 + 1] = rv.y;
          rr[4 * q4 + 2] = rv.z;
          rr[4 * q4 + 3] = rv.w;
        }
      }
      // Fast path: every logit of the chunk stays within 2^8 of its head's reference, so the
      // reference does not move (factor 1) and no per-head maximum is needed.  The first chunk of
      // an item, or any logit above the band, takes the exact path for the whole chunk.
      bool over = c == 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) over |= z[i] > rr[i] + kRescaleLog2;
      const bool slow = tc::named_bar_or(BAR_SOFTMAX, 256, over);
      float ff[16];
      if (slow) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = z[i];
        butterfly16<true>(v, lane);
        if ((lane & 1) == 0) red[quarter * HG + hq * 16 + (lane >> 1)] = v[0];
        tc::named_bar_sync(BAR_SOFTMAX, 256);
        if (quarter == 0) {                              // even lanes own a head each
          const int h = hq * 16 + (lane >> 1);
          bool need = false;
          if ((lane & 1) == 0) {
            const float cm = fmaxf(red[h], red[HG + h]);
            const float rold = c == 0 ? -INFINITY : ref[h];   // a new item starts from -inf
            float f = 1.f;
            if (cm > rold + kRescaleLog2 || (rold == -INFINITY && cm > -INFINITY)) {
              f = (rold == -INFINITY) ? 0.f : exp2f(rold - cm);
              need = c > 0 && rold > -INFINITY;          // O^T holds terms scaled by rold
              ref[h] = cm;
            } else if (c == 0) {
              ref[h] = rold;
            }
            facb[buf * HG + h] = f;
          }
          const bool any = __any_sync(0xffffffffu, need);
          if (lane == 0) flag[buf * 4 + hq] = any ? 1 : 0;
        }
        tc::named_bar_sync(BAR_SOFTMAX, 256);
        const float4* rf4 = reinterpret_cast<const float4*>(ref + hq * 16);
        const float4* fc4 = reinterpret_cast<const float4*>(facb + buf * HG + hq * 16);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 rv = rf4[q4], fv = fc4[q4];
          rr[4 * q4 + 0] = rv.x; rr[4 * q4 + 1] = rv.y; rr[4 * q4 + 2] = rv.z; rr[4 * q4 + 3] = rv.w;
          ff[4 * q4 + 0] = fv.x; ff[4 * q4 + 1] = fv.y; ff[4 * q4 + 2] = fv.z; ff[4 * q4 + 3] = fv.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) ff[i] = 1.f;
        if (quarter == 0 && (lane & 1) == 0) facb[buf * HG + hq * 16 + (lane >> 1)] = 1.f;
        if (quarter == 0 && lane == 0) flag[buf * 4 + hq] = 0;
      }
      // p = exp2(z - ref) rounded to bf16 into P^T[h][j]; running sums of the unrounded p
      unsigned char* pt = pts + buf * PTB;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int h = hq * 16 + i;
        const float p = exp2f(z[i] - (rr[i] == -INFINITY ? 0.f : rr[i]));
        ps[i] = fmaf(ps[i], ff[i], p);
        *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + (((j >> 3) ^ (h & 7)) << 4) + (j & 7) * 2) =
            __float2bfloat16_rn(p);
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::named_bar_sync(BAR_SOFTMAX, 256);
      if (sid == 0) tc::mbar_arrive(&bars[B_PFULL + buf]);
      if (c + 1 == cur.I.nch) {
        // the item's sums over its rows, per head
        butterfly16<false>(ps, lane);
        if ((lane & 1) == 0) red[quarter * HG + hq * 16 + (lane >> 1)] = ps[0];
        tc::named_bar_sync(BAR_SOFTMAX, 256);
        if (quarter == 0 && (lane & 1) == 0) {
          const int h = hq * 16 + (lane >> 1);
          fref[par * HG + h] = ref[h];
          fl[par * HG + h] = red[h] + red[HG + h];
        }
        tc::named_bar_sync(BAR_SOFTMAX, 256);
        if (sid == 0) tc::mbar_arrive(&bars[B_SMDONE + par]);
#pragma unroll
        for (int i = 0; i < 16; ++i) ps[i] = 0.f;
      }
      cur.advance(a, items);
    }
  } else if (is_loader_warp(warp)) {
    // ------------------------------------------------------------ loader warps
    const int lt = loader_index(warp) * 32 + lane;       // 0..223
    const unsigned char* kvb = static_cast<const unsigned char*>(a.kv);
    const unsigned char* winb = static_cast<const unsigned char*>(a.win);
    const unsigned char* dummy = static_cast<const unsigned char*>(a.q);   // source of zero-size copies
    Cursor cur;
    cur.start(a, items);
    while (cur.valid()) {
      const Item& I = cur.I;
      const long long g = cur.g;
      const int buf = static_cast<int>(g & 1);
      const int s = I.s_begin + cur.c * CK + lt;
      const int raw = (lt < CK && s < I.s_end && s < I.Kq && a.idx != nullptr) ? a.idx[I.qi * a.k + s] : 0;
      if (g >= 2) wait(B_KVEMPTY + buf, (g - 2) >> 1, 63);   // the PV of chunk g-2 has read this buffer
      if (lt < CK) {
        const unsigned char* p = nullptr;
        if (s < I.s_end) {
          if (s < I.Kq) {
            const int e = (a.idx == nullptr) ? s : raw;
            if (e >= 0 && e < a.N) {
              p = kvb + (static_cast<size_t>(I.b) * a.N + e) * (D * 2);
            } else if (e != -1) {
              report_error(a.status, CSA_ERR_DEVICE_CHECK, e);
            }
          } else {
            const int jw = s - I.Kq;
            const int u = I.t - a.window + 1 + jw;
            if (jw < a.window && u >= 0) p = winb + (static_cast<size_t>(I.b) * a.Wcap + u % a.Wcap) * (D * 2);
          }
        }
        rowptr[buf * CK + lt] = p;
      }
      tc::named_bar_sync(BAR_LOAD, kNLoad);
      if (!*abort_flag) {
        unsigned char* dst0 = kvs + buf * CK * 128;
        for (int i = lt; i < CK * 64; i += kNLoad) {
          const int row = i >> 6, col = i & 63;
          const unsigned char* rp = rowptr[buf * CK + row];
          cp_async16(dst0 + (col >> 3) * KVREG + row * 128 + (((col & 7) ^ (row & 7)) << 4), rp ? rp + col * 16 : dummy,
                     rp != nullptr);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      tc::named_bar_sync(BAR_LOAD, kNLoad);
      if (lt == 0) tc::mbar_arrive(&bars[B_KVFULL + buf]);
      cur.advance(a, items);
    }
  } else if (warp >= 16) {
    // ------------------------------------------------------------ correction warps
    const int quarter = warp & 3;                        // TMEM lanes 32 * quarter + lane
    const int ct = tid - 16 * 32;                        // 0..127
    long long n = 0, g = 0, qtma_uses = 0;
    // query block of item J into the operand regions; logit factors and rotation table of parity par
    auto prep = [&](const Item& J, int par) {
      if (ct == 0) {
        tc::mbar_arrive_expect_tx(&bars[B_QTMA], HG * D * 2);
#pragma unroll
        for (int r = 0; r < NREG; ++r)
          tc::tma_load_2d(qs + r * QREG, &qmap, r * 64, static_cast<int>(J.qi * a.H + J.h0), &bars[B_QTMA]);
      }
      if (ct < a.rp.r / 2) {
        float cs, sn;
        rope_cos_sin(J.t, a.rp.phase[ct], cs, sn);
        rope[par * 32 + ct] = make_float2(cs, sn);
      }
      // the copies land whatever happened elsewhere: wait for them without the abort flag
      if (!tc::mbar_wait(&bars[B_QTMA], static_cast<uint32_t>(qtma_uses & 1), nullptr, kWaitNs)) fail(64);
      ++qtma_uses;
      tc::named_bar_sync(BAR_CORR, 128);
      // two threads per head: thread ct owns head ct / 2, dims [256 (ct & 1), + 256) = regions
      // 4 (ct & 1) .. + 3; the odd thread also holds the rotated dims (region 7)
      const int h = ct >> 1, half = ct & 1;
      float ss = 0.f;
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const int region = half * 4 + (k >> 3), ch = k & 7;
        const uint4 u = *reinterpret_cast<const uint4*>(qs + region * QREG + h * 128 + ((ch ^ (h & 7)) << 4));
        const float x[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                            bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (half == 0) {
        const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + a.eps);
        cscale[par * HG + h] = a.q_norm_rope ? sl2 * inv : sl2;
      }
      if (n_lo && half == 1) {
        // rotated dims 448..511: hi back into region 7, lo into region 8
#pragma unroll 2
        for (int ch = 0; ch < 8; ++ch) {
          unsigned char* at = qs + (NREG - 1) * QREG + h * 128 + ((ch ^ (h & 7)) << 4);
          const uint4 u = *reinterpret_cast<const uint4*>(at);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 cssn = rope[par * 32 + ch * 4 + p];
            const float x0 = bf16lo(w[p]), x1 = bf16hi(w[p]);
            const float y0 = x0 * cssn.x - x1 * cssn.y, y1 = x0 * cssn.y + x1 * cssn.x;
            hw[p] = pack_bf16x2(y0, y1);
            lw[p] = pack_bf16x2(y0 - bf16lo(hw[p]), y1 - bf16hi(hw[p]));
          }
          *reinterpret_cast<uint4*>(at) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(qs + (OFF_QLO - OFF_Q) + h * 128 + ((ch ^ (h & 7)) << 4)) =
              make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::named_bar_sync(BAR_CORR, 128);
      if (ct == 0) tc::mbar_arrive(&bars[B_QREADY + par]);
    };

    {
      Item J0;
      if (next_with_rows(a, static_cast<long long>(blockIdx.x) - gridDim.x, items, J0) >= 0) prep(J0, 0);
    }
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
    const int Q = a.B * a.Tq;
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
      const Item I = item_at(a, it);
      if (I.nch == 0) {
        // no rows in this item: the output is the sink alone (zeros) or an empty partial
        if (a.cluster_merge) {
          if (ct < HG) reinterpret_cast<float2*>(misc + M_PML)[ct] = make_float2(-INFINITY, 0.f);
        } else if (a.n_splits == 1) {
          for (int e = ct; e < HG * D / 8; e += 128) {
            const int h = e / (D / 8), d8 = e % (D / 8);
            *reinterpret_cast<uint4*>(outp + (I.qi * a.H + I.h0 + h) * static_cast<long long>(D) + d8 * 8) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          if (a.lse != nullptr && ct < HG) a.lse[I.qi * a.H + I.h0 + ct] = a.sink[I.h0 + ct];
        } else {
          float* po = a.partial;
          float* pml = a.partial + static_cast<size_t>(Q) * a.n_splits * a.H * D;
          for (int e = ct; e < HG * D / 4; e += 128) {
            const int h = e / (D / 4), d4 = e % (D / 4);
            const size_t rowi = (static_cast<size_t>(I.qi) * a.n_splits + I.split) * a.H + I.h0 + h;
            *reinterpret_cast<float4*>(po + rowi * D + d4 * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          if (ct < HG) {
            const size_t rowi = (static_cast<size_t>(I.qi) * a.n_splits + I.split) * a.H + I.h0 + ct;
            pml[rowi * 2 + 0] = -INFINITY;
            pml[rowi * 2 + 1] = 0.f;
          }
        }
        continue;
      }
      const int par = static_cast<int>(n & 1);
      for (int c = 0; c < I.nch; ++c, ++g) {
        if (c == I.nch - 1) {
          Item J;
          if (next_with_rows(a, it, items, J) >= 0) {
            wait(B_QFREE, n, 65);                        // the last S^T of this item has read the query block
            prep(J, par ^ 1);
          }
        }
        if (c == 0) continue;                            // the first chunk starts the accumulator: no rescale
        const int buf = static_cast<int>(g & 1);
        wait(B_PFULL + buf, g >> 1, 66);
        if (flag[buf * 4] | flag[buf * 4 + 1] | flag[buf * 4 + 2] | flag[buf * 4 + 3]) {
          // a reference moved: O^T (this quarter's lanes, all heads) times the chunk's factors, once
          // the PV of chunk g-1 has landed
          wait(B_KVEMPTY + ((g - 1) & 1), (g - 1) >> 1, 67);
          tc::tc_fence_after();
#pragma unroll 1
          for (int part = 0; part < 8; ++part) {
            const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 2 * HG + part * 32;
            const int hb = (part & 1) * 32;
            float o[32];
            tc::tmem_ld32_wait(ta, o);
#pragma unroll
            for (int h = 0; h < 32; ++h) o[h] *= facb[buf * HG + hb + h];
            tc::tmem_st32_wait(ta, o);
          }
        }
        tc::tc_fence_before();
        tc::named_bar_sync(BAR_CORR, 128);
        if (ct == 0) tc::mbar_arrive(&bars[B_CDONE + buf]);
      }
      // ---------------- epilogue: O^T out of TMEM, normalised (one split) or as a partial
      wait(B_OREADY, n, 68);
      wait(B_SMDONE + par, n >> 1, 69);
      tc::tc_fence_after();
      if (ct < HG) {
        const int h = ct, hgl = I.h0 + h;
        const float r = fref[par * HG + h], l = fl[par * HG + h];
        if (a.n_splits == 1) {
          const float a2 = a.sink[hgl] * kLog2e;
          const float M = fmaxf(r, a2);
          const float f = (r == -INFINITY) ? 0.f : exp2f(r - M);
          const float L = l * f + exp2f(a2 - M);
          efac[h] = f / L;
          if (a.lse != nullptr) a.lse[I.qi * a.H + hgl] = (M + log2f(L)) * kLn2;
        } else if (a.cluster_merge) {
          reinterpret_cast<float2*>(misc + M_PML)[h] = make_float2(r, l);
        } else {
          float* pml = a.partial + static_cast<size_t>(Q) * a.n_splits * a.H * D;
          const size_t rowi = (static_cast<size_t>(I.qi) * a.n_splits + I.split) * a.H + hgl;
          pml[rowi * 2 + 0] = r;
          pml[rowi * 2 + 1] = l;
        }
      }
      tc::named_bar_sync(BAR_CORR, 128);
      float* po = a.partial;
      const bool odd = (lane & 1) != 0;
#pragma unroll 1
      for (int part = 0; part < 8; ++part) {
        const int mt = part >> 1, hb = (part & 1) * 32;  // O^T tile mt, heads hb .. hb + 31
        float o[32];
        tc::tmem_ld32_wait(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 2 * HG + mt * HG + hb, o);
        if (part == 7) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bars[B_OFREE]);   // the next item's PV may overwrite O^T
        }
        const int dim = mt * 128 + quarter * 32 + lane;
        if (a.n_splits == 1 && !(a.out_unrotate && (dim & ~1) >= D - a.rp.r)) {
          // dims that are not rotated back (warp-uniform: the rotated dims are the last r of the
          // row, r a multiple of 32): one bf16 per (head, dim), a warp storing 64 contiguous bytes
          // of one head's row
          __nv_bfloat16* op = outp + (I.qi * a.H + I.h0 + hb) * static_cast<long long>(D) + dim;
#pragma unroll
          for (int h = 0; h < 32; ++h) op[static_cast<size_t>(h) * D] = __float2bfloat16_rn(o[h] * efac[hb + h]);
        } else if (a.n_splits == 1) {
          // lanes 2i and 2i+1 swap one value per head pair, so that each lane holds two adjacent
          // dims of one head: the even lane head hb + 2hp, the odd lane head hb + 2hp + 1
          const int dd = dim & ~1;
          const bool unrot = a.out_unrotate && dd >= D - a.rp.r;
          float cs = 1.f, sn = 0.f;
          if (unrot) {                                  // rotation by -t
            const float2 cssn = rope[par * 32 + ((dd - (D - a.rp.r)) >> 1)];
            cs = cssn.x;
            sn = -cssn.y;
          }
#pragma unroll
          for (int hp = 0; hp < 16; ++hp) {
            const float xe = o[2 * hp] * efac[hb + 2 * hp];
            const float xo = o[2 * hp + 1] * efac[hb + 2 * hp + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? xe : xo, 1);
            float x0 = odd ? recv : xe, x1 = odd ? xo : recv;
            if (unrot) {
              const float y0 = x0 * cs - x1 * sn, y1 = x0 * sn + x1 * cs;
              x0 = y0;
              x1 = y1;
            }
            const int h = I.h0 + hb + 2 * hp + (odd ? 1 : 0);
            *reinterpret_cast<uint32_t*>(outp + (I.qi * a.H + h) * static_cast<long long>(D) + dd) =
                pack_bf16x2(x0, x1);
          }
        } else if (a.cluster_merge) {
          // stage the split's accumulator as fp32 [head][dim] over the (now idle) chunk buffers
          float* stage = reinterpret_cast<float*>(kvs);
#pragma unroll
          for (int h = 0; h < 32; ++h) stage[(hb + h) * D + dim] = o[h];
        } else {
          const size_t row0 = (static_cast<size_t>(I.qi) * a.n_splits + I.split) * a.H + I.h0 + hb;
#pragma unroll
          for (int h = 0; h < 32; ++h) po[(row0 + h) * D + dim] = o[h];
        }
      }
      tc::named_bar_sync(BAR_CORR, 128);                 // efac and this parity's tables are free again
      ++n;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (lane 0 only)
    if (lane == 0) {
      constexpr uint32_t idS = tc::umma_idesc_bf16(128, HG, 0, 0);
      constexpr uint32_t idPV = tc::umma_idesc_bf16(128, HG, 1, 0);
      const uint32_t kva = tc::sptr(kvs), qa = tc::sptr(qs), pa = tc::sptr(pts);
      bool issued = false;
      // S^T(g): K = 512 over the query block, then the lo half of the rotated dims against region 7
      auto issue_s = [&](long long g) {
        const int buf = static_cast<int>(g & 1);
        const uint32_t abase = kva + buf * CK * 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t ad = tc::umma_desc_sw128(abase + (k >> 2) * KVREG + (k & 3) * 32);
          const uint64_t bd = tc::umma_desc_sw128(qa + (k >> 2) * QREG + (k & 3) * 32);
          tc::umma_bf16(tmem + buf * HG, ad, bd, idS, k > 0 ? 1u : 0u);
        }
        if (n_lo) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = tc::umma_desc_sw128(abase + (NREG - 1) * KVREG + k * 32);
            const uint64_t bd = tc::umma_desc_sw128(qa + (OFF_QLO - OFF_Q) + k * 32);
            tc::umma_bf16(tmem + buf * HG, ad, bd, idS, 1u);
          }
        }
        issued = true;
      };
      auto issue_pv = [&](long long g, int c) {
        const int buf = static_cast<int>(g & 1);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int k = 0; k < CK / 16; ++k) {
            const uint64_t ad = tc::umma_desc_sw128_mn(kva + (2 * mt) * KVREG + (buf * CK + 16 * k) * 128, KVREG, 1024);
            const uint64_t bd = tc::umma_desc_sw128(pa + buf * PTB + k * 32);
            tc::umma_bf16(tmem + 2 * HG + mt * HG, ad, bd, idPV, (c > 0 || k > 0) ? 1u : 0u);
          }
        }
        tc::umma_commit(&bars[B_KVEMPTY + buf]);
      };
      // Two cursors over the same chunk sequence: S^T runs at most one chunk ahead of PV (its
      // TMEM buffer is free once the softmax of the chunk two back is done, i.e. once that
      // chunk's PV could be issued).  Measured alternatives that were slower: a ready PV before a
      // ready S^T, and S^T issued in slices with PVs between them.
      Cursor cs, cp;
      cs.start(a, items);
      cp.start(a, items);
      int cd_cnt[2] = {0, 0};
      int s_k = -1;                                      // 0: S^T(cs.g) ready to issue
      bool ok = true;
      long long t_last = clock64();
      uint32_t spins = 0;
      while (ok && cp.valid()) {
        bool progress = false;
        if (cs.valid() && cs.g <= cp.g + 1) {
          if (s_k < 0) {
            const int buf = static_cast<int>(cs.g & 1);
            const bool qok = cs.c != 0 || tc::mbar_test_wait(&bars[B_QREADY + static_cast<int>(cs.n & 1)],
                                                             static_cast<uint32_t>((cs.n >> 1) & 1));
            if (qok && tc::mbar_test_wait(&bars[B_KVFULL + buf], static_cast<uint32_t>((cs.g >> 1) & 1))) {
              tc::tc_fence_after();
              s_k = 0;
            }
          }
          if (s_k >= 0) {
            issue_s(cs.g);
            tc::umma_commit(&bars[B_SFULL + static_cast<int>(cs.g & 1)]);
            if (cs.c + 1 == cs.I.nch) tc::umma_commit(&bars[B_QFREE]);
            cs.advance(a, items);
            s_k = -1;
            progress = true;
          }
        }
        if (cp.g < cs.g) {
          const int buf = static_cast<int>(cp.g & 1);
          bool ready = tc::mbar_test_wait(&bars[B_PFULL + buf], static_cast<uint32_t>((cp.g >> 1) & 1));
          if (ready && cp.c > 0)
            ready = tc::mbar_test_wait(&bars[B_CDONE + buf], static_cast<uint32_t>(cd_cnt[buf] & 1));
          if (ready && cp.c == 0 && cp.n > 0)
            ready = tc::mbar_test_wait(&bars[B_OFREE], static_cast<uint32_t>((cp.n - 1) & 1));
          if (ready) {
            if (cp.c > 0) ++cd_cnt[buf];
            tc::tc_fence_after();
            issue_pv(cp.g, cp.c);
            if (cp.c + 1 == cp.I.nch) tc::umma_commit(&bars[B_OREADY]);
            cp.advance(a, items);
            progress = true;
          }
        }
        if (progress) {
          spins = 0;
          t_last = clock64();
        } else if ((++spins & 63u) == 0) {
          if (*abort_flag) {
            ok = false;
          } else if (clock64() - t_last > 4000000000ll) {   // about 2 s of SM clock
            fail(70);
            ok = false;
          }
        }
      }
      if (issued) {                                      // all MMAs done before TMEM is released
        tc::umma_commit(&bars[B_DRAIN]);
        if (!tc::mbar_wait(&bars[B_DRAIN], 0, nullptr, kWaitNs)) report_error(a.status, CSA_ERR_TIMEOUT, 77);
      }
    }
    __syncwarp();
  }

  // ---------------- teardown: every MMA complete (the MMA thread drained) before TMEM is released
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, TMEM_COLS);

  if (a.cluster_merge) {
    // ---------------- the splits of one query are the CTAs of this cluster (one item each, split =
    // cluster rank).  Each staged its (m, l) and fp32 accumulator; CTA r merges output units
    // [r U / S, (r + 1) U / S) of the U = 64 heads x 128 groups of 4 dims, reading every split's
    // staged accumulator over distributed shared memory (one 16-byte load per split and unit) in
    // fixed split order:
    //   out = sum_s O_s 2^(m_s - M) / (sum_s l_s 2^(m_s - M) + 2^(a_h - M)),  M = max(a_h, max_s m_s)
    cluster_barrier();
    const int S = a.n_splits;
    const uint32_t rank = cluster_rank();
    const Item I = item_at(a, blockIdx.x);
    float* facm = reinterpret_cast<float*>(pts);                 // [S][HG] merge factors
    const float* pml = reinterpret_cast<const float*>(misc + M_PML);
    if (tid < HG) {
      const int h = tid, hgl = I.h0 + h;
      const float a2 = a.sink[hgl] * kLog2e;
      float ms[8], ls[8];
      float M = a2;
#pragma unroll
      for (int sp = 0; sp < 8; ++sp) {
        if (sp < S) {
          const float2 v = ld_peer2(pml + 2 * h, static_cast<uint32_t>(sp));
          ms[sp] = v.x;
          ls[sp] = v.y;
          M = fmaxf(M, v.x);
        }
      }
      float L = exp2f(a2 - M);
#pragma unroll
      for (int sp = 0; sp < 8; ++sp)
        if (sp < S && ms[sp] != -INFINITY) L = fmaf(ls[sp], exp2f(ms[sp] - M), L);
      const float linv = 1.0f / L;
#pragma unroll
      for (int sp = 0; sp < 8; ++sp)
        if (sp < S) facm[sp * HG + h] = (ms[sp] == -INFINITY) ? 0.f : exp2f(ms[sp] - M) * linv;
      if (rank == 0 && a.lse != nullptr) a.lse[I.qi * a.H + hgl] = (M + log2f(L)) * kLn2;
    } else if (tid >= 128 && tid - 128 < a.rp.r / 2) {
      float cs, sn;
      rope_cos_sin(I.t, a.rp.phase[tid - 128], cs, sn);
      rope[32 + tid - 128] = make_float2(cs, -sn);                // rotation by -t
    }
    __syncthreads();
    const float* stage = reinterpret_cast<const float*>(kvs);
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
    constexpr int U = HG * (D / 4);
    const int u1 = static_cast<int>((rank + 1) * static_cast<long long>(U) / S);
    for (int u = static_cast<int>(rank * static_cast<long long>(U) / S) + tid; u < u1; u += NT) {
      const int h = u / (D / 4), d = 4 * (u % (D / 4));
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      for (int sp = 0; sp < S; ++sp) {
        const float f = facm[sp * HG + h];       // 0 for a split without rows (nothing staged)
        if (f != 0.f) {
          const float4 v = ld_peer4f(stage + h * D + d, static_cast<uint32_t>(sp));
          x[0] = fmaf(v.x, f, x[0]);
          x[1] = fmaf(v.y, f, x[1]);
          x[2] = fmaf(v.z, f, x[2]);
          x[3] = fmaf(v.w, f, x[3]);
        }
      }
      if (a.out_unrotate && d >= D - a.rp.r) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float2 cssn = rope[32 + ((d + 2 * p - (D - a.rp.r)) >> 1)];
          const float y0 = x[2 * p] * cssn.x - x[2 * p + 1] * cssn.y, y1 = x[2 * p] * cssn.y + x[2 * p + 1] * cssn.x;
          x[2 * p] = y0;
          x[2 * p + 1] = y1;
        }
      }
      *reinterpret_cast<uint2*>(outp + (I.qi * a.H + I.h0 + h) * static_cast<long long>(D) + d) =
          make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    }
    cluster_barrier();                                           // no CTA leaves while a peer reads it
  }
}

}  // namespace

bool attend_tc_supported(const AttendArgs& a) {
  return a.d == D && !a.fp8 && a.H % HG == 0 && (a.rp.r == 64 || a.rp.r == 0);
}

cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t s, int* launches) {
  const long long Q = static_cast<long long>(a.B) * a.Tq;
  const long long items = Q * (a.H / HG) * a.n_splits;
  if (items == 0) return cudaSuccess;
  CUtensorMap qmap;
  const uint64_t dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Q) * a.H};
  const uint32_t box[2] = {64, HG};
  if (!tc::make_tensor_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, 2, dims, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_attend_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Decode splits (2..8 per query): one CTA per split, the splits of a query in one cluster that
  // merges them in shared memory; no partials in global memory and no second kernel.
  if (a.n_splits > 1 && a.n_splits <= 8 && items <= 0x7fffffffLL) {
    AttendArgs b = a;
    b.cluster_merge = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(items));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = static_cast<size_t>(SMEM);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.n_splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, k_attend_tc, &cfg) == cudaSuccess && clusters >= 1) {
      cfg.numAttrs = 2;
      e = cudaLaunchKernelEx(&cfg, k_attend_tc, b, qmap);
      ++*launches;
      return e;
    }
    (void)cudaGetLastError();                                      // fall back to partials + merge kernel
  }
  AttendArgs b = a;
  b.cluster_merge = 0;
  const long long grid = items < sms ? items : sms;
  e = launch_k(k_attend_tc, dim3(static_cast<unsigned>(grid)), dim3(NT), static_cast<size_t>(SMEM), s, b, qmap);
  ++*launches;
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attend_combine(b, s, launches);
}

}  // namespace csa
