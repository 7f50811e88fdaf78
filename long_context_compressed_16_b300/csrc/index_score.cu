// Lightning-indexer scores I_{t,s} = sum_h w_{t,h} ReLU(q^I_{t,h} . K^I_s), s < floor((t+1)/m)
// ("DeepSeek V4 模型技术大全", CSA path, the I_{t,s} equation), on the 5th-generation tensor cores.
//
// The contraction runs with keys as the MMA's M dimension (128 keys per tile) and the (query,
// head) pairs of a group of G queries as N (G x padded heads <= 256), K = head_dim.  The fp32
// accumulator lives in tensor memory, one TMEM lane per key, so the ReLU / w-weighted head sum is
// a per-thread loop over TMEM columns with no cross-lane reduction.
//
// Persistent CTAs, one or two per SM, warp-specialised:
//   warp 0        TMA producer: key tiles (3-D tensor map, 128-byte swizzle, zero fill past N)
//                 into a ring of shared-memory stages, and each group's query block
//   warp 1        owns the TMEM allocation; one lane issues tcgen05.mma (M=128, N=G*heads,
//                 K=16 per instruction) and tcgen05.commit to release stages and publish results
//   warps 4..     epilogue: tcgen05.ld of the accumulator (double-buffered in TMEM), ReLU,
//                 weighting, head sum, optional FP8 row scale, coalesced score stores
//   FP8 keys only: converter warps widen each staged e4m3 tile to bf16 (exact) in the swizzled
//                 operand layout
// Work is a static split of (group, tile) pairs that all roles walk identically; every score is
// one MMA chain over the same K order, so results do not depend on the batch or the split.
// Every wait is bounded: a stuck pipeline sets CSA_ERR_TIMEOUT in the status word and the CTA
// drains its own copies, frees its tensor memory and returns.
#include "common.cuh"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int KT = 128;                 // keys per tile = MMA M
constexpr int kMaxSmem = 232448;        // dynamic shared memory per block on sm_100-class parts
#ifndef CSA_IDX_CTAS
#define CSA_IDX_CTAS 2                  // two CTAs per SM where they fit (N <= 64, no widening warps)
#endif
#ifndef CSA_IDX_MAX_STAGES
#define CSA_IDX_MAX_STAGES 6            // key-tile stages in flight per CTA (capped by shared memory)
#endif
#ifndef CSA_IDX_EVICT_FIRST
#define CSA_IDX_EVICT_FIRST 0           // 1: key tiles loaded with an L2 evict-first hint
#endif
#ifndef CSA_IDX_WALK_CHUNK
#define CSA_IDX_WALK_CHUNK 0            // > 0: CTAs take chunks of this many tiles round-robin
#endif

// FP8: e4m3 keys with per-row scales.  LP (low-precision indexer): the query is e4m3 too and the
// contraction runs on the FP8 tensor cores (kind::f8f6f4, K = 32 per instruction); otherwise FP8
// keys are widened to bf16 in shared memory by converter warps.
// Fused selection (CAND): the epilogue keeps, per query, the (key, entry) pairs above a running
// lower bound of the k-th largest score seen so far, and two selector warps pick each finished
// group's top-k from those lists (see the selector and the candidate epilogue below).
constexpr int kCandG = 4;          // queries per group the fused selection holds
constexpr int kCandBins = 256;     // histogram bins per query (bin 0 collects everything below)
constexpr int kClassShift = 17;    // key class = key >> 17: sign, exponent, 6 mantissa bits (64 per octave)
constexpr int kCandHead = 64;      // classes of headroom above the first tile's largest key (one octave)
constexpr int kSelWarps = 2;       // selector warps (warps 2 and 3, idle otherwise)
constexpr int kSelMembers = 512;   // keys of the k-th entry's class a selector warp holds
constexpr int kSelBitmap = 1024;   // words of a selector warp's entry bitmap (rows of up to 32768 entries)
constexpr int kSelU = 8;           // candidate-list loads in flight per lane

template <int DI, int NCOL, bool FP8, bool LP = false, bool CAND = false>
struct Cfg {
  static constexpr bool WIDEN = FP8 && !LP;               // converter warps widen e4m3 to bf16
  static constexpr int ESIZE = LP ? 1 : 2;                // operand bytes per element
  static constexpr int REG_ELEMS = 128 / ESIZE;           // elements per 128-byte swizzle row
  static constexpr int NREG = DI * ESIZE / 128;           // 128-byte swizzle regions per row
  static constexpr int KSTEPS = LP ? DI / 32 : DI / 16;   // MMAs per key tile
  static constexpr int KEY_REGION = KT * 128;
  static constexpr int STAGE_BYTES = NREG * KEY_REGION;   // bf16 key operand per stage
  static constexpr int STAGED_BYTES = WIDEN ? KT * DI : 0;  // e4m3 staging per stage
  static constexpr int Q_REGION = NCOL * 128;
  static constexpr int Q_BYTES = NREG * Q_REGION;
  // CTAs per SM: two independent pipelines per SM keep twice the key tiles in flight (measured on
  // the 128K decode: 56 -> 47 us, 0.75 -> 0.90 of the copy bandwidth); only when both fit in tensor
  // memory (4 x NCOL columns each) and in the registers (no widening warps)
  static constexpr int CTAS = (CSA_IDX_CTAS == 2 && NCOL <= 64 && !(FP8 && !LP)) ? 2 : 1;
  static constexpr int SMEM_CAP = CTAS == 2 ? 114688 : kMaxSmem;
  static constexpr int QB = (NCOL >= 256 || CTAS == 2) ? 1 : 2;   // query-block buffers
  // FP8 keys with N <= 128: the widening to bf16 is the busiest role, so 8 converter warps and
  // one set of 4 epilogue warps; otherwise 8 epilogue warps (two sets of four) and 4 converters
  static constexpr bool CONV_HEAVY = WIDEN && NCOL <= 128;
  // 256 columns without widening (the prefill groupings): 16 epilogue warps, four per SM
  // sub-partition, so that more tensor-memory loads are in flight (one warp's loads are serial,
  // about 44 bytes per clock each) and each warp sums one query of 64 heads per tile
  static constexpr int EW = (CONV_HEAVY || CTAS == 2) ? 4 : (NCOL == 256 && !WIDEN) ? 16 : 8;   // epilogue warps
  // NCOL <= 128: the two sets take alternate tiles; wider: they split the group's queries
  static constexpr bool TSPLIT = EW == 8 && NCOL <= 128;
  static constexpr int ACC_ARRIVALS = 32 * (TSPLIT ? EW / 2 : EW);   // epilogue threads per tile
  static constexpr int CW = WIDEN ? (CONV_HEAVY ? 8 : 4) : 0;   // converter warps
  static constexpr int THREADS = 32 * (4 + EW + CW);
  static constexpr int SPLIT = TSPLIT ? 1 : EW / 4;        // warp sets splitting a group's queries
  static constexpr int QW = NCOL / 64 / SPLIT > 0 ? NCOL / 64 / SPLIT : 1;   // queries per warp with 64 heads
  static constexpr int W_FLOATS = EW * (NCOL / SPLIT);    // per-epilogue-warp copy of its queries' head weights
  static constexpr int GMAX = 16;                         // queries per group (NCOL / 16 heads at most)
  static constexpr int NV_INTS = EW * GMAX;               // per-epilogue-warp visible counts of the group
  static constexpr int MISC = 1024;                       // barriers, TMEM address, flags
  // fused selection: per-query histograms (two group buffers), the per-tile ballot and maximum
  // exchange (two tile buffers), thresholds / bases / counts, the handoff barriers, and the
  // selector warps' histograms and class-member keys
  static constexpr int CAND_SMEM =
      CAND ? (2 * kCandG * kCandBins + 2 * kCandG * 4 /*maxima*/ + 2 * kCandG * 2 /*thr, lo*/ +
              2 * kCandG * 4 /*counts*/) * 4 + 4 * 8 + kSelWarps * (kCandBins + kSelMembers + kSelBitmap) * 4
           : 0;
  static constexpr int FIXED =
      1024 /*alignment slack*/ + QB * Q_BYTES + W_FLOATS * 4 + NV_INTS * 4 + MISC + CAND_SMEM;
  static constexpr int S_RAW = (SMEM_CAP - FIXED) / (STAGE_BYTES + STAGED_BYTES);
  static constexpr int STAGES = S_RAW > CSA_IDX_MAX_STAGES ? CSA_IDX_MAX_STAGES : S_RAW;
  static constexpr int SMEM = FIXED + STAGES * (STAGE_BYTES + STAGED_BYTES);
  static constexpr int ACC = NCOL <= 128 ? 4 : 2;            // accumulator buffers in tensor memory
  static constexpr int TMEM_COLS = (ACC * NCOL) <= 32 ? 32 : (ACC * NCOL) <= 64 ? 64 : (ACC * NCOL) <= 128 ? 128
                                   : (ACC * NCOL) <= 256 ? 256 : 512;
  static_assert(STAGES >= 2, "shared memory too small for two stages");
  static_assert(SMEM <= SMEM_CAP, "shared memory budget");
  static_assert(CTAS == 1 || TMEM_COLS <= 256, "two CTAs per SM must share the 512 TMEM columns");
  static_assert(NCOL % 16 == 0 && NCOL >= 16 && NCOL <= 256, "UMMA N for M = 128");
  // the candidate epilogue needs every tile seen by both warp sets (each owns half the queries)
  static_assert(!CAND || (!WIDEN && EW == 16 && !TSPLIT && QW == 1), "fused selection layout");
};

struct TcParams {
  int G, NHP;               // queries per group, padded heads per query
  int mode;                 // 0: flattened (group, tile) space split evenly; 1: whole groups, snake order;
                            // 2: chunks of `chunk` tiles of the flattened space, round-robin over CTAs
  int chunk;
  int tiles_max;            // ceil(N / KT)
  long long F;              // groups * tiles_max (mode 0)
  int fill_invisible;
};

struct GroupInfo {
  int b, i0, nq, nt;
};

__device__ __forceinline__ GroupInfo group_info(const IndexArgs& a, const TcParams& p, int g) {
  GroupInfo gi;
  const int ga = a.q_begin + g;
  const int gpb = (a.Tq + p.G - 1) / p.G;
  gi.b = ga / gpb;
  gi.i0 = (ga % gpb) * p.G;
  gi.nq = min(p.G, a.Tq - gi.i0);
  int maxvis = 0;
  for (int j = 0; j < gi.nq; ++j)
    maxvis = max(maxvis, n_visible(a.q_pos[static_cast<size_t>(gi.b) * a.Tq + gi.i0 + j], a.m, a.N));
  gi.nt = p.fill_invisible ? p.tiles_max : (maxvis + KT - 1) / KT;
  return gi;
}

// Walks this CTA's (group, tile) pairs; every role runs its own copy and sees the same sequence.
struct Walker {
  long long f, f_end;       // mode 0
  int round;                // mode 1
  int g, t;
  GroupInfo gi;

  __device__ void init(const TcParams& p, int ngroups) {
    const long long P = gridDim.x, c = blockIdx.x;
    if (p.mode == 0) {
      f = c * p.F / P;
      f_end = (c + 1) * p.F / P;
    } else {
      f = f_end = 0;
    }
    round = 0;
    g = -1;
    t = 0;
    (void)ngroups;
  }

  // Advances to the next pair; returns false when the CTA has no more work.  new_group is set
  // when the pair belongs to a different group than the previous one.
  __device__ bool next(const IndexArgs& a, const TcParams& p, int ngroups, bool& new_group) {
    new_group = false;
    if (p.mode == 2) {
      for (;;) {
        while (f < f_end) {
          const int gg = static_cast<int>(f / p.tiles_max);
          const int tt = static_cast<int>(f % p.tiles_max);
          if (gg != g) {
            g = gg;
            gi = group_info(a, p, g);
            new_group = true;
          }
          if (tt < gi.nt) {
            t = tt;
            ++f;
            return true;
          }
          f = static_cast<long long>(gg + 1) * p.tiles_max;
        }
        const long long ci = static_cast<long long>(blockIdx.x) + static_cast<long long>(round) * gridDim.x;
        ++round;
        f = ci * p.chunk;
        if (f >= p.F) return false;
        f_end = f + p.chunk < p.F ? f + p.chunk : p.F;
      }
    }
    if (p.mode == 0) {
      while (f < f_end) {
        const int gg = static_cast<int>(f / p.tiles_max);
        const int tt = static_cast<int>(f % p.tiles_max);
        if (gg != g) {
          g = gg;
          gi = group_info(a, p, g);
          new_group = true;
        }
        if (tt < gi.nt) {
          t = tt;
          ++f;
          return true;
        }
        f = static_cast<long long>(gg + 1) * p.tiles_max;
      }
      return false;
    }
    if (g >= 0 && t + 1 < gi.nt) {
      ++t;
      return true;
    }
    const int P = gridDim.x, c = blockIdx.x;
    for (;;) {
      const long long base = static_cast<long long>(round) * P;
      if (base >= ngroups) return false;
      const long long gg = base + ((round & 1) ? (P - 1 - c) : c);
      ++round;
      if (gg >= ngroups) continue;
      g = static_cast<int>(gg);
      gi = group_info(a, p, g);
      if (gi.nt == 0) continue;
      t = 0;
      new_group = true;
      return true;
    }
  }
};

// How many of the first n round-robin items (item j goes to slot j % P) went to slot i.
__device__ __forceinline__ long long issued_into(long long n, int i, int P) {
  return n > i ? (n - 1 - i) / P + 1 : 0;
}

// Two e4m3 codes -> two bf16 values, exact: the hardware widening to f16 is exact, f16 -> f32 is
// exact, and an e4m3 value (at most 4 significant bits, exponent within bf16's range) is a bf16
// value, so the rounding f32 -> bf16 changes nothing.  Four instructions per pair.
__device__ __forceinline__ uint32_t e4m3x2_to_bf162(uint16_t v) {
  const uint32_t h2 = e4m3x2_to_half2(v);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return pack_bf16x2(f.x, f.y);
}

// ------------------------------------------------------------------ fused selection: selector
//
// The selection is the TopK_k equation of the CSA path ("DeepSeek V4 模型技术大全") with ties to
// the smaller entry.  It reads the query's candidates (every entry that can still be among its
// top k: four sub-lists, one per quarter of each tile's keys, each in increasing entry order, of
// key << 32 | entry) instead of the whole score row.

constexpr uint32_t kEntryMax = 0x3FFFFu;   // entries are below 2^18: kEntryMax - entry orders them reversed

// The bin of a kCandBins-bin histogram (bins in increasing key order) where the count of entries
// in it and in the bins above first reaches K, in every lane: returns the bin (-1 when the whole
// histogram holds fewer than K), with the count above it (fa) and its own count (fc).  Lane l
// reads bins 8l .. 8l+7 as two 16-byte loads (no bank conflicts) and the counts above come from a
// suffix sum across the lanes.  The loads are volatile: other warps may still be adding to the
// bins, and any partial view only undercounts.
__device__ __forceinline__ int hist_kth_bin(const uint32_t* h, uint32_t K, uint32_t& fa, uint32_t& fc) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8];
  asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3]) : "r"(tc::sptr(h + 8 * lane)));
  asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(c[4]), "=r"(c[5]), "=r"(c[6]), "=r"(c[7]) : "r"(tc::sptr(h + 8 * lane + 4)));
  uint32_t csum = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) csum += c[u];
  uint32_t suf = csum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += y;
  }
  uint32_t above = suf - csum;                 // entries in the bins above 8l + 7
  int fb = -1;
  uint32_t a0 = 0, c0 = 0;
#pragma unroll
  for (int u = 7; u >= 0; --u) {
    if (above < K && K <= above + c[u]) {
      fb = 8 * lane + u;
      a0 = above;
      c0 = c[u];
    }
    above += c[u];
  }
  const uint32_t fm = __ballot_sync(0xffffffffu, fb >= 0);
  if (fm == 0u) {
    fa = fc = 0;
    return -1;
  }
  const int src = __ffs(fm) - 1;
  fa = __shfl_sync(0xffffffffu, a0, src);
  fc = __shfl_sync(0xffffffffu, c0, src);
  return __shfl_sync(0xffffffffu, fb, src);
}

// The smallest score whose order key (order_key) is at least T, so that order_key(s) >= T exactly
// when s >= key_floor_float(T) (non-NaN s): the inverse of order_key.  A T above every finite
// key's range decodes to a NaN (nothing compares >= it, as nothing has such a key); a T below
// every finite key gives -inf (everything passes).
__device__ __forceinline__ float key_floor_float(uint32_t T) {
  if (T & 0x80000000u) return __uint_as_float(T & 0x7FFFFFFFu);
  const float f = __uint_as_float(~T);
  return (f != f) ? -INFINITY : f;
}

struct CandLists {
  const unsigned long long* base;   // sub-list q at base + q * sub_cap
  int sub_cap;
  int n[4];
};

// f(e, valid) for every candidate, warp-uniform: 32 consecutive entries of a sub-list per call
// round, kSelU rounds of loads in flight
template <typename F>
__device__ __forceinline__ void for_each_cand(const CandLists& cl, F f) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {
    const unsigned long long* sub = cl.base + static_cast<long long>(q) * cl.sub_cap;
    const int n = cl.n[q];
    for (int b = 0; b < n; b += 32 * kSelU) {
      unsigned long long e[kSelU];
#pragma unroll
      for (int u = 0; u < kSelU; ++u) {
        const int i = b + u * 32 + lane;
        e[u] = i < n ? sub[i] : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kSelU; ++u) f(e[u], b + u * 32 + lane < n);
    }
  }
}

// Warp-wide radix select, 8 bits at a time.  each(g) calls g(key, valid) for every element
// (warp-uniform).  Among the valid keys whose bits at and above `pos` equal `prefix`, finds the
// rem-th largest.  On return prefix holds the threshold's bits at and above cmp_shift, rem how
// many keys equal to it at that level are taken, and eq how many there are (eq = rem when the
// threshold bin is taken whole; unchanged when no pass ran).  wh: kCandBins zeroed shared bins,
// zeroed again on return.  False when the counts cannot hold the rem-th key.
template <typename Each>
__device__ bool warp_radix(Each each, int pos, uint32_t& prefix, int& rem, int& cmp_shift, uint32_t& eq, uint32_t* wh) {
  const int lane = threadIdx.x & 31;
  cmp_shift = pos;
  while (pos > 0) {
    const int nbits = pos < 8 ? pos : 8;
    const int sh = pos - nbits;
    const uint32_t dmask = (1u << nbits) - 1u;
    const uint32_t hmask = pos >= 32 ? 0u : ~((1u << pos) - 1u);
    const uint32_t pf = prefix;
    each([&](uint32_t kk, bool v) {
      if (v && (kk & hmask) == pf) atomicAdd(&wh[(kk >> sh) & dmask], 1u);
    });
    __syncwarp();
    // lane owns 8 bins at descending positions and clears them for the next pass
    const int nb = 1 << nbits;
    uint32_t c[8];
    uint32_t csum = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int bin = nb - 1 - (8 * lane + u);
      c[u] = 0u;
      if (bin >= 0) {
        c[u] = wh[bin];
        wh[bin] = 0u;
      }
      csum += c[u];
    }
    uint32_t incl = csum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t above = incl - csum;
    const uint32_t r = static_cast<uint32_t>(rem);
    int fb = -1;
    uint32_t fa = 0, fc = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (above < r && r <= above + c[u]) {
        fb = nb - 1 - (8 * lane + u);
        fa = above;
        fc = c[u];
      }
      above += c[u];
    }
    const uint32_t fm = __ballot_sync(0xffffffffu, fb >= 0);
    __syncwarp();
    if (fm == 0u) return false;
    const int src = __ffs(fm) - 1;
    fb = __shfl_sync(0xffffffffu, fb, src);
    fa = __shfl_sync(0xffffffffu, fa, src);
    fc = __shfl_sync(0xffffffffu, fc, src);
    prefix |= static_cast<uint32_t>(fb) << sh;
    rem -= static_cast<int>(fa);
    eq = fc;
    pos = sh;
    cmp_shift = sh;
    if (fc == static_cast<uint32_t>(rem)) break;   // the threshold bin is taken whole
  }
  return true;
}

// Writes the entries marked in the bitmap bm (nwords words) to out in increasing entry order; lane
// l reads words [l W, (l + 1) W).  False (nothing written) unless exactly K entries are marked.
__device__ bool emit_bitmap(const uint32_t* bm, int nwords, int32_t* out, int K) {
  const int lane = threadIdx.x & 31;
  const int W = (nwords + 31) / 32;
  const int w0 = min(nwords, lane * W), w1 = min(nwords, w0 + W);
  uint32_t cnt = 0;
  for (int i = w0; i < w1; ++i) cnt += __popc(bm[i]);
  uint32_t ex = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, ex, o);
    if (lane >= o) ex += y;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, ex, 31);
  if (total != static_cast<uint32_t>(K)) return false;
  uint32_t o = ex - cnt;
  for (int i = w0; i < w1; ++i) {
    uint32_t bits = bm[i];
    while (bits != 0u) {
      const int b = __ffs(bits) - 1;
      out[o++] = i * 32 + b;
      bits &= bits - 1u;
    }
  }
  return true;
}

// Top-k row of query qi from its candidates and the final histogram of their key classes (bins
// 1 .. kCandBins-2 hold the single class lo + bin - 1).  The class of the k-th largest key comes
// from the histogram.  When it is one of those bins and holds at most kSelMembers keys, one pass
// over the lists decides every entry (see below); otherwise the lists are radix-selected whole,
// keys equal to the threshold beyond what is taken going by smallest entry (a radix select on
// kEntryMax - entry).  The selected entries are marked in a bitmap of the row, which is read in
// order: the output lists them in increasing entry, as the TopK definition's ties need, and the
// lists may be visited in any order.
__device__ void select_query(const IndexArgs& a, long long qi, const CandLists& cl, const uint32_t* hist, int lo,
                             int shift, uint32_t* wh, uint32_t* mem, uint32_t* bm) {
  const int lane = threadIdx.x & 31;
  const int K = a.k;
  int32_t* out = a.idx_out + qi * K;
  const int nv = n_visible(a.q_pos[qi], a.m, a.N);
  if (nv <= K) {
    for (int i = lane; i < K; i += 32) out[i] = i < nv ? i : -1;
    return;
  }
  const int L = cl.n[0] + cl.n[1] + cl.n[2] + cl.n[3];
  if (L < K || (nv + 31) / 32 > kSelBitmap) {   // cannot happen: the lists hold the row's top k
    if (lane == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2000);
    return;
  }
  uint32_t fa = 0, fc = 0;
  const int fb = hist_kth_bin(hist, static_cast<uint32_t>(K), fa, fc);
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t thr = 0, eq = 0;
  int rem = K, cmp = 0;
  bool ok = true;
  const int lowb = kClassShift - shift;        // key bits below the class
  const int nwords = (nv + 31) / 32;
  if (fb >= 1 && fb <= kCandBins - 2 && fc <= static_cast<uint32_t>(kSelMembers)) {
    // one pass over the lists: entries of the classes above the k-th one are marked at once;
    // the k-th class's keys go to shared memory as (low key bits, kEntryMax15 - entry), one
    // 32-bit value each (entries are below 2^15), whose larger values are exactly the better
    // entries (larger key, or equal key and smaller entry): its rem largest are marked next
    const uint32_t cls = static_cast<uint32_t>(lo + fb - 1);
    const uint32_t lmask = (1u << lowb) - 1u;
    for (int i = lane; i < nwords; i += 32) bm[i] = 0u;
    __syncwarp();
    uint32_t m = 0;
    for_each_cand(cl, [&](unsigned long long e, bool v) {
      const uint32_t ks = static_cast<uint32_t>(e >> 32);
      const uint32_t entry = static_cast<uint32_t>(e & 0xFFFFFFFFull);
      const uint32_t c = ks >> lowb;
      if (v && c > cls && entry < static_cast<uint32_t>(nv)) atomicOr(&bm[entry >> 5], 1u << (entry & 31));
      const bool hit = v && c == cls;
      const uint32_t hm = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        const uint32_t q = m + __popc(hm & lt);
        if (q < static_cast<uint32_t>(kSelMembers)) mem[q] = ((ks & lmask) << 15) | (0x7FFFu - (entry & 0x7FFFu));
      }
      m += __popc(hm);
    });
    __syncwarp();
    if (m != fc) {
      if (lane == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2001);
      return;
    }
    int rem1 = K - static_cast<int>(fa);
    uint32_t pre = 0, eq1 = fc;
    int cmp1 = lowb + 15;                        // every member taken: compare nothing below the class
    const int nm = static_cast<int>(fc);
    if (fc != static_cast<uint32_t>(rem1)) {
      ok = warp_radix([&](auto g) {
        for (int b = 0; b < nm; b += 32) g(b + lane < nm ? mem[b + lane] : 0u, b + lane < nm);
      }, lowb + 15, pre, rem1, cmp1, eq1, wh);
      if (!ok) {
        if (lane == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2002);
        return;
      }
    }
    // the member values are distinct, so every value at or above the threshold is taken
    const uint32_t tcm = cmp1 >= 32 ? 0u : pre >> cmp1;
    for (int b = 0; b < nm; b += 32) {
      if (b + lane < nm) {
        const uint32_t val = mem[b + lane];
        if ((cmp1 >= 32 ? 0u : val >> cmp1) >= tcm) {
          const uint32_t entry = 0x7FFFu - (val & 0x7FFFu);
          if (entry < static_cast<uint32_t>(nv)) atomicOr(&bm[entry >> 5], 1u << (entry & 31));
        }
      }
    }
    __syncwarp();
    if (!emit_bitmap(bm, nwords, out, K) && lane == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2003);
    return;
  } else {
    uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
    for_each_cand(cl, [&](unsigned long long e, bool v) {
      if (v) {
        const uint32_t ks = static_cast<uint32_t>(e >> 32);
        kmax = max(kmax, ks);
        kmin = min(kmin, ks);
      }
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    }
    const int pos = kmax == kmin ? 0 : 32 - __clz(kmax ^ kmin);
    uint32_t pre = pos >= 32 ? 0u : (kmax >> pos) << pos;
    rem = K;
    eq = static_cast<uint32_t>(L);               // no pass: every key equals kmax
    ok = warp_radix([&](auto g) {
      for_each_cand(cl, [&](unsigned long long e, bool v) { g(static_cast<uint32_t>(e >> 32), v); });
    }, pos, pre, rem, cmp, eq, wh);
    thr = pre;
  }
  // keys equal to the threshold, more of them than are taken: the smallest entries go first
  const bool ties = ok && cmp == 0 && eq > static_cast<uint32_t>(rem);
  uint32_t tpre = 0;
  int tcmp_shift = 0;
  if (ties) {
    int trem = rem;
    uint32_t teq = 0;
    const uint32_t t = thr;
    ok = warp_radix([&](auto g) {
      for_each_cand(cl, [&](unsigned long long e, bool v) {
        g(kEntryMax - static_cast<uint32_t>(e & 0xFFFFFFFFull), v && static_cast<uint32_t>(e >> 32) == t);
      });
    }, 18, tpre, trem, tcmp_shift, teq, wh);
  }
  if (!ok) {
    if (lane == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2002);
    return;
  }
  for (int i = lane; i < nwords; i += 32) bm[i] = 0u;
  __syncwarp();
  const uint32_t tc_ = cmp >= 32 ? 0u : thr >> cmp;
  for_each_cand(cl, [&](unsigned long long e, bool v) {
    const uint32_t ks = static_cast<uint32_t>(e >> 32);
    const uint32_t entry = static_cast<uint32_t>(e & 0xFFFFFFFFull);
    const uint32_t kt = cmp >= 32 ? 0u : ks >> cmp;
    bool sel = v && kt >= tc_;
    if (sel && kt == tc_ && ties) sel = ((kEntryMax - entry) >> tcmp_shift) >= (tpre >> tcmp_shift);
    if (sel && entry < static_cast<uint32_t>(nv)) atomicOr(&bm[entry >> 5], 1u << (entry & 31));
  });
  __syncwarp();
  if (!emit_bitmap(bm, nwords, out, K) && lane == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -2003);
}

template <int DI, int NCOL, bool FP8, bool LP, bool CAND>
__global__ void __launch_bounds__(Cfg<DI, NCOL, FP8, LP, CAND>::THREADS, Cfg<DI, NCOL, FP8, LP, CAND>::CTAS)
k_index_score(const IndexArgs a, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
              const TcParams p) {
  using C = Cfg<DI, NCOL, FP8, LP, CAND>;
  constexpr int S = C::STAGES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA destinations and the 128-byte swizzle atoms need 1024-byte alignment of the shared-window
  // offset (not of the generic address)
  unsigned char* smem = smem_raw + ((1024u - (tc::sptr(smem_raw) & 1023u)) & 1023u);
  unsigned char* qbuf = smem;                                         // QB x Q_BYTES
  unsigned char* kbuf = qbuf + C::QB * C::Q_BYTES;                    // S x STAGE_BYTES
  unsigned char* sbuf = kbuf + S * C::STAGE_BYTES;                    // S x STAGED_BYTES (FP8)
  float* wsm = reinterpret_cast<float*>(sbuf + S * C::STAGED_BYTES);  // [EW][NCOL / SPLIT]
  int* nvsm = reinterpret_cast<int*>(wsm + C::W_FLOATS);                // [EW][GMAX]
  uint64_t* bars = reinterpret_cast<uint64_t*>(nvsm + C::NV_INTS);
  uint64_t* full = bars;              // [S] operand ready (TMA bytes, or converters)
  uint64_t* empty = full + S;         // [S] operand consumed (MMA commit)
  uint64_t* sfull = empty + S;        // [S] e4m3 staging landed (TMA)
  uint64_t* sempty = sfull + S;       // [S] e4m3 staging consumed (converters)
  uint64_t* qfull = sempty + S;       // [2]
  uint64_t* qempty = qfull + 2;       // [2]
  uint64_t* accfull = qempty + 2;     // [ACC]
  uint64_t* accempty = accfull + 4;   // [ACC]
  uint64_t* drain = accempty + 4;     // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // fused selection (CAND only; past the barriers' area).  Index [buf] is the group buffer (group
  // parity), [G] the query in the group, [4] the quarter of the tile's keys (epilogue warp).
  uint32_t* chist = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(bars) + C::MISC);  // [2][G][bins]
  uint32_t* cwmax = chist + 2 * kCandG * kCandBins;   // [2][G][4] largest key of a group's first tile
  volatile uint32_t* cthr = cwmax + 2 * kCandG * 4;   // [2][G] bits of the float t: emit scores >= t
  int* clo = reinterpret_cast<int*>(cwmax + 2 * kCandG * 4 + 2 * kCandG);   // [2][G] class of bin 1
  int* ccnt = clo + 2 * kCandG;                        // [2][G][4] sub-list lengths
  uint64_t* gdone = reinterpret_cast<uint64_t*>(ccnt + 2 * kCandG * 4);   // [2] group's lists complete
  uint64_t* gfree = gdone + 2;                         // [2] selectors done with a buffer
  uint32_t* selh = reinterpret_cast<uint32_t*>(gfree + 2);   // [kSelWarps][bins]
  uint32_t* selm = selh + kSelWarps * kCandBins;             // [kSelWarps][kSelMembers]
  uint32_t* selb = selm + kSelWarps * kSelMembers;           // [kSelWarps][kSelBitmap]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = a.q_count;
  grid_dep_wait();
  grid_dep_launch();

  // alignment the TMA / tensor-core path relies on; a violation is reported, never executed
  {
    const uint32_t bad = (tc::sptr(smem) & 1023u) | (tc::sptr(bars) & 7u) |
                         (CAND ? (tc::sptr(gdone) & 7u) | (tc::sptr(chist) & 15u) : 0u) |
                         static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&kmap) & 63u) |
                         static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&qmap) & 63u);
    if (bad != 0u) {
      if (threadIdx.x == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -1000 - static_cast<int>(bad));
      return;
    }
    // the candidate lists were sized for cand_ctas CTAs of at most kCandG queries per group
    if (CAND && (static_cast<int>(blockIdx.x) >= a.cand_ctas || p.G > kCandG || p.mode != 1)) {
      if (threadIdx.x == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -1100);
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], C::WIDEN ? C::CW * 32 : 1);
      tc::mbar_init(&empty[s], 1);
      tc::mbar_init(&sfull[s], 1);
      tc::mbar_init(&sempty[s], C::CW * 32 > 0 ? C::CW * 32 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < C::ACC; ++i) {
      tc::mbar_init(&accfull[i], 1);
      tc::mbar_init(&accempty[i], C::ACC_ARRIVALS);
    }
    tc::mbar_init(drain, 1);
    if (CAND) {
      for (int i = 0; i < 2; ++i) {
        tc::mbar_init(&gdone[i], 32 * C::EW);
        tc::mbar_init(&gfree[i], kSelWarps);
      }
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensormap(&kmap);
    tc::prefetch_tensormap(&qmap);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&](int where) {
    *abort_flag = 1;
    report_error(a.status, CSA_ERR_TIMEOUT, where);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Walker wk;
      wk.init(p, ngroups);
      long long n = 0;           // key-tile loads issued (load j went to stage j % S, phase j / S)
      int nq = 0;                // query-block loads issued (load j went to buffer j % QB)
      int gc = -1;
      bool nw;
      bool ok = true;
      while (ok && wk.next(a, p, ngroups, nw)) {
        if (nw) {
          ++gc;
          const int qb = gc % C::QB;
          if (!tc::mbar_wait(&qempty[qb], ((gc / C::QB) & 1) ^ 1, abort_flag)) { fail(1); ok = false; break; }
          tc::mbar_arrive_expect_tx(&qfull[qb], C::Q_BYTES);
          const int z = wk.gi.b * a.Tq + wk.gi.i0;
          for (int r = 0; r < C::NREG; ++r)
            tc::tma_load_3d(qbuf + qb * C::Q_BYTES + r * C::Q_REGION, &qmap, r * C::REG_ELEMS, 0, z, &qfull[qb]);
          ++nq;
        }
        const int s = static_cast<int>(n % S);
        const uint32_t ph = static_cast<uint32_t>((n / S) & 1);
        if (C::WIDEN) {
          if (!tc::mbar_wait(&sempty[s], ph ^ 1, abort_flag)) { fail(2); ok = false; break; }
          tc::mbar_arrive_expect_tx(&sfull[s], C::STAGED_BYTES);
          tc::tma_load_3d(sbuf + s * C::STAGED_BYTES, &kmap, 0, wk.t * KT, wk.gi.b, &sfull[s]);
        } else {
          if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag)) { fail(2); ok = false; break; }
          tc::mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          for (int r = 0; r < C::NREG; ++r) {
            if (CSA_IDX_EVICT_FIRST)
              tc::tma_load_3d_hint(kbuf + s * C::STAGE_BYTES + r * C::KEY_REGION, &kmap, r * C::REG_ELEMS, wk.t * KT,
                                   wk.gi.b, &full[s], tc::policy_evict_first());
            else
              tc::tma_load_3d(kbuf + s * C::STAGE_BYTES + r * C::KEY_REGION, &kmap, r * C::REG_ELEMS, wk.t * KT,
                              wk.gi.b, &full[s]);
          }
        }
        ++n;
      }
      // drain: every copy this CTA issued has landed before the CTA may exit (the last phase of
      // each barrier follows from the issue counts; no per-stage arrays in local memory)
      for (int s = 0; s < S; ++s) {
        const long long cnt = issued_into(n, s, S);
        if (cnt > 0 && !tc::mbar_wait(C::WIDEN ? &sfull[s] : &full[s], static_cast<uint32_t>((cnt - 1) & 1), nullptr))
          report_error(a.status, CSA_ERR_TIMEOUT, 9);
      }
      for (int i = 0; i < C::QB; ++i) {
        const long long cnt = issued_into(nq, i, C::QB);
        if (cnt > 0 && !tc::mbar_wait(&qfull[i], static_cast<uint32_t>((cnt - 1) & 1), nullptr))
          report_error(a.status, CSA_ERR_TIMEOUT, 9);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0 only)
    if (lane == 0) {
      constexpr uint32_t idesc = LP ? tc::umma_idesc_e4m3(KT, NCOL) : tc::umma_idesc_bf16(KT, NCOL);
      Walker wk;
      wk.init(p, ngroups);
      long long n = 0;
      int gc = -1;
      bool nw;
      bool issued = false;
      while (wk.next(a, p, ngroups, nw)) {     // tile n's commit goes to empty[n % S]
        if (nw) {
          ++gc;
          if (gc >= 1) tc::umma_commit(&qempty[(gc - 1) % C::QB]);   // group j's commit: qempty[j % QB]
          if (!tc::mbar_wait(&qfull[gc % C::QB], (gc / C::QB) & 1, abort_flag)) { fail(3); break; }
        }
        const int s = static_cast<int>(n % S);
        const uint32_t ph = static_cast<uint32_t>((n / S) & 1);
        const int acc = static_cast<int>(n % C::ACC);
        if (!tc::mbar_wait(&full[s], ph, abort_flag)) { fail(4); break; }
        if (!tc::mbar_wait(&accempty[acc], ((n / C::ACC) & 1) ^ 1, abort_flag)) { fail(5); break; }
        tc::tc_fence_after();
        // descriptors of the tile's first K step; a later step only moves the start address
        // (its 16-byte units fill the descriptor's low 14 bits, and every operand address of the
        // kernel stays below 256 KB, so the sum never carries out of that field)
        const uint64_t ad0 = tc::umma_desc_sw128(tc::sptr(kbuf + s * C::STAGE_BYTES));
        const uint64_t bd0 = tc::umma_desc_sw128(tc::sptr(qbuf + (gc % C::QB) * C::Q_BYTES));
#pragma unroll
        for (int k = 0; k < C::KSTEPS; ++k) {               // 32 bytes of K per instruction
          const int r = k >> 2, off = (k & 3) * 32;
          const uint64_t ad = ad0 + static_cast<uint64_t>((r * C::KEY_REGION + off) >> 4);
          const uint64_t bd = bd0 + static_cast<uint64_t>((r * C::Q_REGION + off) >> 4);
          if (LP) tc::umma_e4m3(tmem + acc * NCOL, ad, bd, idesc, k > 0 ? 1u : 0u);
          else tc::umma_bf16(tmem + acc * NCOL, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        tc::umma_commit(&empty[s]);
        tc::umma_commit(&accfull[acc]);
        issued = true;
        ++n;
      }
      // drain: all MMAs issued here have completed, and every arrival their commits trigger has
      // landed, before tensor memory is released and the CTA's shared memory reused
      if (issued) {
        tc::umma_commit(drain);
        if (!tc::mbar_wait(drain, 0, nullptr)) report_error(a.status, CSA_ERR_TIMEOUT, 10);
      }
      for (int s = 0; s < S; ++s) {
        const long long cnt = issued_into(n, s, S);
        if (cnt > 0 && !tc::mbar_wait(&empty[s], static_cast<uint32_t>((cnt - 1) & 1), nullptr))
          report_error(a.status, CSA_ERR_TIMEOUT, 11);
      }
      const int nqc = gc > 0 ? gc : 0;           // groups 0 .. gc-1 had their commit
      for (int i = 0; i < C::QB; ++i) {
        const long long cnt = issued_into(nqc, i, C::QB);
        if (cnt > 0 && !tc::mbar_wait(&qempty[i], static_cast<uint32_t>((cnt - 1) & 1), nullptr))
          report_error(a.status, CSA_ERR_TIMEOUT, 11);
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + C::EW) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;
    const int quarter = warp & 3;                 // TMEM lanes [32*quarter, +32)
    const int set = ew >> 2;                      // warp set: its tile parity or its query half
    const int half = C::TSPLIT ? 0 : set;
    constexpr int SPLIT = C::SPLIT;
    const int NHP = p.NHP, G = p.G;
    const int qs_per = (G + SPLIT - 1) / SPLIT;
    const int j_lo = half * qs_per, j_hi = min(G, j_lo + qs_per);
    float* wb = wsm + ew * (NCOL / SPLIT);        // this warp's copy of its queries' head weights
    int* nvb = nvsm + ew * C::GMAX;               // and of its queries' visible entry counts
    const int jn = j_hi - j_lo;                  // this warp's queries j_lo + jj, jj < jn (<= C::QW for 64 heads)
    // w-weighted ReLU head sums of the warp's queries at this thread's key (TMEM lane) of the tile
    // in tbase: per query four independent partial sums in a fixed order, sum = (p0 + p1) +
    // (p2 + p3); head h always feeds partial sum h % 4, in increasing h, whatever the load width.
    // 64 heads (at most C::QW queries per warp): 32-column loads, the next one in flight while the
    // current one is summed, and the pairs (p0, p1), (p2, p3) updated by packed fused
    // multiply-adds (the same roundings as one at a time).
    auto head_sums = [&](uint32_t tbase, float (&sums)[C::QW]) {
      float ps[C::QW][4];
#pragma unroll
      for (int jj = 0; jj < C::QW; ++jj) ps[jj][0] = ps[jj][1] = ps[jj][2] = ps[jj][3] = 0.f;
      uint32_t ra[32], rb[32];
      const int nch = 2 * jn;
      tc::tmem_ld32_issue(tbase + j_lo * 64, ra);
      tc::tmem_ld_wait();
      tc::reg_fence32(ra);
#pragma unroll
      for (int c = 0; c < 2 * C::QW; ++c) {
        if (c < nch) {
          if (c + 1 < nch) {
            const uint32_t col = static_cast<uint32_t>((j_lo + ((c + 1) >> 1)) * 64 + ((c + 1) & 1) * 32);
            if (c & 1) tc::tmem_ld32_issue(tbase + col, ra);
            else tc::tmem_ld32_issue(tbase + col, rb);
          }
          const uint32_t(&cur)[32] = (c & 1) ? rb : ra;
          const float4* w4 = reinterpret_cast<const float4*>(wb + (c >> 1) * 64 + (c & 1) * 32);
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 ww = w4[h >> 2];
            const float x2 = __uint_as_float(cur[h + 2]), x3 = __uint_as_float(cur[h + 3]);
            tc::fma_f32x2(ps[c >> 1][0], ps[c >> 1][1], ww.x, ww.y, fmaxf(__uint_as_float(cur[h]), 0.f),
                          fmaxf(__uint_as_float(cur[h + 1]), 0.f));
            tc::fma_f32x2(ps[c >> 1][2], ps[c >> 1][3], ww.z, ww.w, x2 + fabsf(x2), x3 + fabsf(x3));
          }
          if (c + 1 < nch) {
            tc::tmem_ld_wait();
            if (c & 1) tc::reg_fence32(ra);
            else tc::reg_fence32(rb);
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < C::QW; ++jj) sums[jj] = (ps[jj][0] + ps[jj][1]) + (ps[jj][2] + ps[jj][3]);
    };
    // 16 or 32 heads: one query at a time, one load of its columns
    auto head_sum1 = [&](uint32_t tbase, int j) -> float {
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      auto accum = [&](const float* v, const float* wrow, int cnt) {
        const float4* w4 = reinterpret_cast<const float4*>(wrow);
#pragma unroll
        for (int h = 0; h < cnt; h += 4) {
          const float4 ww = w4[h >> 2];
          ps[0] = fmaf(ww.x, fmaxf(v[h], 0.f), ps[0]);
          ps[1] = fmaf(ww.y, fmaxf(v[h + 1], 0.f), ps[1]);
          ps[2] = fmaf(ww.z, v[h + 2] + fabsf(v[h + 2]), ps[2]);
          ps[3] = fmaf(ww.w, v[h + 3] + fabsf(v[h + 3]), ps[3]);
        }
      };
      if (NHP == 16) {
        float v[16];
        tc::tmem_ld16_wait(tbase + j * NHP, v);
        accum(v, wb + (j - j_lo) * NHP, 16);
      } else {
        float v[32];
        tc::tmem_ld32_wait(tbase + j * NHP, v);
        accum(v, wb + (j - j_lo) * NHP, 32);
      }
      return (ps[0] + ps[1]) + (ps[2] + ps[3]);
    };
    // fused selection state.  Every warp keeps its own sub-list per query (its quarter of each
    // tile's keys, in entry order) and its length; the set agrees on each group's histogram base
    const int tis = quarter * 32 + lane;          // thread index inside the warp set
    const int cshift = a.bf16_scores ? 16 : 0;
    const int sub_cap = a.cand_cap / 4;
    int gce = -1, cbuf = 0;
    int ccount[C::QW], clos[C::QW];
#pragma unroll
    for (int jj = 0; jj < C::QW; ++jj) ccount[jj] = clos[jj] = 0;
    unsigned long long* csub = nullptr;           // this warp's sub-list of query j_lo
    bool dead = false;                            // a wait of this warp gave up: walk on, do nothing
    float* srow[C::QW];                           // 64 heads: this warp's score rows of the group
    int snv[C::QW];                               // and their visible entry counts
#pragma unroll
    for (int jj = 0; jj < C::QW; ++jj) {
      srow[jj] = nullptr;
      snv[jj] = 0;
    }
    Walker wk;
    wk.init(p, ngroups);
    long long n = 0;
    bool nw;
    while (wk.next(a, p, ngroups, nw)) {
      if (nw) {
        // per-group values are read from global memory once per group, not once per tile
        __syncwarp();
        for (int c = j_lo * NHP + lane; c < j_hi * NHP; c += 32) {
          const int j = c / NHP, h = c % NHP;
          float v = 0.f;
          if (j < wk.gi.nq && h < a.nI)
            v = a.w[(static_cast<size_t>(wk.gi.b) * a.Tq + wk.gi.i0 + j) * a.nI + h];
          // heads 2 and 3 of every four take ReLU(x) as (x + |x|) / 2 on the FMA pipe (the fmax
          // of the other two runs on the ALU pipe): their weight is stored halved, and
          // (w / 2) (x + |x|) = w ReLU(x) exactly, so each product and sum rounds as before
          wb[c - j_lo * NHP] = (h & 2) ? 0.5f * v : v;
        }
        for (int j = j_lo + lane; j < j_hi; j += 32)
          nvb[j] = j < wk.gi.nq ? n_visible(a.q_pos[static_cast<size_t>(wk.gi.b) * a.Tq + wk.gi.i0 + j], a.m, a.N)
                                : 0;
        __syncwarp();
        if (!CAND && NHP == 64) {
#pragma unroll
          for (int jj = 0; jj < C::QW; ++jj) {
            const int j = j_lo + jj;
            const bool live = jj < jn && j < wk.gi.nq;
            srow[jj] = live ? a.scores + (static_cast<long long>(wk.gi.b) * a.Tq + wk.gi.i0 + j - a.score_row_offset) *
                                             static_cast<long long>(a.N)
                            : nullptr;
            snv[jj] = live ? nvb[j] : 0;
          }
        }
        if (CAND) {
          // the selectors are done with this buffer (it held group gce - 2); clear this set's
          // histograms and thresholds (ordered before any use by the first tile's barrier)
          ++gce;
          cbuf = gce & 1;
          if (!dead && !__all_sync(0xffffffffu, tc::mbar_wait(&gfree[cbuf], ((gce >> 1) & 1) ^ 1, abort_flag))) {
            dead = true;
            fail(12);
          }
          if (!dead) {
            uint32_t* hb = chist + (cbuf * kCandG + j_lo) * kCandBins;
            for (int i = tis; i < jn * kCandBins; i += 128) hb[i] = 0u;
            if (tis < jn) cthr[cbuf * kCandG + j_lo + tis] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int jj = 0; jj < C::QW; ++jj) ccount[jj] = 0;
#pragma unroll
          for (int jj = 0; jj < C::QW; ++jj) {    // entries a query's list takes: none at most k visible
            const int j = j_lo + jj;
            snv[jj] = (jj < jn && j < wk.gi.nq && nvb[j] > a.k) ? nvb[j] : 0;
          }
          csub = a.cand + ((static_cast<long long>(blockIdx.x) * 2 + cbuf) * p.G + j_lo) *
                              static_cast<long long>(a.cand_cap) + static_cast<long long>(quarter) * sub_cap;
        }
      }
      if (C::TSPLIT && static_cast<int>(n & 1) != set) {   // the other set's tile
        ++n;
        continue;
      }
      const int acc = static_cast<int>(n % C::ACC);
      const int key = wk.t * KT + quarter * 32 + lane;
      float kscale = 1.f;                         // issued before the wait so its latency overlaps it
      if (FP8 && key < a.N) kscale = a.kI_scale[static_cast<size_t>(wk.gi.b) * a.N + key];
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * NCOL;
      if (CAND) {
        // ---- candidate epilogue.  Per query, each warp appends the visible entries of its
        // quarter whose key is at least the query's threshold to its sub-list, and counts them in
        // the query's histogram of key classes (the key's top 15 bits: 64 classes per octave; bin 0
        // collects the classes below the range, the top bin those above).  One warp of the set per
        // tile raises one query's threshold to just above the lowest edge of a class whose bins at
        // and above it already hold k entries: every entry of a later tile at or below that edge
        // is beaten by those k (smaller entries, keys at least as large), so the lists keep every
        // entry of the row's top k.  Any partial view of the histogram undercounts, so a threshold
        // read early, or computed while other warps still add to the bins, is still a valid bound.
        const bool first = wk.t == 0, last = wk.t == wk.gi.nt - 1;
        float sv[C::QW];
#pragma unroll
        for (int jj = 0; jj < C::QW; ++jj) sv[jj] = 0.f;
        if (!dead) {
          if (__all_sync(0xffffffffu, tc::mbar_wait(&accfull[acc], (n / C::ACC) & 1, abort_flag))) {
            tc::tc_fence_after();
            head_sums(tbase, sv);
            tc::tc_fence_before();
            tc::mbar_arrive(&accempty[acc]);      // tensor memory is free for the next tile
          } else {
            dead = true;
            fail(6);
          }
        }
        float scv[C::QW];                         // the scores, as the unfused path stores them
        bool vis[C::QW];
#pragma unroll
        for (int jj = 0; jj < C::QW; ++jj) {
          float v = sv[jj] * kscale;
          if (a.bf16_scores) v = __bfloat162float(__float2bfloat16_rn(v));
          scv[jj] = v;
          vis[jj] = jj < jn && key < snv[jj];
        }
        if (first) {
          // the histogram base of each query: the largest key of the group's first tile, agreed by
          // the set (the only barrier of the group; a warp that gave up makes the set leave here)
          if (!dead) {
#pragma unroll
            for (int jj = 0; jj < C::QW; ++jj) {
              if (jj < jn) {
                uint32_t mx = vis[jj] ? order_key(scv[jj]) : 0u;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) cwmax[(cbuf * kCandG + j_lo + jj) * 4 + quarter] = mx;
              }
            }
          }
          if (tc::named_bar_or(1 + set, 128, dead)) break;
#pragma unroll
          for (int jj = 0; jj < C::QW; ++jj) {
            if (jj < jn) {
              const uint32_t* wm = cwmax + (cbuf * kCandG + j_lo + jj) * 4;
              const uint32_t mx = max(max(wm[0], wm[1]), max(wm[2], wm[3]));
              clos[jj] = static_cast<int>(mx >> kClassShift) + kCandHead - (kCandBins - 2);
              if (tis == 0) clo[cbuf * kCandG + j_lo + jj] = clos[jj];
            }
          }
        }
        if (dead) {
          ++n;
          continue;
        }
#pragma unroll
        for (int jj = 0; jj < C::QW; ++jj) {
          if (jj < jn) {
            const int j = j_lo + jj;
            // key(s) >= T exactly when s >= the float T encodes (the key order is the score order)
            const float thr = first ? -INFINITY : __uint_as_float(cthr[cbuf * kCandG + j]);
            const bool pass = vis[jj] && scv[jj] >= thr;
            const uint32_t m = __ballot_sync(0xffffffffu, pass);
            if (pass) {
              const uint32_t kk = order_key(scv[jj]);
              const int pos = ccount[jj] + __popc(m & ((1u << lane) - 1u));
              if (pos < sub_cap)
                csub[static_cast<long long>(jj) * a.cand_cap + pos] =
                    (static_cast<unsigned long long>(kk >> cshift) << 32) | static_cast<uint32_t>(key);
              const int bin = min(max(static_cast<int>(kk >> kClassShift) - clos[jj] + 1, 0), kCandBins - 1);
              atomicAdd(&chist[(cbuf * kCandG + j) * kCandBins + bin], 1u);
            }
            ccount[jj] += __popc(m);
          }
        }
        if (!last) {
          // tile t: query t % jn, refreshed by warp (t / jn) % 4 of the set (one query per warp
          // set when the selection is fused: query 0, warp t % 4)
          const int jj = C::QW == 1 ? 0 : wk.t % jn;
          if (((C::QW == 1 ? wk.t : wk.t / jn) & 3) == quarter) {
            const int j = j_lo + jj;
            int lo_q = clos[0];
#pragma unroll
            for (int u = 1; u < C::QW; ++u)
              if (jj == u) lo_q = clos[u];
            uint32_t fa, fc;
            const int b = hist_kth_bin(chist + (cbuf * kCandG + j) * kCandBins, static_cast<uint32_t>(a.k), fa, fc);
            if (b >= 1 && lane == 0)
              cthr[cbuf * kCandG + j] = __float_as_uint(
                  key_floor_float((static_cast<uint32_t>(lo_q + b - 1) << kClassShift) + (1u << cshift)));
          }
        } else {
          // the group's sub-lists are complete: hand them to the selectors
          if (lane == 0) {
#pragma unroll
            for (int jj = 0; jj < C::QW; ++jj)
              if (jj < jn) ccnt[(cbuf * kCandG + j_lo + jj) * 4 + quarter] = ccount[jj];
          }
          tc::mbar_arrive(&gdone[cbuf]);
        }
        ++n;
        continue;
      }
      // the warp leaves together: a wait that gave up on any lane ends the loop for all lanes
      const bool got = tc::mbar_wait(&accfull[acc], (n / C::ACC) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got)) { fail(6); break; }
      tc::tc_fence_after();
      auto store = [&](int j, float sum) {
        if (j < wk.gi.nq && key < a.N) {
          const size_t qi = static_cast<size_t>(wk.gi.b) * a.Tq + wk.gi.i0 + j;
          const int nv = nvb[j];
          float* dst = a.scores + (static_cast<long long>(qi) - a.score_row_offset) * a.N;
          if (key < nv) {
            const float v = sum * kscale;
            dst[key] = a.bf16_scores ? __bfloat162float(__float2bfloat16_rn(v)) : v;
          }
          else if (p.fill_invisible) dst[key] = -INFINITY;
        }
      };
      if (NHP == 64) {                            // at most C::QW queries per warp
        float sv[C::QW];
        head_sums(tbase, sv);
        tc::tc_fence_before();
        tc::mbar_arrive(&accempty[acc]);          // tensor memory is free before the stores
#pragma unroll
        for (int jj = 0; jj < C::QW; ++jj) {
          if (srow[jj] != nullptr && key < a.N) {
            if (key < snv[jj]) {
              const float v = sv[jj] * kscale;
              srow[jj][key] = a.bf16_scores ? __bfloat162float(__float2bfloat16_rn(v)) : v;
            } else if (p.fill_invisible) {
              srow[jj][key] = -INFINITY;
            }
          }
        }
      } else {
        for (int j = j_lo; j < j_hi; ++j) store(j, head_sum1(tbase, j));
        tc::tc_fence_before();
        tc::mbar_arrive(&accempty[acc]);
      }
      ++n;
    }
  } else if (C::WIDEN && warp >= 4 + C::EW) {
    // ------------------------------------------------------------ e4m3 -> bf16 converters
    const int ctid = threadIdx.x - 32 * (4 + C::EW);
    Walker wk;
    wk.init(p, ngroups);
    long long n = 0;
    bool nw;
    constexpr int CPR = DI / 8;                   // 8-element chunks per row
    while (wk.next(a, p, ngroups, nw)) {
      const int s = static_cast<int>(n % S);
      const uint32_t ph = static_cast<uint32_t>((n / S) & 1);
      if (!tc::mbar_wait(&sfull[s], ph, abort_flag)) { fail(7); break; }
      if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag)) { fail(8); break; }
      const unsigned char* src = sbuf + s * C::STAGED_BYTES;
      unsigned char* dst = kbuf + s * C::STAGE_BYTES;
      for (int c = ctid; c < KT * CPR; c += C::CW * 32) {
        const int r = c / CPR, cc = c % CPR;
        const uint2 v = *reinterpret_cast<const uint2*>(src + r * DI + cc * 8);
        uint4 o;
        o.x = e4m3x2_to_bf162(static_cast<uint16_t>(v.x & 0xFFFF));
        o.y = e4m3x2_to_bf162(static_cast<uint16_t>(v.x >> 16));
        o.z = e4m3x2_to_bf162(static_cast<uint16_t>(v.y & 0xFFFF));
        o.w = e4m3x2_to_bf162(static_cast<uint16_t>(v.y >> 16));
        const int region = cc >> 3, chunk = cc & 7;
        *reinterpret_cast<uint4*>(dst + region * C::KEY_REGION + r * 128 + ((chunk ^ (r & 7)) << 4)) = o;
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&full[s]);
      tc::mbar_arrive(&sempty[s]);
      ++n;
    }
  } else if (CAND && (warp == 2 || warp == 3)) {
    // ------------------------------------------------------------ selectors (fused selection)
    // Walk this CTA's groups in the producer's order (groups no query of which sees an entry are
    // skipped by the other roles: their rows are all padding), wait for each group's lists, and
    // select the top k of queries sw, sw + 2, ... of the group.
    const int sw = warp - 2;
    uint32_t* wh = selh + sw * kCandBins;
    uint32_t* mem = selm + sw * kSelMembers;
    uint32_t* bm = selb + sw * kSelBitmap;
    for (int i = lane; i < kCandBins; i += 32) wh[i] = 0u;
    __syncwarp();
    const int shift = a.bf16_scores ? 16 : 0;
    const int sub_cap = a.cand_cap / 4;
    const int P = gridDim.x, c = blockIdx.x;
    int gcs = 0;
    for (int round = 0;; ++round) {
      const long long base = static_cast<long long>(round) * P;
      if (base >= ngroups) break;
      const long long gg = base + ((round & 1) ? (P - 1 - c) : c);
      if (gg >= ngroups) continue;
      const GroupInfo gi = group_info(a, p, static_cast<int>(gg));
      if (gi.nt == 0) {
        for (int j = sw; j < gi.nq; j += kSelWarps) {
          int32_t* out = a.idx_out + (static_cast<long long>(gi.b) * a.Tq + gi.i0 + j) * a.k;
          for (int i = lane; i < a.k; i += 32) out[i] = -1;
        }
        continue;
      }
      const int buf = gcs & 1;
      const bool got = tc::mbar_wait(&gdone[buf], (gcs >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got)) { fail(13); break; }
      for (int j = sw; j < gi.nq; j += kSelWarps) {
        CandLists cl;
        cl.base = a.cand + ((static_cast<long long>(blockIdx.x) * 2 + buf) * p.G + j) * static_cast<long long>(a.cand_cap);
        cl.sub_cap = sub_cap;
#pragma unroll
        for (int q = 0; q < 4; ++q) cl.n[q] = ccnt[(buf * kCandG + j) * 4 + q];
        select_query(a, static_cast<long long>(gi.b) * a.Tq + gi.i0 + j, cl, chist + (buf * kCandG + j) * kCandBins,
                     clo[buf * kCandG + j], shift, wh, mem, bm);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&gfree[buf]);
      ++gcs;
    }
  }

  // ------------------------------------------------------------ teardown
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------ host side

bool make_map_3d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint32_t box[3] = {b0, b1, b2};
  return tc::make_tensor_map(map, dt, 3, base, esize, dims, box, sw);
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

template <int DI, int NCOL, bool FP8, bool LP, bool CAND = false>
cudaError_t launch_t(const IndexArgs& a, const IndexGrouping& gr, int fill_invisible, cudaStream_t s,
                     int* launches) {
  using C = Cfg<DI, NCOL, FP8, LP, CAND>;
  CUtensorMap kmap, qmap;
  bool ok;
  if (LP)
    ok = make_map_3d(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.kI, DI, a.N, a.B, DI, KT, 1,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  else if (FP8)
    ok = make_map_3d(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.kI, DI, a.N, a.B, DI, KT, 1,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    ok = make_map_3d(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kI, DI, a.N, a.B, 64, KT, 1,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (LP)
    ok = ok && make_map_3d(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.qI, DI, a.nI,
                           static_cast<uint64_t>(a.B) * a.Tq, C::REG_ELEMS, gr.NHP, gr.G, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = ok && make_map_3d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.qI, DI, a.nI,
                           static_cast<uint64_t>(a.B) * a.Tq, 64, gr.NHP, gr.G, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  TcParams p;
  p.G = gr.G;
  p.NHP = gr.NHP;
  p.tiles_max = (a.N + KT - 1) / KT;
  p.fill_invisible = fill_invisible;
  const int sms = sm_count();
  const long long groups = a.q_count;
  // fused selection: whole groups per CTA in tile order (the lists are built in entry order)
  p.mode = (CAND || groups >= 4LL * sms) ? 1 : (CSA_IDX_WALK_CHUNK > 0 ? 2 : 0);
  p.chunk = CSA_IDX_WALK_CHUNK > 0 ? CSA_IDX_WALK_CHUNK : 1;
  p.F = groups * p.tiles_max;
  long long grid = static_cast<long long>(sms) * C::CTAS;
  if (p.mode != 1 && p.F < grid) grid = p.F;
  if (CAND && grid > a.cand_ctas) grid = a.cand_ctas;
  if (grid < 1) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_index_score<DI, NCOL, FP8, LP, CAND>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  e = launch_k(k_index_score<DI, NCOL, FP8, LP, CAND>, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS),
               static_cast<size_t>(C::SMEM), s, a, kmap, qmap, p);
  ++*launches;
  return e;
}

template <int DI, bool FP8, bool LP>
cudaError_t launch_di(const IndexArgs& a, const IndexGrouping& gr, int fill, cudaStream_t s, int* launches) {
  switch (gr.NCOL) {
    case 16: return launch_t<DI, 16, FP8, LP>(a, gr, fill, s, launches);
    case 32: return launch_t<DI, 32, FP8, LP>(a, gr, fill, s, launches);
    case 64: return launch_t<DI, 64, FP8, LP>(a, gr, fill, s, launches);
    case 128: return launch_t<DI, 128, FP8, LP>(a, gr, fill, s, launches);
    case 256: return launch_t<DI, 256, FP8, LP>(a, gr, fill, s, launches);
  }
  return cudaErrorInvalidValue;
}

// Low-precision indexer query: one warp per (query, head) row of 128 dims.  scale = amax / 448
// (1 for an all-zero row), codes = e4m3 RNE-saturated (q / scale) with the quotient in fp32, and
// the head weight absorbs the scale (ReLU commutes with a positive factor): wp = w * scale.
__global__ void __launch_bounds__(128) k_quant_q(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                                                 uint8_t* __restrict__ q8, float* __restrict__ wp, long long row0,
                                                 long long rows) {
  grid_dep_wait();
  grid_dep_launch();
  const long long r = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint2 u = *reinterpret_cast<const uint2*>(qI + (row0 + r) * 128 + lane * 4);
  const float v[4] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(__fdiv_rn(v[1], scale)), "f"(__fdiv_rn(v[0], scale)));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(__fdiv_rn(v[3], scale)), "f"(__fdiv_rn(v[2], scale)));
  *reinterpret_cast<uint32_t*>(q8 + r * 128 + lane * 4) = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  if (lane == 0) wp[r] = w[row0 + r] * scale;
}

}  // namespace

// a.q_begin / a.q_count: range of query GROUPS (gr.G consecutive queries of one sequence).
cudaError_t launch_index_score_groups(const IndexArgs& a, const IndexGrouping& gr, int fill_invisible,
                                      cudaStream_t s, int* launches) {
  if (a.q_count <= 0 || a.N <= 0) return cudaSuccess;
  if (a.lowp) return a.dI == 128 ? launch_di<128, true, true>(a, gr, fill_invisible, s, launches)
                                  : cudaErrorInvalidValue;
  if (a.dI == 128) return a.fp8 ? launch_di<128, true, false>(a, gr, fill_invisible, s, launches)
                                : launch_di<128, false, false>(a, gr, fill_invisible, s, launches);
  if (a.dI == 64) return a.fp8 ? launch_di<64, true, false>(a, gr, fill_invisible, s, launches)
                               : launch_di<64, false, false>(a, gr, fill_invisible, s, launches);
  return cudaErrorInvalidValue;
}

bool index_select_supported(const IndexGrouping& gr, int dI, int fp8, int lowp, int N) {
  if (gr.NCOL != 256 || gr.G > kCandG || gr.NHP != 64) return false;
  if (N < 1 || N > 32 * kSelBitmap) return false;   // the selector's entry bitmap
  if (fp8 && !lowp) return false;             // widened FP8 keys: no shared memory left for the lists' state
  return lowp ? dI == 128 : (dI == 64 || dI == 128);
}

int index_select_ctas() { return sm_count(); }

// per query: four sub-lists of (tiles x 32) slots, one per quarter of each tile's keys
int index_select_cap(int N) { return (N + KT - 1) / KT * KT; }

size_t index_select_bytes(const IndexGrouping& gr, int N) {
  return static_cast<size_t>(index_select_ctas()) * 2 * gr.G * static_cast<size_t>(index_select_cap(N)) *
         sizeof(unsigned long long);
}

// a.cand: index_select_bytes(gr, a.N) bytes; a.cand_cap = index_select_cap(N); a.cand_ctas = the SM count those
// bytes were sized for.  Writes a.idx_out for the queries of groups [q_begin, q_begin + q_count).
cudaError_t launch_index_select(const IndexArgs& a, const IndexGrouping& gr, cudaStream_t s, int* launches) {
  if (a.q_count <= 0 || a.N <= 0) return cudaErrorInvalidValue;
  if (!index_select_supported(gr, a.dI, a.fp8, a.lowp, a.N) || a.cand == nullptr || a.idx_out == nullptr ||
      a.cand_cap != index_select_cap(a.N) || a.cand_ctas < 1 || a.k < 1)
    return cudaErrorInvalidValue;
  if (a.lowp) return launch_t<128, 256, true, true, true>(a, gr, 0, s, launches);
  if (a.dI == 128) return launch_t<128, 256, false, false, true>(a, gr, 0, s, launches);
  return launch_t<64, 256, false, false, true>(a, gr, 0, s, launches);
}

// rows [row0, row0 + rows) of qI [.., 128] bf16 / w -> q8 [rows, 128] e4m3 / wp [rows] (rows
// counted from row0)
cudaError_t launch_quant_q(const void* qI, const float* w, void* q8, float* wp, long long row0, long long rows,
                           cudaStream_t s, int* launches) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 3) / 4;
  if (blocks > 2147483647LL) return cudaErrorInvalidValue;
  const cudaError_t e = launch_k(k_quant_q, dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s,
                                 static_cast<const __nv_bfloat16*>(qI), w, static_cast<uint8_t*>(q8), wp, row0, rows);
  ++*launches;
  return e;
}

}  // namespace csa
