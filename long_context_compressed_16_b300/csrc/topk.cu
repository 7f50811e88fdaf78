// Per-query top-k over the visible indexer scores ("DeepSeek V4 模型技术大全", CSA path, the TopK_k
// equation), ties to the smaller entry index.
//
// Radix select on order-preserving 32-bit keys of the fp32 scores, one CTA per slice of at most
// 32768 candidates, the slice's keys in that CTA's shared memory.
// The first 8-bit digit starts at the highest bit where the slice's largest and smallest keys
// differ (the bits above are common to all of them), so the histogram spreads over the scores'
// actual range; each pass narrows the threshold bin, and the search stops once the threshold bin
// is taken whole or all 32 bits are fixed.  A pass costs two block barriers: every thread adds
// its keys to a 256-bin shared histogram, then one warp scans the bins from the top, finds the
// threshold bin and clears the histogram for the next pass.  The selected set is written in
// increasing entry index: entries above the threshold bin and, inside it, the smallest indices
// first.
//
// Rows longer than one slice: up to 16 x 32768 entries, one thread-block cluster per row selects
// in one stage (k_topk_cluster, below: the slices' histograms are summed over distributed shared
// memory).  Longer rows run in two stages: every slice writes its own top-k (key, index)
// candidates in index order, and a merge CTA selects the top-k of the concatenation.  This is
// exact: an entry of the row's top-k is also in its slice's top-k (with the same smaller-index
// rule for ties), and the concatenated candidates stay in increasing index order.
// The result depends only on the query's own scores (batch-invariant and deterministic).
#include "common.cuh"

namespace csa {

namespace {

constexpr int kSlice = 32768;        // longest slice per CTA (128 KB of keys in shared memory)
constexpr int kMinSlice = 4096;      // slices are not split below this length
constexpr int kMergeCap = 16384;     // candidates one merge CTA holds (keys + indices: 128 KB)
#ifndef CSA_TOPK_TARGET_CTAS
#define CSA_TOPK_TARGET_CTAS 128
#endif

#ifndef CSA_TOPK_CLUSTER
#define CSA_TOPK_CLUSTER 1           // rows of 2..8 slices: one cluster per row instead of slices + merge
#endif
#ifndef CSA_TOPK_CLUSTER_LONG
#define CSA_TOPK_CLUSTER_LONG 1      // rows of more than 8 two-stage slices: 8 longer slices in a cluster
#endif
#ifndef CSA_TOPK_CLUSTER_NT
#define CSA_TOPK_CLUSTER_NT 1024     // threads per CTA of the cluster selection
#endif
constexpr int kClusterMax = 16;      // clusters of up to 16 CTAs (above 8: the non-portable size)
constexpr int kPeerBatch = 8;         // peers whose histogram words are loaded together
constexpr int kTargetCtas = CSA_TOPK_TARGET_CTAS;   // split rows until the first stage has about this many CTAs
constexpr int kMergeRounds = 16;     // 32-candidate rounds per merge warp (registers per thread)
constexpr int kDigit = 8;
constexpr int kBins = 1 << kDigit;          // one warp scans them: kBins / 32 per lane
constexpr int kBinsPerLane = kBins / 32;
constexpr uint32_t kNoIndex = 0xFFFFFFFFu;

// Exclusive block-wide scan of 64-bit values.  ws: 33 slots of shared memory.
__device__ __forceinline__ unsigned long long block_excl_scan(unsigned long long v, unsigned long long* ws,
                                                              unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long x = lane < nwarps ? ws[lane] : 0ull;
    unsigned long long xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += y;
    }
    ws[lane] = xi - x;
    if (lane == 31) ws[32] = xi;
  }
  __syncthreads();
  const unsigned long long r = ws[warp] + incl - v;
  *total = ws[32];
  __syncthreads();
  return r;
}

struct TkSmem {
  uint32_t* keys;              // [cap]
  uint32_t* idx;               // [cap] (merge stage) or nullptr (index = base + position)
  uint32_t* hist;              // [kBins]
  uint32_t* red;               // [64]
  unsigned long long* ws;      // [34]
  uint32_t* xchg;              // [8]
};

// Block-wide top-k of keys[0, L) (L > k), written in increasing position order through emit(pos,
// j) for the j-th selected element, j in [0, k).  gmax / gmin: the largest and smallest key of
// the list.  sm.hist must be all zero on entry; it is all zero again on return.
template <int NT, typename Emit>
__device__ void select_block(const TkSmem& sm, int L, int k, uint32_t gmax, uint32_t gmin, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // bits at and above `pos` are common to every key of the list
  int pos = (gmax == gmin) ? 0 : 32 - __clz(gmax ^ gmin);
  uint32_t prefix = pos >= 32 ? 0u : (gmax >> pos) << pos;
  int remaining = k;
  int cmp_shift = pos;
  while (pos > 0) {
    const int nbits = pos < kDigit ? pos : kDigit;
    const int shift = pos - nbits;
    const uint32_t dmask = (1u << nbits) - 1u;
    const uint32_t hmask = pos >= 32 ? 0u : ~((1u << pos) - 1u);
    for (int i = tid; i < L; i += NT) {
      const uint32_t kk = sm.keys[i];
      if ((kk & hmask) == prefix) atomicAdd(&sm.hist[(kk >> shift) & dmask], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane owns kBinsPerLane bins at descending positions; clears them for the next pass
      const int nb = 1 << nbits;
      uint32_t c[kBinsPerLane];
      uint32_t csum = 0;
#pragma unroll
      for (int u = 0; u < kBinsPerLane; ++u) {
        const int bin = nb - 1 - (kBinsPerLane * lane + u);
        c[u] = 0u;
        if (bin >= 0) {
          c[u] = sm.hist[bin];
          sm.hist[bin] = 0u;
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
      const uint32_t rem = static_cast<uint32_t>(remaining);
#pragma unroll
      for (int u = 0; u < kBinsPerLane; ++u) {
        if (above < rem && rem <= above + c[u]) {
          sm.xchg[2] = static_cast<uint32_t>(nb - 1 - (kBinsPerLane * lane + u));
          sm.xchg[3] = rem - above;
          sm.xchg[4] = c[u];
        }
        above += c[u];
      }
    }
    __syncthreads();
    prefix |= (sm.xchg[2] & dmask) << shift;
    remaining = static_cast<int>(min(sm.xchg[3], static_cast<uint32_t>(remaining)));
    const uint32_t bin_count = sm.xchg[4];
    pos = shift;
    cmp_shift = shift;
    // xchg is rewritten only after the next pass's first barrier, which every thread reaches
    // after these reads
    if (bin_count == static_cast<uint32_t>(remaining)) break;   // the threshold bin is taken whole
  }
  // selected: key >> cmp_shift above thr, or equal to it among the first `remaining` positions.
  // Each warp owns a contiguous range and walks it 32 consecutive keys at a time (conflict-free
  // shared-memory reads); ballots give every lane its rank inside the range, so the output keeps
  // increasing position order.
  const uint32_t thr = cmp_shift >= 32 ? 0u : prefix >> cmp_shift;
  constexpr int NW = NT / 32;
  const int per_w = ((L + NW - 1) / NW + 31) & ~31;
  const int w_lo = min(L, warp * per_w), w_hi = min(L, w_lo + per_w);
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t gt = 0, eq = 0;
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    uint32_t kt = 0;
    const bool in = i < w_hi;
    if (in) kt = cmp_shift >= 32 ? 0u : sm.keys[i] >> cmp_shift;
    gt += __popc(__ballot_sync(0xffffffffu, in && kt > thr));
    eq += __popc(__ballot_sync(0xffffffffu, in && kt == thr));
  }
  unsigned long long tot;
  // one value per warp enters the scan (lanes other than 0 contribute zero)
  const unsigned long long ex = block_excl_scan(lane == 0 ? (static_cast<unsigned long long>(gt) << 32) | eq : 0ull,
                                                sm.ws, &tot);
  const unsigned long long exw = __shfl_sync(0xffffffffu, ex, 0);
  uint32_t g_before = static_cast<uint32_t>(exw >> 32);
  uint32_t e_before = static_cast<uint32_t>(exw & 0xFFFFFFFFu);
  const uint32_t rem = static_cast<uint32_t>(remaining);
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    uint32_t kt = 0;
    const bool in = i < w_hi;
    if (in) kt = cmp_shift >= 32 ? 0u : sm.keys[i] >> cmp_shift;
    const uint32_t mg = __ballot_sync(0xffffffffu, in && kt > thr);
    const uint32_t me = __ballot_sync(0xffffffffu, in && kt == thr);
    const uint32_t g_rank = g_before + __popc(mg & lt_mask);
    const uint32_t e_rank = e_before + __popc(me & lt_mask);
    bool take = false;
    if (in && kt > thr) take = true;
    if (in && kt == thr) take = e_rank < rem;
    if (take) {
      const uint32_t j = g_rank + min(e_rank, rem);
      if (j < static_cast<uint32_t>(k)) emit(i, static_cast<int>(j));
    }
    g_before += __popc(mg);
    e_before += __popc(me);
  }
}

// Block-wide max and min of per-thread values; every thread gets both.  Ends with a barrier.
template <int NT>
__device__ __forceinline__ void block_minmax(const TkSmem& sm, uint32_t& kmax, uint32_t& kmin) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
  }
  if (lane == 0) {
    sm.red[warp] = kmax;
    sm.red[32 + warp] = kmin;
  }
  __syncthreads();
  uint32_t mx = lane < NT / 32 ? sm.red[lane] : 0u;
  uint32_t mn = lane < NT / 32 ? sm.red[32 + lane] : 0xFFFFFFFFu;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  kmax = mx;
  kmin = mn;
}

// keys[i] = order_key(src[i]) >> shift for i < L, eight independent loads in flight per thread;
// returns this thread's largest and smallest key through kmax / kmin.  shift 16: scores rounded
// to bf16, whose keys differ only in their top 16 bits (two radix passes instead of four).
template <int NT>
__device__ __forceinline__ void load_keys(uint32_t* keys, const float* src, int L, uint32_t& kmax, uint32_t& kmin,
                                          int shift) {
  constexpr int U = NT >= 1024 ? 8 : (NT >= 512 ? 16 : 32);   // loads in flight per thread
  for (int base = 0; base < L; base += NT * U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT + threadIdx.x;
      v[u] = i < L ? __ldg(src + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT + threadIdx.x;
      if (i < L) {
        const uint32_t kk = order_key(v[u]) >> shift;
        keys[i] = kk;
        kmax = max(kmax, kk);
        kmin = min(kmin, kk);
      }
    }
  }
}

__device__ __forceinline__ void clear_hist(const TkSmem& sm) {
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) sm.hist[i] = 0u;
}

__device__ __forceinline__ TkSmem carve(uint32_t* base, int cap, bool with_idx) {
  TkSmem s;
  s.keys = base;
  s.idx = with_idx ? base + cap : nullptr;
  s.hist = base + cap * (with_idx ? 2 : 1);
  s.red = s.hist + kBins;
  s.ws = reinterpret_cast<unsigned long long*>(s.red + 64);
  s.xchg = reinterpret_cast<uint32_t*>(s.ws + 34);
  return s;
}

// Stage 1: one CTA per (query, slice of slice_len candidates).  S == 1 writes the final row;
// S > 1 writes the slice's k candidates (key << 32 | index, index order, unused slots
// (0, kNoIndex)) to cand.
template <int NT>
__global__ void __launch_bounds__(NT) k_topk_slice(TopkArgs a, int S, int slice_len, int cap,
                                                   unsigned long long* cand) {
  extern __shared__ __align__(16) uint32_t tsm[];
  grid_dep_wait();
  grid_dep_launch();
  const TkSmem sm = carve(tsm, cap, false);
  const int tid = threadIdx.x;
  const long long qrel = blockIdx.x / S;
  const int sl = static_cast<int>(blockIdx.x % S);
  const long long qi = a.q_begin + qrel;
  const int n = n_visible(a.q_pos[qi], a.m, a.N);
  const int k = a.k;
  const int lo = sl * slice_len;
  const int L = max(0, min(n, lo + slice_len) - lo);
  if (S == 1) {
    int32_t* out = a.idx_out + qi * k;
    if (n <= k) {
      for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
      return;
    }
    if (L > cap) {                       // cannot happen with a valid launch; never index past cap
      if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, L);
      return;
    }
    const float* row = a.scores + (qi - a.score_row_offset) * static_cast<long long>(a.N);
    uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
    clear_hist(sm);
    load_keys<NT>(sm.keys, row + lo, L, kmax, kmin, a.key_shift);
    block_minmax<NT>(sm, kmax, kmin);
    select_block<NT>(sm, L, k, kmax, kmin, [&](int i, int j) { out[j] = lo + i; });
    return;
  }
  unsigned long long* crow = cand + (qrel * S + sl) * static_cast<long long>(k);
  if (L <= k) {
    const float* row = a.scores + (qi - a.score_row_offset) * static_cast<long long>(a.N);
    for (int i = tid; i < k; i += NT)
      crow[i] = i < L ? (static_cast<unsigned long long>(order_key(row[lo + i]) >> a.key_shift) << 32) |
                            static_cast<uint32_t>(lo + i)
                      : static_cast<unsigned long long>(kNoIndex);
    return;
  }
  if (L > cap) {
    if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, L);
    return;
  }
  const float* row = a.scores + (qi - a.score_row_offset) * static_cast<long long>(a.N);
  uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
  clear_hist(sm);
  load_keys<NT>(sm.keys, row + lo, L, kmax, kmin, a.key_shift);
  block_minmax<NT>(sm, kmax, kmin);
  select_block<NT>(sm, L, k, kmax, kmin, [&](int i, int j) {
    crow[j] = (static_cast<unsigned long long>(sm.keys[i]) << 32) | static_cast<uint32_t>(lo + i);
  });
}

// ------------------------------------------------------------------ one-stage cluster selection
// A row of S <= 16 slices is selected by one thread-block cluster of S CTAs (CTA r = slice r)
// instead of slices plus a merge: every radix pass adds the slices' local histograms through
// distributed shared memory, so all CTAs see the row's histogram and take the same decisions.
// Each CTA then counts its keys above the threshold and its ties, the CTAs exchange these counts,
// and each writes its selected entries at its own offset of the output row (lower slices first,
// so the row stays in increasing index order; ties go to the lower slices first, then to the
// smaller index inside a slice).  Same result as the two-stage path.
//
// The cluster barriers are hardware barriers that every thread of every CTA reaches the same
// number of times: the pass decisions come from the same summed histogram in every CTA, and no
// CTA leaves before the last barrier (not even on a failed range check, which only empties its
// slice), so no wait depends on a peer taking another path.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Words at the same shared-memory offset as `p` in CTA `rank` of this cluster.  The loads carry
// no memory clobber, so a lane's independent remote loads are all in flight together; they stay
// between the cluster barriers around them because those are volatile asm with a memory clobber.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  return ra;
}
__device__ __forceinline__ uint32_t ld_peer(const uint32_t* p, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(peer_addr(p, rank)));
  return v;
}
__device__ __forceinline__ uint4 ld_peer4(const uint32_t* p, uint32_t rank) {   // p 16-byte aligned
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(peer_addr(p, rank)));
  return v;
}

size_t cluster_smem(int cap) {
  return static_cast<size_t>(cap) * 4 + 2 * kBins * 4 + 64 * 4 + 34 * 8 + 8 * 4 + 4 * 4;
}

template <int NT>
__global__ void __launch_bounds__(NT) k_topk_cluster(TopkArgs a, int S, int slice_len, int cap) {
  extern __shared__ __align__(16) uint32_t tsm[];
  grid_dep_wait();
  grid_dep_launch();
  TkSmem sm;
  sm.keys = tsm;
  sm.idx = nullptr;
  uint32_t* hist2 = tsm + cap;                                  // [2][kBins], one per pass parity
  sm.hist = hist2;
  sm.red = hist2 + 2 * kBins;
  sm.ws = reinterpret_cast<unsigned long long*>(sm.red + 64);
  sm.xchg = reinterpret_cast<uint32_t*>(sm.ws + 34);
  uint32_t* pub = sm.xchg + 8;                                  // [0..1] key max / min, [2..3] counts
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const long long qrel = blockIdx.x / S;                        // a cluster = S consecutive blocks
  const long long qi = a.q_begin + qrel;
  const int n = n_visible(a.q_pos[qi], a.m, a.N);
  const int k = a.k;
  int32_t* out = a.idx_out + qi * k;
  if (n <= k) {                      // the same in every CTA of the cluster: no selection, no barrier
    if (rank == 0)
      for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
    return;
  }
  const int lo = static_cast<int>(rank) * slice_len;
  int L = max(0, min(n, lo + slice_len) - lo);
  if (L > cap) {                     // cannot happen with a valid launch; the CTA still takes part
    if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, L);
    L = 0;
  }
  for (int i = tid; i < 2 * kBins; i += NT) hist2[i] = 0u;
  const float* row = a.scores + (qi - a.score_row_offset) * static_cast<long long>(a.N);
  uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
  load_keys<NT>(sm.keys, row + lo, L, kmax, kmin, a.key_shift);
  block_minmax<NT>(sm, kmax, kmin);
  if (tid == 0) {
    pub[0] = kmax;
    pub[1] = kmin;
  }
  cluster_barrier();                                            // keys, zeroed histograms, max / min
  if (warp == 0) {                       // lane r reads CTA r's pair; one warp reduction
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
    if (lane < S) {
      mx = ld_peer(&pub[0], lane);
      mn = ld_peer(&pub[1], lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
      sm.xchg[0] = mx;
      sm.xchg[1] = mn;
    }
  }
  __syncthreads();
  const uint32_t gmax = sm.xchg[0], gmin = sm.xchg[1];

  int pos = (gmax == gmin) ? 0 : 32 - __clz(gmax ^ gmin);
  uint32_t prefix = pos >= 32 ? 0u : (gmax >> pos) << pos;
  int remaining = k;
  int cmp_shift = pos;
  int buf = 0;
  while (pos > 0) {
    const int nbits = pos < kDigit ? pos : kDigit;
    const int shift = pos - nbits;
    const uint32_t dmask = (1u << nbits) - 1u;
    const uint32_t hmask = pos >= 32 ? 0u : ~((1u << pos) - 1u);
    uint32_t* hist = hist2 + buf * kBins;
    for (int i = tid; i < L; i += NT) {
      const uint32_t kk = sm.keys[i];
      if ((kk & hmask) == prefix) atomicAdd(&hist[(kk >> shift) & dmask], 1u);
    }
    cluster_barrier();                                          // every slice's histogram of this pass
    if (warp == 0) {
      const int nb = 1 << nbits;
      uint32_t c[kBinsPerLane];
      uint32_t csum = 0;
      // lane's bins nb-1-8*lane-u (u = 0..7) are the 8 consecutive words from lo8 = nb-8-8*lane;
      // sums run over the CTAs in fixed order, so every CTA gets the same counts
#pragma unroll
      for (int u = 0; u < kBinsPerLane; ++u) c[u] = 0u;
      const int lo8 = nb - kBinsPerLane * (lane + 1);
      if (lo8 >= 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {                  // 4 bins at a time, 8 CTAs' loads in flight
#pragma unroll
          for (int r0 = 0; r0 < kClusterMax; r0 += kPeerBatch) {
            if (r0 >= S) break;
            uint4 v[kPeerBatch];
#pragma unroll
            for (int r = 0; r < kPeerBatch; ++r)
              if (r0 + r < S) v[r] = ld_peer4(&hist[lo8 + 4 * h], r0 + r);
#pragma unroll
            for (int r = 0; r < kPeerBatch; ++r) {
              if (r0 + r < S) {
                c[7 - 4 * h] += v[r].x; c[6 - 4 * h] += v[r].y;
                c[5 - 4 * h] += v[r].z; c[4 - 4 * h] += v[r].w;
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < kBinsPerLane; ++u) {
          const int bin = nb - 1 - (kBinsPerLane * lane + u);
          if (bin >= 0)
            for (int r = 0; r < S; ++r) c[u] += ld_peer(&hist[bin], r);
        }
      }
#pragma unroll
      for (int u = 0; u < kBinsPerLane; ++u) csum += c[u];
      // the other parity's histogram was last read by the peers before they reached this
      // pass's barrier: clear it for the next pass
      uint32_t* other = hist2 + (buf ^ 1) * kBins;
      for (int i = lane; i < kBins; i += 32) other[i] = 0u;
      uint32_t incl = csum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t above = incl - csum;
      const uint32_t rem = static_cast<uint32_t>(remaining);
#pragma unroll
      for (int u = 0; u < kBinsPerLane; ++u) {
        if (above < rem && rem <= above + c[u]) {
          sm.xchg[2] = static_cast<uint32_t>(nb - 1 - (kBinsPerLane * lane + u));
          sm.xchg[3] = rem - above;
          sm.xchg[4] = c[u];
        }
        above += c[u];
      }
    }
    __syncthreads();
    prefix |= (sm.xchg[2] & dmask) << shift;
    remaining = static_cast<int>(min(sm.xchg[3], static_cast<uint32_t>(remaining)));
    const uint32_t bin_count = sm.xchg[4];
    pos = shift;
    cmp_shift = shift;
    buf ^= 1;
    if (bin_count == static_cast<uint32_t>(remaining)) break;
  }

  // this slice's keys above the threshold (gt) and in it (eq), per warp and in total
  const uint32_t thr = cmp_shift >= 32 ? 0u : prefix >> cmp_shift;
  constexpr int NW = NT / 32;
  const int per_w = ((L + NW - 1) / NW + 31) & ~31;
  const int w_lo = min(L, warp * per_w), w_hi = min(L, w_lo + per_w);
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t gt = 0, eq = 0;
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    uint32_t kt = 0;
    const bool in = i < w_hi;
    if (in) kt = cmp_shift >= 32 ? 0u : sm.keys[i] >> cmp_shift;
    gt += __popc(__ballot_sync(0xffffffffu, in && kt > thr));
    eq += __popc(__ballot_sync(0xffffffffu, in && kt == thr));
  }
  unsigned long long tot;
  const unsigned long long ex = block_excl_scan(lane == 0 ? (static_cast<unsigned long long>(gt) << 32) | eq : 0ull,
                                                sm.ws, &tot);
  if (tid == 0) {
    pub[2] = static_cast<uint32_t>(tot >> 32);
    pub[3] = static_cast<uint32_t>(tot & 0xFFFFFFFFu);
  }
  cluster_barrier();                                            // every slice's counts
  const uint32_t rem = static_cast<uint32_t>(remaining);
  if (warp == 0) {
    // lane r < rank reads CTA r's counts.  Ties are taken greedily from the lowest slice, so the
    // lower slices together take min(their ties, rem) of them: this slice's output offset is
    // (their entries above the threshold) + min(their ties, rem)
    uint32_t g = 0u, e = 0u;
    if (static_cast<uint32_t>(lane) < rank) {
      g = ld_peer(&pub[2], lane);
      e = ld_peer(&pub[3], lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if (lane == 0) {
      sm.xchg[5] = g + min(e, rem);
      sm.xchg[6] = e;
    }
  }
  __syncthreads();
  const uint32_t out_base = sm.xchg[5], eq_lower = sm.xchg[6];
  const uint32_t my_eq = static_cast<uint32_t>(tot & 0xFFFFFFFFu);
  const uint32_t my_rem = rem > eq_lower ? min(rem - eq_lower, my_eq) : 0u;   // ties this slice takes
  const unsigned long long exw = __shfl_sync(0xffffffffu, ex, 0);
  uint32_t g_before = static_cast<uint32_t>(exw >> 32);
  uint32_t e_before = static_cast<uint32_t>(exw & 0xFFFFFFFFu);
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    uint32_t kt = 0;
    const bool in = i < w_hi;
    if (in) kt = cmp_shift >= 32 ? 0u : sm.keys[i] >> cmp_shift;
    const uint32_t mg = __ballot_sync(0xffffffffu, in && kt > thr);
    const uint32_t me = __ballot_sync(0xffffffffu, in && kt == thr);
    const uint32_t g_rank = g_before + __popc(mg & lt_mask);
    const uint32_t e_rank = e_before + __popc(me & lt_mask);
    bool take = false;
    if (in && kt > thr) take = true;
    if (in && kt == thr) take = e_rank < my_rem;
    if (take) {
      const uint32_t j = out_base + g_rank + min(e_rank, my_rem);
      if (j < static_cast<uint32_t>(k)) out[j] = lo + i;
    }
    g_before += __popc(mg);
    e_before += __popc(me);
  }
  cluster_barrier();                         // no CTA leaves while a peer may still read its counts
}

// Stage 2: one CTA per query merges the S * k candidates of its slices.
template <int NT>
__global__ void __launch_bounds__(NT) k_topk_merge(TopkArgs a, int S, int cap, const unsigned long long* cand) {
  extern __shared__ __align__(16) uint32_t tsm[];
  grid_dep_wait();
  grid_dep_launch();
  const TkSmem sm = carve(tsm, cap, true);
  const int tid = threadIdx.x;
  const long long qrel = blockIdx.x;
  const long long qi = a.q_begin + qrel;
  const int k = a.k;
  int32_t* out = a.idx_out + qi * k;
  const int n = n_visible(a.q_pos[qi], a.m, a.N);
  if (n <= k) {
    for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
    return;
  }
  const int total = S * k;
  if (total > cap) {
    if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, total);
    return;
  }
  // compact the valid candidates (they are already in increasing index order); each warp owns a
  // contiguous range, read 32 consecutive candidates at a time, all of them loaded up front so the
  // loads overlap
  const unsigned long long* crow = cand + qrel * static_cast<long long>(total);
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NT / 32;
  constexpr int UMAX = kMergeRounds;                // 32-candidate rounds per warp at most
  const int per_w = ((total + NW - 1) / NW + 31) & ~31;
  const int w_lo = min(total, warp * per_w), w_hi = min(total, w_lo + per_w);
  if (per_w > UMAX * 32) {               // cannot happen: the launch picks NT >= total / UMAX
    if (tid == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, per_w);
    return;
  }
  unsigned long long c[UMAX];
#pragma unroll
  for (int u = 0; u < UMAX; ++u) {
    const int i = w_lo + u * 32 + lane;
    c[u] = i < w_hi ? crow[i] : static_cast<unsigned long long>(kNoIndex);
  }
  uint32_t cnt = 0;
#pragma unroll
  for (int u = 0; u < UMAX; ++u)
    cnt += __popc(__ballot_sync(0xffffffffu, static_cast<uint32_t>(c[u] & 0xFFFFFFFFull) != kNoIndex));
  clear_hist(sm);
  unsigned long long tot;
  const unsigned long long exs = block_excl_scan(lane == 0 ? cnt : 0u, sm.ws, &tot);
  uint32_t p = static_cast<uint32_t>(__shfl_sync(0xffffffffu, exs, 0));
  uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
#pragma unroll
  for (int u = 0; u < UMAX; ++u) {
    const bool valid = static_cast<uint32_t>(c[u] & 0xFFFFFFFFull) != kNoIndex;
    const uint32_t m = __ballot_sync(0xffffffffu, valid);
    const uint32_t q = p + __popc(m & ((1u << lane) - 1u));
    if (valid && q < static_cast<uint32_t>(cap)) {
      const uint32_t kk = static_cast<uint32_t>(c[u] >> 32);
      sm.keys[q] = kk;
      sm.idx[q] = static_cast<uint32_t>(c[u] & 0xFFFFFFFFull);
      kmax = max(kmax, kk);
      kmin = min(kmin, kk);
    }
    p += __popc(m);
  }
  block_minmax<NT>(sm, kmax, kmin);
  const int L = static_cast<int>(min(tot, static_cast<unsigned long long>(cap)));
  if (L <= k) {                          // fewer valid candidates than k (n > k makes this rare)
    for (int i = tid; i < k; i += NT) out[i] = i < L ? static_cast<int32_t>(sm.idx[i]) : -1;
    return;
  }
  select_block<NT>(sm, L, k, kmax, kmin, [&](int i, int j) { out[j] = static_cast<int32_t>(sm.idx[i]); });
}

size_t slice_smem(int cap, bool with_idx) {
  return static_cast<size_t>(cap) * 4 * (with_idx ? 2 : 1) + kBins * 4 + 64 * 4 + 34 * 8 + 8 * 4;
}

}  // namespace

// Slice length for Q queries of N candidates: one slice when the batch alone fills the GPU,
// otherwise halved (down to kMinSlice) until about kTargetCtas first-stage CTAs run, as long as
// the merge still holds every candidate.  Depends only on (Q, N, k), never on the device.
int topk_slice_len(int Q, int N, int k) {
  int len = kSlice;
  auto slices = [&](int l) { return (N + l - 1) / l; };
  while (len > kMinSlice && static_cast<long long>(Q) * slices(len) < kTargetCtas && slices(len / 2) > 1 &&
         static_cast<long long>(slices(len / 2)) * k <= kMergeCap)
    len /= 2;
  return len;
}

int topk_slices(int Q, int N, int k) {
  const int len = topk_slice_len(Q, N, k);
  return N <= len ? 1 : (N + len - 1) / len;
}

size_t topk_candidate_bytes(int Q, int N, int k) {
  const int S = topk_slices(Q, N, k);
  return S > 1 ? static_cast<size_t>(Q) * S * k * sizeof(unsigned long long) : 0;
}

template <int NT>
cudaError_t launch_slice(const TopkArgs& a, int S, int len, int cap, unsigned long long* cand, cudaStream_t s) {
  const size_t smem = slice_smem(cap, false);
  cudaError_t e = cudaFuncSetAttribute(k_topk_slice<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(k_topk_slice<NT>, dim3(static_cast<unsigned>(a.q_count) * S), dim3(NT), smem, s, a, S, len, cap,
                  cand);
}

template <int NT>
cudaError_t launch_merge(const TopkArgs& a, int S, int cap, const unsigned long long* cand, cudaStream_t s) {
  const size_t smem = slice_smem(cap, true);
  cudaError_t e = cudaFuncSetAttribute(k_topk_merge<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(k_topk_merge<NT>, dim3(static_cast<unsigned>(a.q_count)), dim3(NT), smem, s, a, S, cap, cand);
}

// One cluster of S CTAs per query (S <= 16).  Returns cudaErrorNotSupported, before launching,
// when the device cannot hold such a cluster.
template <int NT>
cudaError_t launch_cluster(const TopkArgs& a, int S, int len, cudaStream_t s) {
  const size_t smem = cluster_smem(len);
  cudaError_t e = cudaFuncSetAttribute(k_topk_cluster<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (S > 8) {                       // above the portable size; a device that cannot is not asked
    e = cudaFuncSetAttribute(k_topk_cluster<NT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return cudaErrorNotSupported;
    }
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.q_count) * S);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, k_topk_cluster<NT>, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorNotSupported;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_topk_cluster<NT>, a, S, len, len);
}

cudaError_t launch_topk(const TopkArgs& a, void* cand_ws, cudaStream_t s, int* launches) {
  if (a.q_count == 0) return cudaSuccess;
  const int len = topk_slice_len(a.q_count, a.N, a.k);
  const int S = topk_slices(a.q_count, a.N, a.k);
  if (S > 1 && CSA_TOPK_CLUSTER && a.N <= kClusterMax * kSlice) {
    // one-stage selection by a cluster per query (at most 16 slices: rows cut for the two-stage
    // path into more are re-cut into 16 of at most 32768); falls through to the two stages only
    // when the device cannot hold the cluster (the result is the same either way)
    int cl_len = len, cl_S = S;
    if (S > kClusterMax && CSA_TOPK_CLUSTER_LONG) {
      cl_len = ((a.N + kClusterMax - 1) / kClusterMax + kMinSlice - 1) / kMinSlice * kMinSlice;
      cl_S = (a.N + cl_len - 1) / cl_len;
    }
    const cudaError_t e = cl_S <= kClusterMax ? launch_cluster<CSA_TOPK_CLUSTER_NT>(a, cl_S, cl_len, s)
                                              : cudaErrorNotSupported;
    if (e != cudaErrorNotSupported) {
      ++*launches;
      return e;
    }
    (void)cudaGetLastError();
  }
  if (S > 1 && (cand_ws == nullptr || static_cast<long long>(S) * a.k > kMergeCap)) return cudaErrorInvalidValue;
  const int cap1 = S == 1 ? ((a.N + 3) & ~3) : len;
  unsigned long long* cand = static_cast<unsigned long long*>(cand_ws);
  // threads per selecting CTA: whole rows (many queries, one slice each) on 256 threads, several
  // CTAs per SM; the slices of a small batch's long rows on 1024 (measured: 1024 threads were 2.5x
  // slower than 256 on prefill rows; 256 and 512 threads 20% and 8% slower than 1024 on the 8192-key
  // decode slices).  The result does not depend on the choice.
  cudaError_t e = S == 1 ? launch_slice<256>(a, S, len, cap1, cand, s) : launch_slice<1024>(a, S, len, cap1, cand, s);
  ++*launches;
  if (e != cudaSuccess || S == 1) return e;
  const int total = S * a.k;
  const int cap2 = (total + 3) & ~3;
  // the fewest threads that still hold every candidate in registers (kMergeRounds per warp)
  if (total <= 256 * kMergeRounds) e = launch_merge<256>(a, S, cap2, cand, s);
  else if (total <= 512 * kMergeRounds) e = launch_merge<512>(a, S, cap2, cand, s);
  else e = launch_merge<1024>(a, S, cap2, cand, s);
  ++*launches;
  return e;
}

}  // namespace csa
