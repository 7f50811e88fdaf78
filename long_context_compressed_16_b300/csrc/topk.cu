// Per-query top-k over the visible indexer scores ("DeepSeek V4 模型技术大全", CSA path, the TopK_k
// equation), ties to the smaller entry index.
//
// Radix select on order-preserving 32-bit keys of the fp32 scores, three digit passes
// (11 / 11 / 10 bits).  One thread-block cluster of CS CTAs owns one query: each CTA keeps a
// contiguous slice of the candidates in shared memory, builds its digit histogram with shared
// atomics, and every CTA sums the CS histograms through distributed shared memory, so all CTAs
// agree on the digit without a second kernel.  The final compaction writes, in increasing entry
// index, the entries above the k-th score and then the ties taken in increasing index, so the
// output is deterministic and depends only on the query's own scores.
#include <cooperative_groups.h>

#include "common.cuh"

namespace csa {

namespace {

namespace cg = cooperative_groups;

constexpr int TK_THREADS = 1024;
constexpr int kMaxSlice = 32768;     // candidates held per CTA (128 KB of keys)

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide scan of 64-bit sums.  ws: 33 slots of shared memory.
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
    unsigned long long x = lane < nwarps ? ws[lane] : 0ull;
    unsigned long long xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += y;
    }
    ws[lane] = xi - x;          // exclusive prefix of warp totals
    if (lane == 31) ws[32] = xi;
  }
  __syncthreads();
  const unsigned long long r = ws[warp] + incl - v;
  *total = ws[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(TK_THREADS) k_topk(TopkArgs a, int CS, int cap) {
  extern __shared__ __align__(16) uint32_t tsm[];
  uint32_t* keys = tsm;                                       // [cap]
  uint32_t* hist = tsm + cap;                                 // [2][2048]
  unsigned long long* ws = reinterpret_cast<unsigned long long*>(hist + 4096);   // [33]
  uint32_t* xchg = reinterpret_cast<uint32_t*>(ws + 34);     // [0] gt count, [1] eq count, [2..3] sel

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x;
  const long long qi = a.q_begin + blockIdx.x / CS;          // flattened query index
  const int t = a.q_pos[qi];
  const int n = n_visible(t, a.m, a.N);
  int32_t* out = a.idx_out + qi * a.k;

  if (n <= a.k) {      // every visible entry is selected; no cluster communication
    if (rank == 0)
      for (int i = tid; i < a.k; i += TK_THREADS) out[i] = i < n ? i : -1;
    return;
  }

  const float* row = a.scores + (qi - a.score_row_offset) * static_cast<long long>(a.N);
  const int lo = static_cast<int>(static_cast<long long>(n) * rank / CS);
  const int hi = static_cast<int>(static_cast<long long>(n) * (rank + 1) / CS);
  const int L = hi - lo;
  for (int i = tid; i < L; i += TK_THREADS) keys[i] = order_key(row[lo + i]);

  if (tid == 0) { xchg[2] = 0; xchg[3] = 0; }
  uint32_t prefix = 0, pmask = 0;
  int remaining = a.k;
  for (int p = 0; p < 3; ++p) {
    const int shift = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const int nb = p == 2 ? 1024 : 2048;
    uint32_t* h = hist + (p & 1) * 2048;
    for (int i = tid; i < 2048; i += TK_THREADS) h[i] = 0;
    __syncthreads();
    // warp-aggregated histogram: the scores of one query crowd into a few leading-digit bins, so
    // lanes that hit the same bin are merged with a match before one atomic per distinct bin
    const int rounds = (L + TK_THREADS - 1) / TK_THREADS;
    for (int rd = 0; rd < rounds; ++rd) {
      const int i = rd * TK_THREADS + tid;
      uint32_t bin = 0xFFFFFFFFu;
      if (i < L) {
        const uint32_t kk = keys[i];
        if ((kk & pmask) == prefix) bin = (kk >> shift) & static_cast<uint32_t>(nb - 1);
      }
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && (tid & 31) == __ffs(grp) - 1) atomicAdd(&h[bin], static_cast<uint32_t>(__popc(grp)));
    }
    cluster.sync();
    // thread tid owns the bins at descending positions 2*tid and 2*tid+1
    const int bA = nb - 1 - 2 * tid, bB = nb - 2 - 2 * tid;
    uint32_t cA = 0, cB = 0;
    for (int r = 0; r < CS; ++r) {
      const uint32_t* rh = cluster.map_shared_rank(h, r);
      if (bA >= 0) cA += rh[bA];
      if (bB >= 0) cB += rh[bB];
    }
    unsigned long long tot;
    const unsigned long long above = block_excl_scan(cA + cB, ws, &tot);
    const unsigned long long rem = static_cast<unsigned long long>(remaining);
    if (bA >= 0 && above < rem && rem <= above + cA) {
      xchg[2] = static_cast<uint32_t>(bA);
      xchg[3] = static_cast<uint32_t>(rem - above);
    } else if (bB >= 0 && above + cA < rem && rem <= above + cA + cB) {
      xchg[2] = static_cast<uint32_t>(bB);
      xchg[3] = static_cast<uint32_t>(rem - above - cA);
    }
    __syncthreads();
    prefix |= xchg[2] << shift;
    pmask |= static_cast<uint32_t>(nb - 1) << shift;
    remaining = static_cast<int>(xchg[3]);
    __syncthreads();
  }
  const uint32_t thr = prefix;     // key of the k-th largest score; `remaining` ties are taken

  // counts per thread over a contiguous run of the slice (keeps index order)
  const int per = (L + TK_THREADS - 1) / TK_THREADS;
  const int i_lo = min(L, tid * per), i_hi = min(L, i_lo + per);
  uint32_t gt = 0, eq = 0;
  for (int i = i_lo; i < i_hi; ++i) {
    const uint32_t kk = keys[i];
    gt += kk > thr;
    eq += kk == thr;
  }
  unsigned long long tot;
  const unsigned long long ex = block_excl_scan((static_cast<unsigned long long>(gt) << 32) | eq, ws, &tot);
  if (tid == 0) {
    xchg[0] = static_cast<uint32_t>(tot >> 32);
    xchg[1] = static_cast<uint32_t>(tot & 0xFFFFFFFFu);
  }
  cluster.sync();
  uint32_t gt_off = 0, eq_off = 0;
  for (int r = 0; r < rank; ++r) {
    const uint32_t* rx = cluster.map_shared_rank(xchg, r);
    gt_off += rx[0];
    eq_off += rx[1];
  }
  uint32_t g_rank = gt_off + static_cast<uint32_t>(ex >> 32);
  uint32_t e_rank = eq_off + static_cast<uint32_t>(ex & 0xFFFFFFFFu);
  const uint32_t base_eq = static_cast<uint32_t>(a.k - min(remaining, a.k));
  for (int i = i_lo; i < i_hi; ++i) {
    const uint32_t kk = keys[i];
    if (kk > thr) {
      if (g_rank < base_eq) out[g_rank] = lo + i;
      ++g_rank;
    } else if (kk == thr) {
      if (e_rank < static_cast<uint32_t>(remaining)) out[base_eq + e_rank] = lo + i;
      ++e_rank;
    }
  }
  cluster.sync();   // no CTA leaves while another may still read its shared memory
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, int* launches) {
  if (a.q_count == 0) return cudaSuccess;
  // one CTA holds up to 32768 candidates in shared memory; longer rows spread over a cluster
  int CS = (a.N + kMaxSlice - 1) / kMaxSlice;
  if (CS < 1) CS = 1;
  if (CS > 8) CS = 8;
  const int cap = ((a.N + CS - 1) / CS + 3) & ~3;   // keeps the 64-bit scan slots 8-byte aligned
  if (cap > kMaxSlice) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(cap) * 4 + 4096 * 4 + 34 * 8 + 16;
  cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.q_count) * CS, 1, 1);
  cfg.blockDim = dim3(TK_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_topk, a, CS, cap);
  ++*launches;
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace csa
