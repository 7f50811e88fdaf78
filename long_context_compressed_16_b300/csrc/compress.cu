// Token-level compressor: softmax-gated weighted sum over m (HCA) or 2m overlapped (CSA) rows,
// fused with RMSNorm and partial RoPE.  ("DeepSeek V4 模型技术大全", CSA path, Softmax_row and
// C^Comp equations; HCA path, S and C^Comp equations.)
//
// Pure HBM stream: every input row is read exactly once (entry i owns a-block i and b-block i-1),
// in 16-byte vectors of 8 channels; a thread owns 8 channels of one entry.
//   - CSA with m = 4 (the method's ratio): an exact two-pass softmax per channel over the entry's
//     8 rows (4 for entry 0): the maximum first, then one hardware exp2 per logit (csa4_entry).
//     Whole sequences run in k_compress_staged, which bulk-copies a block of entries' rows into
//     shared memory first; cache appends run the same routine in k_compress, so both agree bit
//     for bit.
//   - Other cases (HCA, m' = 128; other m): the softmax runs online over chunks of 2 (CSA) or 4
//     (HCA) rows in k_compress; long blocks are split over row groups whose partial (max, sum,
//     acc) are merged in shared memory in fixed order, so results are deterministic.
#include "common.cuh"
#include "tc.cuh"

namespace csa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;


__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// One online-softmax step over the nr (<= RC) rows in zv / cv (8 channels each, bf16 pairs),
// with their bias rows (or null).  Both compressor kernels run exactly this code, so their
// results agree bit for bit.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int RC>
__device__ __forceinline__ void softmax_step(const uint4* zv, const uint4* cv, const float* const* bptr, int nr,
                                             float* mx, float* sm, float* acc) {
  // the rows' biases, 8 channels each, loaded once per row (zero without a bias)
  float bias[RC][8];
#pragma unroll
  for (int u = 0; u < RC; ++u) {
    float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
    if (u < nr && bptr[u] != nullptr) {
      b0 = __ldg(reinterpret_cast<const float4*>(bptr[u]));
      b1 = __ldg(reinterpret_cast<const float4*>(bptr[u] + 4));
    }
    bias[u][0] = b0.x; bias[u][1] = b0.y; bias[u][2] = b0.z; bias[u][3] = b0.w;
    bias[u][4] = b1.x; bias[u][5] = b1.y; bias[u][6] = b1.z; bias[u][7] = b1.w;
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float z[RC], cvals[RC];
    float cm = mx[c];
#pragma unroll
    for (int u = 0; u < RC; ++u) {
      if (u < nr) {
        const uint32_t zw = (&zv[u].x)[c >> 1];
        const uint32_t cw = (&cv[u].x)[c >> 1];
        const float zb = (c & 1) ? bf16hi(zw) : bf16lo(zw);
        cvals[u] = (c & 1) ? bf16hi(cw) : bf16lo(cw);
        z[u] = (zb + bias[u][c]) * kLog2e;
        cm = fmaxf(cm, z[u]);
      }
    }
    const float alpha = (mx[c] == -INFINITY) ? 0.f : ex2_approx(mx[c] - cm);
    float s = sm[c] * alpha, ac = acc[c] * alpha;
#pragma unroll
    for (int u = 0; u < RC; ++u) {
      if (u < nr) {
        const float p = ex2_approx(z[u] - cm);
        s += p;
        ac = fmaf(p, cvals[u], ac);
      }
    }
    mx[c] = cm; sm[c] = s; acc[c] = ac;
  }
}

// CSA entry with m = 4 (R = 4 rows for entry 0, 8 otherwise), exact two-pass softmax per channel:
// the maximum over all R logits first, then one exp2 per logit and the weighted sum, with no
// rescaling.  fetch(r, zv, cv) returns row r (a-rows 0..3, then b-rows 4..7) for this thread's 8
// channels; it is called in both passes.  Both kernels that compress m = 4 CSA entries (the
// staged whole-sequence kernel and the cache-append path of k_compress) run exactly this code.
template <int R, class Fetch>
__device__ __forceinline__ void csa4_entry(Fetch fetch, const float* bias_a, const float* bias_b, int d, int c0,
                                           float* outv) {
  auto logits = [&](int r, const uint4& zv, float* z) {
    const float* bp = r < 4 ? bias_a : bias_b;
    float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
    if (bp != nullptr) {
      b0 = __ldg(reinterpret_cast<const float4*>(bp + static_cast<size_t>(r & 3) * d + c0));
      b1 = __ldg(reinterpret_cast<const float4*>(bp + static_cast<size_t>(r & 3) * d + c0 + 4));
    }
    z[0] = (bf16lo(zv.x) + b0.x) * kLog2e; z[1] = (bf16hi(zv.x) + b0.y) * kLog2e;
    z[2] = (bf16lo(zv.y) + b0.z) * kLog2e; z[3] = (bf16hi(zv.y) + b0.w) * kLog2e;
    z[4] = (bf16lo(zv.z) + b1.x) * kLog2e; z[5] = (bf16hi(zv.z) + b1.y) * kLog2e;
    z[6] = (bf16lo(zv.w) + b1.z) * kLog2e; z[7] = (bf16hi(zv.w) + b1.w) * kLog2e;
  };
  float mx[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) mx[c] = -INFINITY;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    uint4 zv, cv;
    fetch(r, zv, cv);
    float z[8];
    logits(r, zv, z);
#pragma unroll
    for (int c = 0; c < 8; ++c) mx[c] = fmaxf(mx[c], z[c]);
  }
  float sm[8], ac[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) { sm[c] = 0.f; ac[c] = 0.f; }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    uint4 zv, cv;
    fetch(r, zv, cv);
    float z[8];
    logits(r, zv, z);
    const float cvals[8] = {bf16lo(cv.x), bf16hi(cv.x), bf16lo(cv.y), bf16hi(cv.y),
                            bf16lo(cv.z), bf16hi(cv.z), bf16lo(cv.w), bf16hi(cv.w)};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float p = ex2_approx(z[c] - mx[c]);
      sm[c] += p;
      ac[c] = fmaf(p, cvals[c], ac[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) outv[c] = ac[c] / sm[c];
}

// RMSNorm over the entry's d channels (the TPE threads of one entry; every thread of the block
// takes part), gamma, RoPE at position m*i + pos_shift, bf16 store.  `writer`: this thread holds
// a finished outv.  `red`: shared scratch of one float per warp (used when TPE > 32).
__device__ __forceinline__ void norm_rope_store(const CompressArgs& a, float* outv, bool writer, int b, int i,
                                                int c0, int TPE, float* red) {
  const int tid = threadIdx.x;
  const int d = a.d;
  if (a.norm) {
    float ss = 0.f;
    if (writer) {
#pragma unroll
      for (int c = 0; c < 8; ++c) ss = fmaf(outv[c], outv[c], ss);
    }
    const int lanes = TPE < 32 ? TPE : 32;
    for (int o = lanes >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (TPE > 32) {
      __syncthreads();
      if ((tid & 31) == 0) red[tid >> 5] = ss;
      __syncthreads();
      const int w0 = (tid / TPE) * (TPE >> 5);
      ss = 0.f;
      for (int k = 0; k < (TPE >> 5); ++k) ss += red[w0 + k];
    }
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + a.eps);
#pragma unroll
    for (int c = 0; c < 8; ++c) outv[c] *= inv;
  }
  if (!writer) return;
  if (a.gamma != nullptr) {
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0 + 4));
    outv[0] *= g0.x; outv[1] *= g0.y; outv[2] *= g0.z; outv[3] *= g0.w;
    outv[4] *= g1.x; outv[5] *= g1.y; outv[6] *= g1.z; outv[7] *= g1.w;
  }
  if (a.rope && c0 >= d - a.rp.r) {
    const double pos = static_cast<double>(static_cast<long long>(a.m) * i + a.pos_shift);
    const int j0 = (c0 - (d - a.rp.r)) >> 1;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float cs, sn;
      rope_cos_sin(pos, a.rp.inv_freq[j0 + p], cs, sn);
      const float x0 = outv[2 * p], x1 = outv[2 * p + 1];
      outv[2 * p] = x0 * cs - x1 * sn;
      outv[2 * p + 1] = x0 * sn + x1 * cs;
    }
  }
  uint4 o;
  o.x = pack_bf16x2(outv[0], outv[1]);
  o.y = pack_bf16x2(outv[2], outv[3]);
  o.z = pack_bf16x2(outv[4], outv[5]);
  o.w = pack_bf16x2(outv[6], outv[7]);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  *reinterpret_cast<uint4*>(out + (static_cast<size_t>(b) * a.out_N + i) * d + c0) = o;
}

// kRowChunk: rows loaded per round (one online-softmax step); measured best at 2 for the
// overlapped 2m = 8 rows and at 4 for the 128 rows of an HCA block.
template <int kRowChunk>
__global__ void __launch_bounds__(256) k_compress(CompressArgs a, int RS, int EPC) {
  extern __shared__ float smem[];
  grid_dep_wait();
  grid_dep_launch();
  const int TPE = a.d >> 3;
  const int tid = threadIdx.x;
  const int cg = tid % TPE;
  const int rg = (tid / TPE) % RS;
  const int e = tid / (TPE * RS);
  const long long total = static_cast<long long>(a.B) * a.N;
  const long long gidx = static_cast<long long>(blockIdx.x) * EPC + e;
  const bool active = gidx < total;
  const int b = active ? static_cast<int>(gidx / a.N) : 0;
  const int i = active ? a.i_begin + static_cast<int>(gidx % a.N) : 0;
  const int c0 = cg * 8;
  const int d = a.d;

  float mx[8], sm[8], acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) { mx[c] = -INFINITY; sm[c] = 0.f; acc[c] = 0.f; }

  const bool csa4 = a.overlap && a.m == 4;        // RS = 1 here: one thread holds all 8 rows
  if (active && csa4) {
    const __nv_bfloat16* Za = static_cast<const __nv_bfloat16*>(a.Za);
    const __nv_bfloat16* Ca = static_cast<const __nv_bfloat16*>(a.Ca);
    const __nv_bfloat16* Zb = static_cast<const __nv_bfloat16*>(a.Zb);
    const __nv_bfloat16* Cb = static_cast<const __nv_bfloat16*>(a.Cb);
    const __nv_bfloat16* rZa = static_cast<const __nv_bfloat16*>(a.ring.Za);
    const __nv_bfloat16* rCa = static_cast<const __nv_bfloat16*>(a.ring.Ca);
    const __nv_bfloat16* rZb = static_cast<const __nv_bfloat16*>(a.ring.Zb);
    const __nv_bfloat16* rCb = static_cast<const __nv_bfloat16*>(a.ring.Cb);
    auto fetch = [&](int r, uint4& zv, uint4& cv) {
      const bool isb = r >= 4;
      // token indices stay below 2^31 (checked by the host), so 32-bit arithmetic: a 64-bit
      // remainder is a long software sequence on the GPU
      const int tok = isb ? 4 * (i - 1) + (r - 4) : 4 * i + r;
      if (tok >= a.t0) {
        const size_t off = (static_cast<size_t>(b) * a.T + (tok - a.t0)) * d + c0;
        zv = ldg_nc((isb ? Zb : Za) + off);
        cv = ldg_nc((isb ? Cb : Ca) + off);
      } else {
        const uint32_t slot = static_cast<uint32_t>(tok) % static_cast<uint32_t>(a.ring.R);
        const size_t off = (static_cast<size_t>(b) * a.ring.R + slot) * d + c0;
        zv = ldg_nc((isb ? rZb : rZa) + off);
        cv = ldg_nc((isb ? rCb : rCa) + off);
      }
    };
    float o4[8];
    if (i >= 1) csa4_entry<8>(fetch, a.bias_a, a.bias_b, d, c0, o4);
    else csa4_entry<4>(fetch, a.bias_a, a.bias_b, d, c0, o4);
#pragma unroll
    for (int c = 0; c < 8; ++c) { mx[c] = 0.f; sm[c] = 1.f; acc[c] = o4[c]; }   // outv = acc / sm below
  } else if (active) {
    const int R = a.m + ((a.overlap && i >= 1) ? a.m : 0);
    const int per = (R + RS - 1) / RS;
    const int r_lo = rg * per;
    const int r_hi = min(R, r_lo + per);
    const __nv_bfloat16* Za = static_cast<const __nv_bfloat16*>(a.Za);
    const __nv_bfloat16* Ca = static_cast<const __nv_bfloat16*>(a.Ca);
    const __nv_bfloat16* Zb = static_cast<const __nv_bfloat16*>(a.Zb);
    const __nv_bfloat16* Cb = static_cast<const __nv_bfloat16*>(a.Cb);
    const __nv_bfloat16* rZa = static_cast<const __nv_bfloat16*>(a.ring.Za);
    const __nv_bfloat16* rCa = static_cast<const __nv_bfloat16*>(a.ring.Ca);
    const __nv_bfloat16* rZb = static_cast<const __nv_bfloat16*>(a.ring.Zb);
    const __nv_bfloat16* rCb = static_cast<const __nv_bfloat16*>(a.ring.Cb);
    for (int r0 = r_lo; r0 < r_hi; r0 += kRowChunk) {
      const int nr = min(kRowChunk, r_hi - r0);
      uint4 zv[kRowChunk], cv[kRowChunk];
      const float* bptr[kRowChunk];
#pragma unroll
      for (int u = 0; u < kRowChunk; ++u) {
        bptr[u] = nullptr;
        if (u < nr) {
          const int r = r0 + u;
          const bool isb = r >= a.m;
          const int j = isb ? r - a.m : r;
          const int tok = isb ? a.m * (i - 1) + j : a.m * i + j;     // < 2^31 (checked by the host)
          if (tok >= a.t0) {              // a row of this call's chunk
            const size_t off = (static_cast<size_t>(b) * a.T + (tok - a.t0)) * d + c0;
            zv[u] = ldg_nc((isb ? Zb : Za) + off);
            cv[u] = ldg_nc((isb ? Cb : Ca) + off);
          } else {                        // an earlier token: the tail ring, slot tok mod R
            const uint32_t slot = static_cast<uint32_t>(tok) % static_cast<uint32_t>(a.ring.R);
            const size_t off = (static_cast<size_t>(b) * a.ring.R + slot) * d + c0;
            zv[u] = ldg_nc((isb ? rZb : rZa) + off);
            cv[u] = ldg_nc((isb ? rCb : rCa) + off);
          }
          const float* bp = isb ? a.bias_b : a.bias_a;
          if (bp != nullptr) bptr[u] = bp + static_cast<size_t>(j) * d + c0;
        }
      }
      softmax_step<kRowChunk>(zv, cv, bptr, nr, mx, sm, acc);
    }
  }

  // merge row groups (fixed order)
  float outv[8];
  if (RS > 1) {
    float* part = smem;  // [EPC][RS][TPE][8][3]
    const size_t base = ((static_cast<size_t>(e) * RS + rg) * TPE + cg) * 24;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      part[base + c * 3 + 0] = mx[c];
      part[base + c * 3 + 1] = sm[c];
      part[base + c * 3 + 2] = acc[c];
    }
    __syncthreads();
    if (rg == 0) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float M = -INFINITY;
        for (int g = 0; g < RS; ++g) {
          const size_t bg = ((static_cast<size_t>(e) * RS + g) * TPE + cg) * 24;
          M = fmaxf(M, part[bg + c * 3]);
        }
        float S = 0.f, A = 0.f;
        for (int g = 0; g < RS; ++g) {
          const size_t bg = ((static_cast<size_t>(e) * RS + g) * TPE + cg) * 24;
          const float mg = part[bg + c * 3];
          const float f = (mg == -INFINITY) ? 0.f : exp2f(mg - M);
          S = fmaf(part[bg + c * 3 + 1], f, S);
          A = fmaf(part[bg + c * 3 + 2], f, A);
        }
        outv[c] = A / S;
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) outv[c] = acc[c] / sm[c];
  }

  float* red = smem + (RS > 1 ? static_cast<size_t>(EPC) * RS * TPE * 24 : 0);
  norm_rope_store(a, outv, active && rg == 0, b, i, c0, TPE, red);
}

// Whole-sequence CSA compression (overlap, m = 4), staged: a CTA owns EPC consecutive entries
// i0 .. i1-1 of one sequence, whose a-rows (tokens m i0 .. m i1 - 1 of Ca, Za) and b-rows (tokens
// m (i0-1) .. m (i1-1) - 1 of Cb, Zb) are four contiguous runs.  One thread issues four bulk
// copies into shared memory on one mbarrier, so a whole block's rows are in flight at once (the
// per-thread loads of k_compress leave too few bytes in flight to reach HBM bandwidth); then every
// thread runs csa4_entry and the same epilogue as the cache-append path of k_compress, so the
// results agree bit for bit.
// Shared layout: [Za | Ca | Zb | Cb] regions of EPC*m rows x d bf16 (b-region slot e holds the
// b-block of entry i0 + e), then one float per warp for the norm, then the mbarrier.
__global__ void __launch_bounds__(256) k_compress_staged(CompressArgs a, int EPC) {
  extern __shared__ __align__(128) unsigned char sraw[];
  grid_dep_wait();
  grid_dep_launch();
  const int TPE = a.d >> 3;
  const int tid = threadIdx.x;
  const int cg = tid % TPE;
  const int e = tid / TPE;
  const int m = a.m, d = a.d;
  const int nblk = (a.N + EPC - 1) / EPC;
  const int b = static_cast<int>(blockIdx.x / nblk);
  const int i0 = static_cast<int>(blockIdx.x % nblk) * EPC;
  const int i1 = min(a.N, i0 + EPC);
  const size_t region = static_cast<size_t>(EPC) * m * d;          // elements per region
  __nv_bfloat16* sZa = reinterpret_cast<__nv_bfloat16*>(sraw);
  __nv_bfloat16* sCa = sZa + region;
  __nv_bfloat16* sZb = sCa + region;
  __nv_bfloat16* sCb = sZb + region;
  float* red = reinterpret_cast<float*>(sCb + region);
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 8);
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t rowb = static_cast<uint32_t>(d) * 2;
    const int e_lo = i0 == 0 ? 1 : 0;                  // entry 0 has no b-block
    const uint32_t abytes = static_cast<uint32_t>(i1 - i0) * m * rowb;
    const uint32_t bbytes = static_cast<uint32_t>(i1 - i0 - e_lo) * m * rowb;
    tc::mbar_arrive_expect_tx(bar, 2 * abytes + 2 * bbytes);
    const size_t aoff = (static_cast<size_t>(b) * a.T + static_cast<size_t>(m) * i0) * d;
    tc::bulk_load(sZa, static_cast<const __nv_bfloat16*>(a.Za) + aoff, abytes, bar);
    tc::bulk_load(sCa, static_cast<const __nv_bfloat16*>(a.Ca) + aoff, abytes, bar);
    if (bbytes > 0) {
      const size_t boff = (static_cast<size_t>(b) * a.T + static_cast<size_t>(m) * (i0 + e_lo - 1)) * d;
      const size_t soff = static_cast<size_t>(e_lo) * m * d;
      tc::bulk_load(sZb + soff, static_cast<const __nv_bfloat16*>(a.Zb) + boff, bbytes, bar);
      tc::bulk_load(sCb + soff, static_cast<const __nv_bfloat16*>(a.Cb) + boff, bbytes, bar);
    }
  }
  // every thread observes the copies' completion; the block leaves together if any wait gave up
  const bool got = tc::mbar_wait(bar, 0, nullptr, 1000000000ull);
  if (!__syncthreads_and(got)) return;

  const int i = i0 + e;
  const bool active = e < EPC && i < i1;
  const int c0 = cg * 8;
  float outv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (active) {
    const uint32_t base = (static_cast<uint32_t>(e) * 4) * d + c0;     // element offset of row 0
    auto fetch = [&](int r, uint4& zv, uint4& cv) {
      const uint32_t off = base + static_cast<uint32_t>(r & 3) * d;
      zv = *reinterpret_cast<const uint4*>((r < 4 ? sZa : sZb) + off);
      cv = *reinterpret_cast<const uint4*>((r < 4 ? sCa : sCb) + off);
    };
    if (i >= 1) csa4_entry<8>(fetch, a.bias_a, a.bias_b, d, c0, outv);
    else csa4_entry<4>(fetch, a.bias_a, a.bias_b, d, c0, outv);
  }
  norm_rope_store(a, outv, active, b, i, c0, TPE, red);
}

// One 16-byte vector per thread; blockIdx.y is the job.  Every job's row width is a multiple
// of 8 channels, so a vector never straddles rows.
__global__ void __launch_bounds__(256) k_ring_rows(RingArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const RingJob jb = a.job[blockIdx.y];
  const int lo = max(a.t0, a.t0 + a.n - jb.R);
  const int keep = a.t0 + a.n - lo;
  const int vpr = jb.w >> 3;
  const long long total = static_cast<long long>(a.B) * keep * vpr;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(v % vpr);
    const long long rb = v / vpr;
    const int u = lo + static_cast<int>(rb % keep);
    const int b = static_cast<int>(rb / keep);
    const uint4 x = ldg_nc(static_cast<const __nv_bfloat16*>(jb.src) +
                           (static_cast<size_t>(b) * a.n + (u - a.t0)) * jb.w + c * 8);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(jb.dst) +
                              (static_cast<size_t>(b) * jb.R + u % jb.R) * jb.w + c * 8) = x;
  }
}

}  // namespace

cudaError_t launch_ring_rows(const RingArgs& a, cudaStream_t s, int* launches) {
  if (a.n_jobs == 0 || a.n == 0 || a.B == 0) return cudaSuccess;
  long long most = 0;
  for (int j = 0; j < a.n_jobs; ++j) {
    const int keep = a.t0 + a.n - max(a.t0, a.t0 + a.n - a.job[j].R);
    most = max(most, static_cast<long long>(a.B) * keep * (a.job[j].w >> 3));
  }
  long long bx = (most + 255) / 256;
  if (bx > 1184) bx = 1184;       // 148 SMs x 8 blocks; the loop covers the rest
  const cudaError_t e = launch_k(k_ring_rows, dim3(static_cast<unsigned>(bx), a.n_jobs), dim3(256), 0, s, a);
  ++*launches;
  return e;
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s, int* launches) {
  const int TPE = a.d / 8;
  if (a.overlap && a.m == 4 && a.t0 == 0 && a.i_begin == 0 && a.out_N == a.N && a.ring.R == 0) {
    // whole-sequence CSA call: the staged kernel (64 KB of rows per CTA)
    const int EPC = 256 / TPE;
    const long long blocks = static_cast<long long>(a.B) * ((a.N + EPC - 1) / EPC);
    if (blocks == 0) return cudaSuccess;
    const size_t smem = 4 * static_cast<size_t>(EPC) * a.m * a.d * 2 + 8 * sizeof(float) + 16;
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(k_compress_staged, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_k(k_compress_staged, dim3(static_cast<unsigned>(blocks)), dim3(EPC * TPE), smem, s,
                                   a, EPC);
    ++*launches;
    return e;
  }
  const int Rmax = a.overlap ? 2 * a.m : a.m;
  int RS = Rmax / 8;
  if (RS < 1) RS = 1;
  if (RS > 8) RS = 8;
  while (RS * TPE > 256 && RS > 1) --RS;
  int EPC = 256 / (RS * TPE);
  if (EPC < 1) EPC = 1;
  const int threads = EPC * RS * TPE;
  const long long total = static_cast<long long>(a.B) * a.N;
  if (total == 0) return cudaSuccess;
  const long long blocks = (total + EPC - 1) / EPC;
  size_t smem = (RS > 1 ? static_cast<size_t>(EPC) * RS * TPE * 24 * sizeof(float) : 0) +
                (threads / 32 + 1) * sizeof(float);
  auto kern = a.overlap ? k_compress<2> : k_compress<4>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch_k(kern, dim3(static_cast<unsigned>(blocks)), dim3(threads), smem, s, a, RS, EPC);
  ++*launches;
  return e;
}

}  // namespace csa
