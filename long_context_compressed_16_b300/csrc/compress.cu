// Token-level compressor: softmax-gated weighted sum over m (HCA) or 2m overlapped (CSA) rows,
// fused with RMSNorm and partial RoPE.  ("DeepSeek V4 模型技术大全", CSA path, Softmax_row and
// C^Comp equations; HCA path, S and C^Comp equations.)
//
// Pure HBM stream: every input row is read exactly once (entry i owns a-block i and b-block i-1),
// with 16-byte vector loads of 8 channels.  A thread owns 8 channels of one entry and a
// contiguous run of that entry's rows; the per-channel softmax runs online over chunks of 4 rows
// (one exp per logit plus one rescale per chunk).  Long blocks (HCA, m' = 128) are split over
// several row groups whose partial (max, sum, acc) are merged in shared memory in fixed order,
// so results are deterministic.
#include "common.cuh"

namespace csa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

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

  if (active) {
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
    for (int r0 = r_lo; r0 < r_hi; r0 += 4) {
      const int nr = min(4, r_hi - r0);
      uint4 zv[4], cv[4];
      const float* bptr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        bptr[u] = nullptr;
        if (u < nr) {
          const int r = r0 + u;
          const bool isb = r >= a.m;
          const int j = isb ? r - a.m : r;
          const long long tok = isb ? static_cast<long long>(a.m) * (i - 1) + j
                                    : static_cast<long long>(a.m) * i + j;
          if (tok >= a.t0) {              // a row of this call's chunk
            const size_t off = (static_cast<size_t>(b) * a.T + (tok - a.t0)) * d + c0;
            zv[u] = ldg_nc((isb ? Zb : Za) + off);
            cv[u] = ldg_nc((isb ? Cb : Ca) + off);
          } else {                        // an earlier token: the tail ring, slot tok mod R
            const size_t off = (static_cast<size_t>(b) * a.ring.R + tok % a.ring.R) * d + c0;
            zv[u] = ldg_nc((isb ? rZb : rZa) + off);
            cv[u] = ldg_nc((isb ? rCb : rCa) + off);
          }
          const float* bp = isb ? a.bias_b : a.bias_a;
          if (bp != nullptr) bptr[u] = bp + static_cast<size_t>(j) * d + c0;
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float z[4], cvals[4];
        float cm = mx[c];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (u < nr) {
            const uint32_t zw = (&zv[u].x)[c >> 1];
            const uint32_t cw = (&cv[u].x)[c >> 1];
            const float zb = (c & 1) ? bf16hi(zw) : bf16lo(zw);
            cvals[u] = (c & 1) ? bf16hi(cw) : bf16lo(cw);
            z[u] = (zb + (bptr[u] ? __ldg(bptr[u] + c) : 0.f)) * kLog2e;
            cm = fmaxf(cm, z[u]);
          }
        }
        const float alpha = (mx[c] == -INFINITY) ? 0.f : exp2f(mx[c] - cm);
        float s = sm[c] * alpha, ac = acc[c] * alpha;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (u < nr) {
            const float p = exp2f(z[u] - cm);
            s += p;
            ac = fmaf(p, cvals[u], ac);
          }
        }
        mx[c] = cm; sm[c] = s; acc[c] = ac;
      }
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

  // RMSNorm over the entry's d channels (threads (e, rg = 0, cg = 0..TPE-1)); all threads take part
  if (a.norm) {
    float ss = 0.f;
    if (active && rg == 0) {
#pragma unroll
      for (int c = 0; c < 8; ++c) ss = fmaf(outv[c], outv[c], ss);
    }
    const int lanes = TPE < 32 ? TPE : 32;
    for (int o = lanes >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (TPE > 32) {
      float* red = smem + (RS > 1 ? static_cast<size_t>(EPC) * RS * TPE * 24 : 0);
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
  if (!active || rg != 0) return;
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
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_compress, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch_k(k_compress, dim3(static_cast<unsigned>(blocks)), dim3(threads), smem, s, a, RS, EPC);
  ++*launches;
  return e;
}

}  // namespace csa
