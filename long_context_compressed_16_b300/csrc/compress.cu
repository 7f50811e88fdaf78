// Token-level compressor: softmax-gated weighted sum over m (HCA) or 2m overlapped (CSA) rows,
// fused with RMSNorm and partial RoPE.  ("DeepSeek V4 模型技术大全", CSA path, Softmax_row and
// C^Comp equations; HCA path, S and C^Comp equations.)
//
// Pure HBM stream: every input row is read exactly once (entry i owns a-block i and b-block i-1),
// in 16-byte vectors of 8 channels; a thread owns 8 channels of one entry.
//   - CSA with m = 4 (the method's ratio): a one-pass softmax per channel over the entry's 8 rows
//     (4 for entry 0) in two chunks of 4, one hardware exp2 per logit (csa4_entry).  Whole
//     sequences run in k_compress_stream, a persistent kernel that bulk-copies stages of entries'
//     rows into double-buffered shared memory; cache appends run the same routine in k_compress,
//     so both agree bit for bit.
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

// Pairs of fp32 lanes (channels 2p, 2p+1), each lane rounded to nearest by its own scalar
// instruction.  (The packed f32x2 forms of these were tried: the same source then gave results
// that differed in the last bit between the two kernels that inline the entry routine, so the
// whole-sequence and cache-append paths no longer agreed bit for bit.)
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
}
// a * b + c, one rounding per lane
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  return make_float2(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y));
}
// maximum of three (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }
// (lo + bx, hi + by) for the two bf16 halves of w, each one mixed-precision add (bf16 + fp32,
// rounded to nearest): the same bits as widening first and adding in fp32, without the widening
__device__ __forceinline__ float2 bf16x2_add(uint32_t w, float bx, float by) {
  float2 r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %4;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "r"(w), "f"(bx), "f"(by));
  return r;
}

// CSA entry with m = 4: softmax over the entry's R rows per channel (R = 4 for entry 0: the a-block
// only; 8 otherwise: the a-block, then the b-block of the previous block of m tokens), in two
// chunks of 4 rows.  Each chunk takes its maximum, rescales what the chunk before it summed by
// 2^(nmx_new - nmx_old), where nmx = -max log2 e, and adds one exp2 per logit:
// every row is read once.  The maximum starts at -FLT_MAX / 2 rather than -inf, so a chunk whose
// logits are all -inf contributes zero weights instead of NaN.  The weighted sum is scaled by the
// correctly rounded reciprocal of the sum.  Every floating-point step here and in the epilogue is
// an explicit instruction or an intrinsic with a fixed rounding, never a contraction left to the
// compiler, so each kernel that inlines it computes the same bits.  fetch_z(r) and
// fetch_c(r) return the logits and the values of row r (a-rows 0..3, then b-rows 4..7) for this
// thread's 8 channels, fetch_bias(r, lo, hi) the row's 8 position biases (read only when kBias);
// the values are fetched only when the weights are known.  Both kernels that
// compress m = 4 CSA entries (the streamed whole-sequence kernel and the cache-append path of
// k_compress) run exactly this code, so their results agree bit for bit.
template <int R, bool kBias, class FetchZ, class FetchC, class FetchB>
__device__ __forceinline__ void csa4_entry(FetchZ fetch_z, FetchC fetch_c, FetchB fetch_bias, float* outv) {
  const float2 kL = make_float2(kLog2e, kLog2e);
  const float2 kNegL = make_float2(-kLog2e, -kLog2e);
  float2 mx[4], nm[4], sm[4], ac[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    mx[p] = make_float2(-1.7014117e38f, -1.7014117e38f);
    sm[p] = make_float2(0.f, 0.f);
    ac[p] = make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int ch = 0; ch < R / 4; ++ch) {
    float2 t[4][4];       // [row][pair]: logit + bias
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 zv = fetch_z(ch * 4 + u);
      if (kBias) {
        float4 b0, b1;
        fetch_bias(ch * 4 + u, b0, b1);
        t[u][0] = bf16x2_add(zv.x, b0.x, b0.y);
        t[u][1] = bf16x2_add(zv.y, b0.z, b0.w);
        t[u][2] = bf16x2_add(zv.z, b1.x, b1.y);
        t[u][3] = bf16x2_add(zv.w, b1.z, b1.w);
      } else {
        t[u][0] = bf16x2_to_f2(zv.x); t[u][1] = bf16x2_to_f2(zv.y);
        t[u][2] = bf16x2_to_f2(zv.z); t[u][3] = bf16x2_to_f2(zv.w);
      }
    }
    float2 nnew[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      mx[p].x = fmax3(fmax3(mx[p].x, t[0][p].x, t[1][p].x), t[2][p].x, t[3][p].x);
      mx[p].y = fmax3(fmax3(mx[p].y, t[0][p].y, t[1][p].y), t[2][p].y, t[3][p].y);
      nnew[p] = f2_mul(mx[p], kNegL);
    }
    if (ch > 0) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 dl = f2_fma(nm[p], make_float2(-1.f, -1.f), nnew[p]);
        const float2 al = make_float2(ex2_approx(dl.x), ex2_approx(dl.y));
        sm[p] = f2_mul(sm[p], al);
        ac[p] = f2_mul(ac[p], al);
      }
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) nm[p] = nnew[p];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 cw = fetch_c(ch * 4 + u);
      const float2 cv[4] = {bf16x2_to_f2(cw.x), bf16x2_to_f2(cw.y), bf16x2_to_f2(cw.z), bf16x2_to_f2(cw.w)};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 g = f2_fma(t[u][p], kL, nm[p]);
        const float2 w = make_float2(ex2_approx(g.x), ex2_approx(g.y));
        sm[p] = f2_add(sm[p], w);
        ac[p] = f2_fma(w, cv[p], ac[p]);
      }
    }
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    outv[2 * p] = __fmul_rn(ac[p].x, __frcp_rn(sm[p].x));
    outv[2 * p + 1] = __fmul_rn(ac[p].y, __frcp_rn(sm[p].y));
  }
}

// RMSNorm over the entry's d channels (the TPE threads of one entry; every thread of the sync
// domain takes part), gamma, RoPE at position m*i + pos_shift, bf16 store.  `writer`: this thread
// holds a finished outv.  `lt`: the thread's index in the sync domain, whose barrier is sync();
// `red`: the domain's shared scratch of one float per warp (used when TPE > 32).  `gam`: this
// thread's 8 RMSNorm weights already in registers, or null to read them from a.gamma.
template <class Sync>
__device__ __forceinline__ void norm_rope_store(const CompressArgs& a, float* outv, bool writer, int b, int i,
                                                int c0, int TPE, int lt, float* red, const float* gam, Sync sync) {
  const int d = a.d;
  if (a.norm) {
    float ss = 0.f;
    if (writer) {
#pragma unroll
      for (int c = 0; c < 8; c += 2) ss = fmaf(outv[c], outv[c], fmaf(outv[c + 1], outv[c + 1], ss));
    }
    const int lanes = TPE < 32 ? TPE : 32;
    for (int o = lanes >> 1; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (TPE > 32) {
      sync();
      if ((lt & 31) == 0) red[lt >> 5] = ss;
      sync();
      const int w0 = (lt / TPE) * (TPE >> 5);
      ss = 0.f;
      for (int k = 0; k < (TPE >> 5); ++k) ss = __fadd_rn(ss, red[w0 + k]);
    }
    // d is a power of two, so 1/d is exact
    const float inv = rsqrtf(fmaf(ss, 1.0f / static_cast<float>(d), a.eps));
#pragma unroll
    for (int c = 0; c < 8; ++c) outv[c] = __fmul_rn(outv[c], inv);
  }
  if (!writer) return;
  if (gam != nullptr) {
#pragma unroll
    for (int c = 0; c < 8; ++c) outv[c] = __fmul_rn(outv[c], gam[c]);
  } else if (a.gamma != nullptr) {
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0 + 4));
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) outv[c] = __fmul_rn(outv[c], gv[c]);
  }
  if (a.rope && c0 >= d - a.rp.r) {
    const long long pos = static_cast<long long>(a.m) * i + a.pos_shift;
    const int j0 = (c0 - (d - a.rp.r)) >> 1;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float cs, sn;
      rope_cos_sin(pos, a.rp.phase[j0 + p], cs, sn);
      const float x0 = outv[2 * p], x1 = outv[2 * p + 1];
      outv[2 * p] = fmaf(x0, cs, -__fmul_rn(x1, sn));
      outv[2 * p + 1] = fmaf(x0, sn, __fmul_rn(x1, cs));
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
    // row r of this entry (a-rows 0..3, b-rows 4..7): this call's chunk, or the tail ring for a
    // token before it.  Token indices stay below 2^31 (checked by the host), so 32-bit
    // arithmetic: a 64-bit remainder is a long software sequence on the GPU.
    auto row_ptr = [&](int r, const __nv_bfloat16* X, const __nv_bfloat16* Y, const __nv_bfloat16* rX,
                       const __nv_bfloat16* rY) {
      const bool isb = r >= 4;
      const int tok = isb ? 4 * (i - 1) + (r - 4) : 4 * i + r;
      if (tok >= a.t0) return (isb ? Y : X) + (static_cast<size_t>(b) * a.T + (tok - a.t0)) * d + c0;
      const uint32_t slot = static_cast<uint32_t>(tok) % static_cast<uint32_t>(a.ring.R);
      return (isb ? rY : rX) + (static_cast<size_t>(b) * a.ring.R + slot) * d + c0;
    };
    auto fetch_z = [&](int r) { return ldg_nc(row_ptr(r, Za, Zb, rZa, rZb)); };
    auto fetch_c = [&](int r) { return ldg_nc(row_ptr(r, Ca, Cb, rCa, rCb)); };
    auto fetch_bias = [&](int r, float4& lo, float4& hi) {
      const float* bp = r < 4 ? a.bias_a : a.bias_b;
      lo = hi = make_float4(0.f, 0.f, 0.f, 0.f);
      if (bp != nullptr) {
        lo = __ldg(reinterpret_cast<const float4*>(bp + static_cast<size_t>(r & 3) * d + c0));
        hi = __ldg(reinterpret_cast<const float4*>(bp + static_cast<size_t>(r & 3) * d + c0 + 4));
      }
    };
    float o4[8];
    const bool hb = a.bias_a != nullptr || a.bias_b != nullptr;
    if (i >= 1) {
      if (hb) csa4_entry<8, true>(fetch_z, fetch_c, fetch_bias, o4);
      else csa4_entry<8, false>(fetch_z, fetch_c, fetch_bias, o4);
    } else {
      if (hb) csa4_entry<4, true>(fetch_z, fetch_c, fetch_bias, o4);
      else csa4_entry<4, false>(fetch_z, fetch_c, fetch_bias, o4);
    }
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
  norm_rope_store(a, outv, active && rg == 0, b, i, c0, TPE, tid, red, nullptr, [] { __syncthreads(); });
}

// Whole-sequence CSA compression (overlap, m = 4), streamed: one persistent CTA per SM walks a
// contiguous range of stages.  A stage is EPG consecutive entries i0 .. i1-1 of one sequence,
// whose a-rows (tokens m i0 .. m i1 - 1 of Ca, Za) and b-rows (tokens m (i0-1) .. m (i1-1) - 1 of
// Cb, Zb) are four contiguous runs: 16 KB for d <= 512.  G groups of GT = max(64, d/8) threads
// take the CTA's stages from a shared counter (the next unclaimed stage of the CTA's range), each
// group with two shared-memory buffers of its own: while the group computes one stage, the bulk
// copies of its next stage land in the other buffer.  Each thread first reads its entry's rows into registers; one thread per
// group then issues the group's next copies into the buffer just read (four per stage, on the
// buffer's mbarrier) as soon as the group's named barrier shows every thread done with it, so a
// buffer is held only while it is read, both buffers are mostly in flight, the copies are spread
// over G issuing threads and a slow group never holds up another.  The position biases are copied into shared memory
// once per CTA, the RMSNorm weights into registers once per thread (a thread keeps its 8
// channels for the whole kernel).  Every wait is bounded; a group that gives up waits (bounded)
// for its own copies in flight before the CTA exits.
// Shared layout: [bias_a | bias_b] fp32 m x d each (zeros where null), 2G stage buffers of
// [Za | Ca | Zb | Cb] regions of EPG*m rows x d bf16 (b-region slot e holds the b-block of entry
// i0 + e), one float per warp for the norm, the mbarriers, the stage counter and the stage index
// held by each buffer (-1: the range is exhausted).
struct StreamShape {
  int GT, EPG, G;
  uint32_t stage_bytes, bias_bytes;
  size_t smem;
};

inline StreamShape stream_shape(int d) {
  StreamShape h;
  const int TPE = d / 8;
  h.GT = TPE > 64 ? TPE : 64;
  h.EPG = h.GT / TPE;
  h.G = 384 / h.GT;                                                   // 12 warps
  h.stage_bytes = static_cast<uint32_t>(h.EPG) * 4 * 4 * d * 2;      // 4 arrays x m = 4 rows x d bf16
  h.bias_bytes = 2u * 4u * d * 4u;
  // biases, 2G buffers, the norm scratch (one float per warp), barriers (2G + 1), the counter and
  // the buffers' stage indices
  h.smem = h.bias_bytes + 2 * static_cast<size_t>(h.G) * h.stage_bytes + 12 * 4 + 8 * (2 * h.G + 1) + 4 * (1 + 2 * h.G);
  return h;
}

template <bool kBias>
__global__ void __launch_bounds__(384, 1) k_compress_stream(CompressArgs a, StreamShape h, int n_stages) {
  extern __shared__ __align__(128) unsigned char sraw[];
  grid_dep_wait();
  grid_dep_launch();
  const int d = a.d, m = a.m;
  const int TPE = d >> 3;
  const int tid = threadIdx.x;
  const int nblk = (a.N + h.EPG - 1) / h.EPG;                      // stages per sequence
  const int j0 = static_cast<int>(static_cast<long long>(n_stages) * blockIdx.x / gridDim.x);
  const int j1 = static_cast<int>(static_cast<long long>(n_stages) * (blockIdx.x + 1) / gridDim.x);
  float* sBa = reinterpret_cast<float*>(sraw);
  float* sBb = sBa + 4 * d;
  unsigned char* stage0 = sraw + h.bias_bytes;
  float* red = reinterpret_cast<float*>(stage0 + 2 * static_cast<size_t>(h.G) * h.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 12);           // after one float per warp (8-byte aligned)
  uint64_t* pbar = full + 2 * h.G;
  int* sctr = reinterpret_cast<int*>(pbar + 1);
  volatile int* sidx = sctr + 1;
  const size_t region = static_cast<size_t>(h.EPG) * m * d;          // elements per region
  const int g = tid / h.GT;
  const int lt = tid - g * h.GT;                                     // thread index in the group
  if (tid == 0) {
    for (int s = 0; s < 2 * h.G; ++s) tc::mbar_init(&full[s], 1);
    tc::mbar_init(pbar, 1);
    tc::fence_barrier_init();
    *sctr = 0;
  }
  // a null bias reads as zeros
  if (kBias) {
    for (int k = tid; k < 4 * d; k += blockDim.x) {
      if (a.bias_a == nullptr) sBa[k] = 0.f;
      if (a.bias_b == nullptr) sBb[k] = 0.f;
    }
  }
  __syncthreads();
  if (kBias && tid == 0) {
    const uint32_t bb = 4u * d * 4u;
    tc::mbar_arrive_expect_tx(pbar, (a.bias_a != nullptr ? bb : 0u) + (a.bias_b != nullptr ? bb : 0u));
    if (a.bias_a != nullptr) tc::bulk_load(sBa, a.bias_a, bb, pbar);
    if (a.bias_b != nullptr) tc::bulk_load(sBb, a.bias_b, bb, pbar);
  }

  // claims the CTA's next stage for buffer s and bulk-copies its rows there; when the range is
  // exhausted it records -1 and completes the buffer's phase with a plain arrival
  const int ncta = j1 - j0;
  auto issue = [&](int s) {
    const int k = atomicAdd(sctr, 1);
    if (k >= ncta) {
      sidx[s] = -1;
      tc::mbar_arrive(&full[s]);
      return;
    }
    sidx[s] = k;
    const int j = j0 + k;
    const int b = j / nblk;
    const int i0 = (j % nblk) * h.EPG;
    const int i1 = min(a.N, i0 + h.EPG);
    const int e_lo = i0 == 0 ? 1 : 0;                                // entry 0 has no b-block
    const uint32_t rowb = static_cast<uint32_t>(d) * 2;
    const uint32_t abytes = static_cast<uint32_t>(i1 - i0) * m * rowb;
    const uint32_t bbytes = static_cast<uint32_t>(i1 - i0 - e_lo) * m * rowb;
    __nv_bfloat16* sZa = reinterpret_cast<__nv_bfloat16*>(stage0 + static_cast<size_t>(s) * h.stage_bytes);
    tc::mbar_arrive_expect_tx(&full[s], 2 * abytes + 2 * bbytes);
    const size_t aoff = (static_cast<size_t>(b) * a.T + static_cast<size_t>(m) * i0) * d;
    tc::bulk_load(sZa, static_cast<const __nv_bfloat16*>(a.Za) + aoff, abytes, &full[s]);
    tc::bulk_load(sZa + region, static_cast<const __nv_bfloat16*>(a.Ca) + aoff, abytes, &full[s]);
    if (bbytes > 0) {
      const size_t boff = (static_cast<size_t>(b) * a.T + static_cast<size_t>(m) * (i0 + e_lo - 1)) * d;
      const size_t soff = static_cast<size_t>(e_lo) * m * d;
      tc::bulk_load(sZa + 2 * region + soff, static_cast<const __nv_bfloat16*>(a.Zb) + boff, bbytes, &full[s]);
      tc::bulk_load(sZa + 3 * region + soff, static_cast<const __nv_bfloat16*>(a.Cb) + boff, bbytes, &full[s]);
    }
  };
  const bool issuer = lt == 0;
  if (issuer) {
    issue(2 * g);
    issue(2 * g + 1);
  }

  const int e = lt / TPE;
  const int cg = lt % TPE;
  const int c0 = cg * 8;
  float gam[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) gam[c] = 1.f;
  if (a.gamma != nullptr) {
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0 + 4));
    gam[0] = g0.x; gam[1] = g0.y; gam[2] = g0.z; gam[3] = g0.w;
    gam[4] = g1.x; gam[5] = g1.y; gam[6] = g1.z; gam[7] = g1.w;
  }
  // the group leaves together if any of its threads' bounded waits gave up
  bool ok = !tc::named_bar_or(1 + g, h.GT, kBias && !tc::mbar_wait(pbar, 0, nullptr));
  auto gsync = [&] { tc::named_bar_sync(1 + g, h.GT); };
  // the group's n-th stage sits in buffer 2g + (n & 1), in that buffer's phase n >> 1
  int n = 0;
  for (; ok; ++n) {
    const int s = 2 * g + (n & 1);
    const bool got = tc::mbar_wait(&full[s], (n >> 1) & 1, nullptr);
    const int k = got ? sidx[s] : -1;
    const int j = j0 + k;
    const int b = k >= 0 ? j / nblk : 0;
    const int i0 = k >= 0 ? (j % nblk) * h.EPG : 0;
    const int i1 = k >= 0 ? min(a.N, i0 + h.EPG) : 0;
    const int i = i0 + e;
    const bool active = i < i1;
    // the entry's rows into registers at once
    const __nv_bfloat16* sZa =
        reinterpret_cast<const __nv_bfloat16*>(stage0 + static_cast<size_t>(s) * h.stage_bytes);
    const uint32_t base = (static_cast<uint32_t>(e) * 4) * d + c0;     // element offset of row 0
    uint4 zr[8], cr[8];
    if (active) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < 4 || i >= 1) {
          const size_t off = (r < 4 ? 0 : 2 * region) + base + static_cast<uint32_t>(r & 3) * d;
          zr[r] = *reinterpret_cast<const uint4*>(sZa + off);
          cr[r] = *reinterpret_cast<const uint4*>(sZa + region + off);
        }
      }
    }
    // every thread of the group has read the buffer (the group leaves together if a wait gave
    // up, or when the range is exhausted: every thread read the same index): refill it with the
    // next unclaimed stage while the rows are reduced from registers
    if (tc::named_bar_or(1 + g, h.GT, !got) || k < 0) break;
    if (issuer) issue(s);
    float outv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (active) {
      auto fetch_z = [&](int r) { return zr[r]; };
      auto fetch_c = [&](int r) { return cr[r]; };
      auto fetch_bias = [&](int r, float4& lo, float4& hi) {
        const float* bp = (r < 4 ? sBa : sBb) + (r & 3) * d + c0;
        lo = *reinterpret_cast<const float4*>(bp);
        hi = *reinterpret_cast<const float4*>(bp + 4);
      };
      if (i >= 1) csa4_entry<8, kBias>(fetch_z, fetch_c, fetch_bias, outv);
      else csa4_entry<4, kBias>(fetch_z, fetch_c, fetch_bias, outv);
    }
    norm_rope_store(a, outv, active, b, i, c0, TPE, lt, red + g * (h.GT / 32), gam, gsync);
  }
  // before the CTA exits, nothing this group issued is still in flight (at once, unless a wait
  // gave up): the pending phases of both its buffers have completed
  if (issuer) {
    tc::mbar_wait(&full[2 * g + (n & 1)], (n >> 1) & 1, nullptr);
    tc::mbar_wait(&full[2 * g + ((n + 1) & 1)], ((n + 1) >> 1) & 1, nullptr);
    if (kBias && g == 0) tc::mbar_wait(pbar, 0, nullptr);
  }
  __syncthreads();
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
    // whole-sequence CSA call: the streamed kernel, one CTA per SM
    const StreamShape h = stream_shape(a.d);
    const int nblk = (a.N + h.EPG - 1) / h.EPG;
    const long long n_stages = static_cast<long long>(a.B) * nblk;
    if (n_stages == 0) return cudaSuccess;
    const bool hb = a.bias_a != nullptr || a.bias_b != nullptr;
    auto kern = hb ? k_compress_stream<true> : k_compress_stream<false>;
    const cudaError_t e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(h.smem));
    if (e0 != cudaSuccess) return e0;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long grid = n_stages < sms ? n_stages : sms;
    const cudaError_t e = launch_k(kern, dim3(static_cast<unsigned>(grid)), dim3(h.G * h.GT), h.smem, s, a, h,
                                   static_cast<int>(n_stages));
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
