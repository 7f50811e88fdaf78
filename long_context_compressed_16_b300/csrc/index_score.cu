// Lightning-indexer scores I_{t,s} = sum_h w_{t,h} ReLU(q^I_{t,h} . K^I_s), s < floor((t+1)/m)
// ("DeepSeek V4 模型技术大全", CSA path, the I_{t,s} equation).
//
// One CTA scores a tile of 128 keys for a group of G queries of the same sequence.  The key tile
// is staged once in shared memory (cp.async, zero-filled past N; e4m3 keys are widened to bf16,
// which is exact) and multiplied by each query's [heads x dI] block on the tensor cores
// (keys as M, heads as N, dI as K).  The ReLU / w-weighted head sum is the MMA epilogue: the
// heads of one key live in one lane quad, so the sum is two shuffles.
#include "common.cuh"

namespace csa {

namespace {

constexpr int KT = 128;         // keys per tile
constexpr int NTHREADS = 128;   // 4 warps x 32 keys

template <int DI, bool FP8>
struct IndexSmem {
  static constexpr int KS = DI + 8;                       // padded row (bf16 elements)
  static constexpr size_t k_bytes = size_t(KT) * KS * 2;
  static constexpr size_t stage_bytes = FP8 ? size_t(KT) * DI : 0;
  __host__ __device__ static size_t q_bytes(int G, int NH) { return size_t(G) * NH * KS * 2; }
  __host__ __device__ static size_t total(int G, int NH) {
    return k_bytes + stage_bytes + q_bytes(G, NH) + size_t(G) * NH * 4 + KT * 4;
  }
};

template <int DI, bool FP8>
__global__ void __launch_bounds__(NTHREADS) k_index_score(IndexArgs a, int G, int NH, int g_begin,
                                                          int fill_invisible) {
  using S = IndexSmem<DI, FP8>;
  constexpr int KS = S::KS;
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem);
  unsigned char* stage = smem + S::k_bytes;
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem + S::k_bytes + S::stage_bytes);
  float* Ws = reinterpret_cast<float*>(smem + S::k_bytes + S::stage_bytes + S::q_bytes(G, NH));
  float* kscale = Ws + G * NH;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const int grp = g_begin + blockIdx.y;
  const int gpb = (a.Tq + G - 1) / G;
  const int b = grp / gpb;
  const int i0 = (grp % gpb) * G;
  const int nq = min(G, a.Tq - i0);
  const int key0 = tile * KT;

  int maxvis = 0;
  for (int j = 0; j < nq; ++j) {
    const int t = a.q_pos[static_cast<size_t>(b) * a.Tq + i0 + j];
    maxvis = max(maxvis, n_visible(t, a.m, a.N));
  }
  if (key0 >= maxvis) {
    if (fill_invisible) {
      for (int j = 0; j < nq; ++j) {
        const long long row = static_cast<long long>(b) * a.Tq + i0 + j - a.score_row_offset;
        float* dst = a.scores + row * a.N;
        for (int s = key0 + tid; s < min(a.N, key0 + KT); s += NTHREADS) dst[s] = -INFINITY;
      }
    }
    return;
  }

  // ---- stage the key tile
  const size_t krow0 = static_cast<size_t>(b) * a.N + key0;
  if (!FP8) {
    constexpr int CPR = DI * 2 / 16;   // 16-byte chunks per row
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.kI);
    for (int c = tid; c < KT * CPR; c += NTHREADS) {
      const int r = c / CPR, q = c % CPR;
      const bool ok = key0 + r < a.N;
      const __nv_bfloat16* g = src + (krow0 + (ok ? r : 0)) * DI + q * 8;
      cp_async16(Ks + r * KS + q * 8, g, ok);
    }
  } else {
    constexpr int CPR = DI / 16;
    const unsigned char* src = static_cast<const unsigned char*>(a.kI);
    for (int c = tid; c < KT * CPR; c += NTHREADS) {
      const int r = c / CPR, q = c % CPR;
      const bool ok = key0 + r < a.N;
      const unsigned char* g = src + (krow0 + (ok ? r : 0)) * DI + q * 16;
      cp_async16(stage + r * DI + q * 16, g, ok);
    }
    for (int r = tid; r < KT; r += NTHREADS)
      kscale[r] = (key0 + r < a.N) ? a.kI_scale[krow0 + r] : 0.f;
  }
  // ---- stage the group's queries (rows >= nI are zero) and weights
  {
    constexpr int CPR = DI * 2 / 16;
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.qI);
    for (int c = tid; c < G * NH * CPR; c += NTHREADS) {
      const int row = c / CPR, q = c % CPR;
      const int j = row / NH, h = row % NH;
      const bool ok = (j < nq) && (h < a.nI);
      const size_t qrow = (static_cast<size_t>(b) * a.Tq + i0 + (ok ? j : 0)) * a.nI + (ok ? h : 0);
      cp_async16(Qs + row * KS + q * 8, src + qrow * DI + q * 8, ok);
    }
    for (int c = tid; c < G * NH; c += NTHREADS) {
      const int j = c / NH, h = c % NH;
      Ws[c] = (j < nq && h < a.nI) ? a.w[(static_cast<size_t>(b) * a.Tq + i0 + j) * a.nI + h] : 0.f;
    }
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (FP8) {
    // widen e4m3 -> bf16 (exact: every e4m3 value is a bf16 value)
    for (int c = tid; c < KT * DI / 8; c += NTHREADS) {
      const int r = c / (DI / 8), q = c % (DI / 8);
      const uint2 v = *reinterpret_cast<const uint2*>(stage + r * DI + q * 8);
      float f[8];
      e4m3x2_to_float2(static_cast<uint16_t>(v.x & 0xFFFF), f[0], f[1]);
      e4m3x2_to_float2(static_cast<uint16_t>(v.x >> 16), f[2], f[3]);
      e4m3x2_to_float2(static_cast<uint16_t>(v.y & 0xFFFF), f[4], f[5]);
      e4m3x2_to_float2(static_cast<uint16_t>(v.y >> 16), f[6], f[7]);
      uint4 o;
      o.x = pack_bf16x2(f[0], f[1]); o.y = pack_bf16x2(f[2], f[3]);
      o.z = pack_bf16x2(f[4], f[5]); o.w = pack_bf16x2(f[6], f[7]);
      *reinterpret_cast<uint4*>(Ks + r * KS + q * 8) = o;
    }
    __syncthreads();
  }

  const int NT = NH / 8;   // n8 tiles of heads (even, <= 8)
  for (int j = 0; j < nq; ++j) {
    const int t = a.q_pos[static_cast<size_t>(b) * a.Tq + i0 + j];
    const int nvis = n_visible(t, a.m, a.N);
    const __nv_bfloat16* Qj = Qs + static_cast<size_t>(j) * NH * KS;
    float acc[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[mt][nt][c] = 0.f;

#pragma unroll
    for (int ks = 0; ks < DI / 16; ++ks) {
      uint32_t af[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int row = warp * 32 + mt * 16 + (lane & 15);
        const int col = ks * 16 + (lane >> 4) * 8;
        ldmatrix_x4(af[mt][0], af[mt][1], af[mt][2], af[mt][3], smem_u32(Ks + row * KS + col));
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        if (np * 2 < NT) {
          uint32_t b0, b1, b2, b3;
          const int h = np * 16 + (lane >> 4) * 8 + (lane & 7);
          const int col = ks * 16 + ((lane >> 3) & 1) * 8;
          ldmatrix_x4(b0, b1, b2, b3, smem_u32(Qj + h * KS + col));
          const uint32_t bb0[2] = {b0, b1};
          const uint32_t bb1[2] = {b2, b3};
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            mma_bf16_16816(acc[mt][2 * np], af[mt], bb0);
            mma_bf16_16816(acc[mt][2 * np + 1], af[mt], bb1);
          }
        }
      }
    }
    // epilogue: ReLU, head weights, sum over heads (quad), write
    const float* Wj = Ws + j * NH;
    const long long row = static_cast<long long>(b) * a.Tq + i0 + j - a.score_row_offset;
    float* dst = a.scores + row * a.N;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt < NT) {
          const int h = nt * 8 + 2 * (lane & 3);
          const float w0 = Wj[h], w1 = Wj[h + 1];
          s0 = fmaf(w0, fmaxf(acc[mt][nt][0], 0.f), s0);
          s0 = fmaf(w1, fmaxf(acc[mt][nt][1], 0.f), s0);
          s1 = fmaf(w0, fmaxf(acc[mt][nt][2], 0.f), s1);
          s1 = fmaf(w1, fmaxf(acc[mt][nt][3], 0.f), s1);
        }
      }
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      if ((lane & 3) == 0) {
        const int r0 = warp * 32 + mt * 16 + (lane >> 2);
        const int r1 = r0 + 8;
        if (FP8) { s0 *= kscale[r0]; s1 *= kscale[r1]; }
        const int k0 = key0 + r0, k1 = key0 + r1;
        if (k0 < a.N && (k0 < nvis || fill_invisible)) dst[k0] = k0 < nvis ? s0 : -INFINITY;
        if (k1 < a.N && (k1 < nvis || fill_invisible)) dst[k1] = k1 < nvis ? s1 : -INFINITY;
      }
    }
  }
}

template <int DI, bool FP8>
cudaError_t launch_t(const IndexArgs& a, int G, int fill_invisible, cudaStream_t s, int* launches) {
  // heads padded to a multiple of 16 (zero q rows, zero weights) so B fragments load in pairs
  const int NH = (a.nI + 15) / 16 * 16;
  const size_t smem = IndexSmem<DI, FP8>::total(G, NH);
  cudaError_t e = cudaFuncSetAttribute(k_index_score<DI, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.N + KT - 1) / KT, a.q_count);
  k_index_score<DI, FP8><<<grid, NTHREADS, smem, s>>>(a, G, NH, a.q_begin, fill_invisible);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace

// a.q_begin / a.q_count: range of query GROUPS (G consecutive queries of one sequence).
cudaError_t launch_index_score_groups(const IndexArgs& a, int G, int fill_invisible, cudaStream_t s,
                                      int* launches) {
  if (a.dI == 128) return a.fp8 ? launch_t<128, true>(a, G, fill_invisible, s, launches)
                                : launch_t<128, false>(a, G, fill_invisible, s, launches);
  if (a.dI == 64) return a.fp8 ? launch_t<64, true>(a, G, fill_invisible, s, launches)
                               : launch_t<64, false>(a, G, fill_invisible, s, launches);
  return cudaErrorInvalidValue;
}

}  // namespace csa
