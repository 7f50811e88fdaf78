// Grouped output projection ("DeepSeek V4 模型技术大全", the grouped output projection equations
// of the CSA path and the component-table row: O = Concat of the n_h head outputs, split into g
// groups O^[u]; z^[u] = O^[u] W_down^[u] with W_down^[u] of (n_h/g) d_h x r_o, r_o = 1024;
// y = Proj(Concat_u z^[u])).
//
// Both products are one batched "TN" GEMM on the 5th-generation tensor cores:
//   C[m][u][n] = sum_k A[m][u][k] * B[u][n][k]
// A = activations (rows m, group u, K contiguous), B = weights stored out-feature major (row n of
// group u holds column n of the group's matrix), C written in bf16 with fp32 accumulation.  The
// grouped product is A = O viewed as [T][g][(n_h/g) d_h]; Proj is the same GEMM with one group.
//
// Persistent kernel, one CTA per SM, 128 x BN output tiles (n fastest, then m, then the group, so
// CTAs working at the same time share their activation panel and their group's weights in L2):
//   warp 0      TMA producer: one 128 x 64 activation tile and one BN x 64 weight tile per stage
//               (128-byte swizzle) into a 4..8-stage ring
//   warp 1      one thread issues tcgen05.mma (M = 128, N = BN, K = 16) into one of two TMEM
//               accumulators, commits stage releases and accumulator-ready barriers
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one output row per
//               thread), bf16 pack, 16-byte stores; the accumulator is released right after, so
//               the next tile's MMAs overlap this tile's stores
// Every wait is bounded; a wait that gives up records CSA_ERR_TIMEOUT in the status word and the
// CTA drains its copies and MMAs before it exits.
#include "common.cuh"
#include "tc.cuh"

namespace csa {

namespace {

constexpr int GBM = 128;   // output rows per tile (TMEM lanes)
constexpr int GBK = 64;    // K elements per stage: one 128-byte swizzled row

// SWAP = false: the MMA's M side is 128 activation rows and its N side BN weight rows.
// SWAP = true (few rows, e.g. a decode batch): the M side is 128 weight rows and the N side BN
// activation rows (16..64), so the weights, which dominate the traffic, fill whole 128-row tiles
// and every SM streams its own slice of them.  Either way each output element is one MMA chain
// over K in the same order (no split of K), so a row's result does not depend on the variant.
#ifndef CSA_GEMM_SWAP_ATOMS
#define CSA_GEMM_SWAP_ATOMS 2
#endif

template <int BN, bool SWAP>
struct GCfg {
  // K atoms (64 elements, one 128-byte swizzled row each) per stage.  The weight-major variant
  // loads two, so each weight row is read 256 contiguous bytes at a time; the MMA chain over K
  // runs in the same order either way.
  static constexpr int ATOMS = SWAP ? CSA_GEMM_SWAP_ATOMS : 1;
  static constexpr int ATOM_A = GBM * GBK * 2;
  static constexpr int ATOM_B = BN * GBK * 2;
  static constexpr int A_BYTES = ATOMS * ATOM_A;
  static constexpr int B_BYTES = ATOMS * ATOM_B;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int MAX_STAGES = SWAP ? 12 : 8;
  static constexpr int STAGES = (200 * 1024) / STAGE_BYTES > MAX_STAGES ? MAX_STAGES : (200 * 1024) / STAGE_BYTES;
  static constexpr int ACC = 2;
  static constexpr int TMEM_COLS = ACC * BN <= 32 ? 32 : ACC * BN <= 64 ? 64 : ACC * BN <= 128 ? 128
                                 : ACC * BN <= 256 ? 256 : 512;
  static constexpr int THREADS = 192;
  static constexpr int BAR_BYTES = (2 * STAGES + 2 * ACC + 1) * 8 + 16;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(SWAP ? (BN % 16 == 0 && BN >= 16 && BN <= 64) : (BN == 64 || BN == 128 || BN == 256), "tile width");
  static_assert(STAGE_BYTES % 1024 == 0, "stage bases stay 1024-byte aligned");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct GemmArgs {
  void* C;                 // bf16 [M][G][N]
  int M, N, K, G;
  int tiles_n;             // tiles along N: N / BN (SWAP: N / 128)
  int tiles_m;             // tiles along M: ceil(M / 128) (SWAP: ceil(M / BN))
  long long tiles;         // tiles_m * G * tiles_n
  int32_t* status;
};

// Tile t -> (m tile, group, n tile).  Default order: n fastest, then m, then the group: CTAs
// working at the same time share an activation panel (its n tiles run side by side), and one
// group's weights stay in L2 while all its activation panels stream past once.  SWAP: m (the
// few activation rows) fastest.
template <bool SWAP>
__device__ __forceinline__ void tile_coords(const GemmArgs& a, long long t, int& mt, int& g, int& nt) {
  if (!SWAP) {
    nt = static_cast<int>(t % a.tiles_n);
    const long long r = t / a.tiles_n;
    mt = static_cast<int>(r % a.tiles_m);
    g = static_cast<int>(r / a.tiles_m);
  } else {
    mt = static_cast<int>(t % a.tiles_m);
    const long long r = t / a.tiles_m;
    nt = static_cast<int>(r % a.tiles_n);
    g = static_cast<int>(r / a.tiles_n);
  }
}

__device__ __forceinline__ long long issued_into(long long n, int i, int P) {
  return n > i ? (n - 1 - i) / P + 1 : 0;
}

// amap: activations [M][G][K], box {64, 1, SWAP ? BN : 128}; bmap: weights [G][N][K], box
// {64, SWAP ? 128 : BN, 1}.
template <int BN, bool SWAP>
__global__ void __launch_bounds__(GCfg<BN, SWAP>::THREADS, 1)
k_gemm_tn(const GemmArgs a, const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap) {
  using C = GCfg<BN, SWAP>;
  constexpr int S = C::STAGES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (tc::sptr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  uint64_t* full = bars;                 // [S] stage landed (TMA bytes)
  uint64_t* empty = full + S;            // [S] stage consumed (MMA commit)
  uint64_t* accfull = empty + S;         // [ACC] accumulator ready (MMA commit)
  uint64_t* accempty = accfull + C::ACC; // [ACC] accumulator read (128 epilogue threads)
  uint64_t* drain = accempty + C::ACC;   // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_wait();
  grid_dep_launch();
  {
    const uint32_t bad = (tc::sptr(smem) & 1023u) | (tc::sptr(bars) & 7u) |
                         static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&amap) & 63u) |
                         static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&bmap) & 63u);
    if (bad != 0u) {
      if (threadIdx.x == 0) report_error(a.status, CSA_ERR_DEVICE_CHECK, -1000 - static_cast<int>(bad));
      return;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < C::ACC; ++i) {
      tc::mbar_init(&accfull[i], 1);
      tc::mbar_init(&accempty[i], 128);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensormap(&amap);
    tc::prefetch_tensormap(&bmap);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int KB = a.K / (GBK * C::ATOMS);

  auto fail = [&](int where) {
    *abort_flag = 1;
    report_error(a.status, CSA_ERR_TIMEOUT, 200 + where);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long long n = 0;   // stage loads issued: load j went to stage j % S, phase j / S
      bool ok = true;
      for (long long t = blockIdx.x; ok && t < a.tiles; t += gridDim.x) {
        int mt, g, nt;
        tile_coords<SWAP>(a, t, mt, g, nt);
        for (int kb = 0; kb < KB; ++kb) {
          const int s = static_cast<int>(n % S);
          const uint32_t ph = static_cast<uint32_t>((n / S) & 1);
          if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag)) { fail(1); ok = false; break; }
          tc::mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          unsigned char* st = smem + static_cast<size_t>(s) * C::STAGE_BYTES;
#pragma unroll
          for (int at = 0; at < C::ATOMS; ++at) {
            const int kx = (kb * C::ATOMS + at) * GBK;
            unsigned char* sa = st + at * C::ATOM_A;
            unsigned char* sb = st + C::A_BYTES + at * C::ATOM_B;
            if (!SWAP) {   // MMA A side: 128 activation rows; B side: BN weight rows
              tc::tma_load_3d(sa, &amap, kx, g, mt * GBM, &full[s]);
              tc::tma_load_3d(sb, &bmap, kx, nt * BN, g, &full[s]);
            } else {       // MMA A side: 128 weight rows; B side: BN activation rows
              tc::tma_load_3d(sa, &bmap, kx, nt * GBM, g, &full[s]);
              tc::tma_load_3d(sb, &amap, kx, g, mt * BN, &full[s]);
            }
          }
          ++n;
        }
      }
      for (int s = 0; s < S; ++s) {
        const long long cnt = issued_into(n, s, S);
        if (cnt > 0 && !tc::mbar_wait(&full[s], static_cast<uint32_t>((cnt - 1) & 1), nullptr))
          report_error(a.status, CSA_ERR_TIMEOUT, 209);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::umma_idesc_bf16(GBM, BN);
      long long n = 0, nt_done = 0;
      bool ok = true, issued = false;
      for (long long t = blockIdx.x; ok && t < a.tiles; t += gridDim.x) {
        const int acc = static_cast<int>(nt_done % C::ACC);
        if (!tc::mbar_wait(&accempty[acc], static_cast<uint32_t>(((nt_done / C::ACC) & 1) ^ 1), abort_flag)) {
          fail(3);
          break;
        }
        tc::tc_fence_after();
        const uint32_t dt = tmem + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          const int s = static_cast<int>(n % S);
          const uint32_t ph = static_cast<uint32_t>((n / S) & 1);
          if (!tc::mbar_wait(&full[s], ph, abort_flag)) { fail(4); ok = false; break; }
          tc::tc_fence_after();
          const uint32_t aaddr = tc::sptr(smem + static_cast<size_t>(s) * C::STAGE_BYTES);
          const uint32_t baddr = aaddr + C::A_BYTES;
#pragma unroll
          for (int at = 0; at < C::ATOMS; ++at)
#pragma unroll
            for (int k = 0; k < GBK / 16; ++k)        // 32 bytes of K per instruction
              tc::umma_bf16(dt, tc::umma_desc_sw128(aaddr + at * C::ATOM_A + k * 32),
                            tc::umma_desc_sw128(baddr + at * C::ATOM_B + k * 32), idesc, (kb | at | k) ? 1u : 0u);
          tc::umma_commit(&empty[s]);
          issued = true;
          ++n;
        }
        if (!ok) break;
        tc::umma_commit(&accfull[acc]);
        ++nt_done;
      }
      if (issued) {
        tc::umma_commit(drain);
        if (!tc::mbar_wait(drain, 0, nullptr)) report_error(a.status, CSA_ERR_TIMEOUT, 210);
      }
      for (int s = 0; s < S; ++s) {
        const long long cnt = issued_into(n, s, S);
        if (cnt > 0 && !tc::mbar_wait(&empty[s], static_cast<uint32_t>((cnt - 1) & 1), nullptr))
          report_error(a.status, CSA_ERR_TIMEOUT, 211);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;                  // TMEM lanes [32 quarter, +32)
    __nv_bfloat16* Cg = static_cast<__nv_bfloat16*>(a.C);
    long long nt_done = 0;
    for (long long t = blockIdx.x; t < a.tiles; t += gridDim.x) {
      int mt, g, nt;
      tile_coords<SWAP>(a, t, mt, g, nt);
      const int acc = static_cast<int>(nt_done % C::ACC);
      const bool got = tc::mbar_wait(&accfull[acc], static_cast<uint32_t>((nt_done / C::ACC) & 1), abort_flag);
      if (!__all_sync(0xffffffffu, got)) { fail(6); break; }
      tc::tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (!SWAP) {
        // thread = output row m; its BN columns are contiguous in C
        const int m = mt * GBM + quarter * 32 + lane;
        __nv_bfloat16* crow = Cg + (static_cast<size_t>(m) * a.G + g) * a.N + static_cast<size_t>(nt) * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tc::tmem_ld32_wait(tbase + c, v);
          if (m < a.M) {
            uint4* dst = reinterpret_cast<uint4*>(crow + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                  pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
          }
        }
      } else {
        // thread = output column n (a weight row); its BN values belong to BN activation rows, and
        // the warp's 32 lanes write 32 consecutive columns of each row
        const int n = nt * GBM + quarter * 32 + lane;
        __nv_bfloat16* ccol = Cg + static_cast<size_t>(g) * a.N + n;
        const size_t rstride = static_cast<size_t>(a.G) * a.N;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tc::tmem_ld16_wait(tbase + c, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = mt * BN + c + j;
            if (m < a.M) ccol[static_cast<size_t>(m) * rstride] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&accempty[acc]);
      ++nt_done;
    }
  }

  // ------------------------------------------------------------ teardown
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
}

int sms_here() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

template <int BN, bool SWAP>
cudaError_t launch_bn(const void* A, const void* B, void* Cout, int M, int N, int K, int G, int32_t* status,
                      cudaStream_t s, int* launches) {
  using C = GCfg<BN, SWAP>;
  CUtensorMap amap, bmap;
  const uint64_t adims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(G), static_cast<uint64_t>(M)};
  const uint32_t abox[3] = {GBK, 1, SWAP ? static_cast<uint32_t>(BN) : GBM};
  const uint64_t bdims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(G)};
  const uint32_t bbox[3] = {GBK, SWAP ? static_cast<uint32_t>(GBM) : BN, 1};
  if (!tc::make_tensor_map(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A, 2, adims, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tensor_map(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, B, 2, bdims, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  GemmArgs ga{};
  ga.C = Cout;
  ga.M = M; ga.N = N; ga.K = K; ga.G = G;
  ga.tiles_n = N / (SWAP ? GBM : BN);
  ga.tiles_m = SWAP ? (M + BN - 1) / BN : (M + GBM - 1) / GBM;
  ga.tiles = static_cast<long long>(ga.tiles_m) * G * ga.tiles_n;
  ga.status = status;
  const long long grid = ga.tiles < sms_here() ? ga.tiles : sms_here();
  cudaError_t e = cudaFuncSetAttribute(k_gemm_tn<BN, SWAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  e = launch_k(k_gemm_tn<BN, SWAP>, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS), static_cast<size_t>(C::SMEM), s,
               ga, amap, bmap);
  ++*launches;
  return e;
}

}  // namespace

// Tile shape for an M x N x K product over G groups: a negative value -BT selects the swapped
// variant with BT activation rows per tile (M <= 64 and N a multiple of 128).
int gemm_tn_tile_n(int M, int N, int K, int G) {
  if (M <= 64 && N % GBM == 0 && K % (GBK * CSA_GEMM_SWAP_ATOMS) == 0) return -((M + 15) / 16 * 16);
  const long long mt = (M + GBM - 1) / GBM;
  const int sms = sms_here();
  if (N % 256 == 0 && mt * G * (N / 256) >= sms) return 256;
  if (N % 128 == 0 && mt * G * (N / 128) >= sms) return 128;
  return 64;
}

cudaError_t launch_gemm_tn(const void* A, const void* B, void* Cout, int M, int N, int K, int G, int32_t* status,
                           cudaStream_t s, int* launches) {
  if (M == 0 || N == 0 || G == 0) return cudaSuccess;
  switch (gemm_tn_tile_n(M, N, K, G)) {
    case 256: return launch_bn<256, false>(A, B, Cout, M, N, K, G, status, s, launches);
    case 128: return launch_bn<128, false>(A, B, Cout, M, N, K, G, status, s, launches);
    case 64: return launch_bn<64, false>(A, B, Cout, M, N, K, G, status, s, launches);
    case -16: return launch_bn<16, true>(A, B, Cout, M, N, K, G, status, s, launches);
    case -32: return launch_bn<32, true>(A, B, Cout, M, N, K, G, status, s, launches);
    case -48: return launch_bn<48, true>(A, B, Cout, M, N, K, G, status, s, launches);
    default: return launch_bn<64, true>(A, B, Cout, M, N, K, G, status, s, launches);
  }
}

}  // namespace csa
