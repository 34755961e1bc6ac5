// gemm.cu -- bf16 GEMM on tcgen05 for the projections around attention.
//
// "Parallel multi-head attention", sections 2.1-2.3 and 3.1: the query, key and value
// projections are ColumnParallelLinear layers and the output projection a
// RowParallelLinear; on one GPU the full weights are local and each is an nn.Linear
// product y = x W^T with W [out][in].  Its forward and both gradients are one GEMM shape,
//     C[M][N] (+)= sum_k A[m][k] B[n][k]          (fp32 accumulation, bf16 C)
// with each operand stored either K-major (k contiguous: x, W in the forward, dy in the
// input gradient) or MN-major (m or n contiguous: W in the input gradient, dy and x in
// the weight gradient); tcgen05 reads both forms from shared memory, so no operand is
// ever transposed in memory.
//
// Design (persistent, one CTA per SM, 192 threads):
//   warp 0      TMA producer: 128 x 64 A and 256 x 64 B tiles through a 4-stage ring
//               (128-byte swizzle; an MN-major operand arrives as 64 x 64 boxes)
//   warp 1      MMA issuer (one thread, M = 128, N = 256, K = 16 per instruction) and
//               TMEM owner: two 256-column fp32 accumulators, so that one tile's
//               epilogue overlaps the next tile's products
//   warps 2..5  epilogue: TMEM -> registers -> bf16 (+ the old C when accumulating)
//               -> global, one output row per thread
// Tiles are visited in bands of 16 tile rows (all 16 row blocks of one column block,
// then the next column block), so the CTAs running at the same time share their A rows
// and B columns through L2.  Edges: TMA fills out-of-range rows and k with zeros, and
// the epilogue stores only rows < M and 8-column groups < N (N is a multiple of 8).
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace sp {
namespace {

constexpr int kBM = 128;          // tile rows (TMEM lanes)
constexpr int kBN = 256;          // tile columns (accumulator columns)
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kBandRows = 16;     // tile rows per band of the visiting order
constexpr uint32_t kABytes = kBM * kBK * 2;    // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;    // 32 KB
constexpr uint32_t kBoxBytes = 64 * 64 * 2;    // one MN-major box: 64 k rows x 64 elements

struct GemmSmem {
  alignas(1024) uint8_t a[kStages][kABytes];
  alignas(1024) uint8_t b[kStages][kBBytes];
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct GemmParams {
  CUtensorMap ta, tb;
  __nv_bfloat16* c;
  int64_t ldc;
  int M, N, K;
  int tiles_m, tiles_n;
  int accumulate;         // 1: C += A B^T (C read back), 0: C = A B^T
  uint32_t* status;
};

// Tile t of the visiting order -> (tile row, tile column).
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int* tm, int* tn) {
  const int per_band = kBandRows * tiles_n;
  const int band = t / per_band;
  const int first = band * kBandRows;
  const int rows = min(kBandRows, tiles_m - first);
  const int r = t - band * per_band;
  *tm = first + r % rows;
  *tn = r / rows;
}

// 2-D tiled load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// kAmn / kBmn: A / B stored MN-major ([K][M] / [K][N], m / n contiguous) instead of
// K-major ([M][K] / [N][K]).
template <bool kAmn, bool kBmn>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tiles = p.tiles_m * p.tiles_n;
  const int kblocks = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    if ((smem_u32(smem_raw) & 1023u) != 0) raise_status(p.status, kStatusBadSmem);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 128);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  int issued = 0;   // producer: k-blocks whose loads were issued, over all of its tiles

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&p.ta);
    tma_prefetch_desc(&p.tb);
    bool ok = true;
    int n = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, &tm, &tn);
      const int m0 = tm * kBM, n0 = tn * kBN;
      for (int kb = 0; kb < kblocks; ++kb, ++n) {
        const int s = n % kStages;
        if (n >= kStages &&
            !(ok = mbar_wait(&sm.empty[s], ((n / kStages) - 1) & 1, p.status, abort_flag)))
          break;
        const int k0 = kb * kBK;
        mbar_expect_tx(&sm.full[s], kABytes + kBBytes);
        if constexpr (kAmn) {
#pragma unroll
          for (int c = 0; c < kBM / 64; ++c)
            tma_load_2d(sm.a[s] + c * kBoxBytes, &p.ta, &sm.full[s], m0 + 64 * c, k0);
        } else {
          tma_load_2d(sm.a[s], &p.ta, &sm.full[s], k0, m0);
        }
        if constexpr (kBmn) {
#pragma unroll
          for (int c = 0; c < kBN / 64; ++c)
            tma_load_2d(sm.b[s] + c * kBoxBytes, &p.tb, &sm.full[s], n0 + 64 * c, k0);
        } else {
          tma_load_2d(sm.b[s], &p.tb, &sm.full[s], k0, n0);
        }
        issued = n + 1;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kId = idesc_bf16(kBM, kBN, kAmn, kBmn);
    bool ok = true;
    int n = 0, local = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t acc = tmem + buf * kBN;
      // the epilogue has read this accumulator's previous tile out of TMEM
      if (local >= 2 &&
          !(ok = mbar_wait(&sm.acc_empty[buf], ((local >> 1) - 1) & 1, p.status, abort_flag)))
        break;
      tc_fence_after();
      for (int kb = 0; kb < kblocks; ++kb, ++n) {
        const int s = n % kStages;
        if (!(ok = mbar_wait(&sm.full[s], (n / kStages) & 1, p.status, abort_flag))) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sm.a[s]), b_addr = smem_u32(sm.b[s]);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // K-major: k advances 32 bytes inside the swizzled 128-byte rows; MN-major: k
          // advances 16 rows of 128 bytes, the 64-element boxes lie 8 KB apart
          const uint64_t ad = kAmn ? sdesc_sw128(a_addr + kk * 2048, kBoxBytes, 1024)
                                   : sdesc_sw128(a_addr + kk * 32, 16, 1024);
          const uint64_t bd = kBmn ? sdesc_sw128(b_addr + kk * 2048, kBoxBytes, 1024)
                                   : sdesc_sw128(b_addr + kk * 32, 16, 1024);
          mma_ss(acc, ad, bd, kId, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&sm.empty[s]);   // the stage is free once these products have read it
      }
      if (!ok) break;
      mma_commit(&sm.acc_full[buf]);
    }
    if (!ok) {
      // unwinding: let every issued MMA finish before TMEM is released
      mma_commit(&sm.drain);
      mbar_wait_settle(&sm.drain, 0, p.status);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp % 4;                 // TMEM lanes 32 * quad .. + 31
    const int row = quad * 32 + lane;          // tile row == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    int local = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local) {
      const int buf = local & 1;
      bool ok = mbar_wait(&sm.acc_full[buf], (local >> 1) & 1, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, &tm, &tn);
      const int m = tm * kBM + row;
      const int n0 = tn * kBN;
      __nv_bfloat16* crow = p.c + static_cast<int64_t>(m) * p.ldc;
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(lane_base + buf * kBN + ch * 32, r);
        tmem_ld_wait();
        if (ch == kBN / 32 - 1) {
          // the whole accumulator is in registers: the MMA thread may reuse it
          tc_fence_before();
          mbar_arrive(&sm.acc_empty[buf]);
        }
        const int col = n0 + ch * 32;
        if (m >= p.M || col >= p.N) continue;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (col + 8 * u >= p.N) break;
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * u + e]);
          uint4* dst = reinterpret_cast<uint4*>(crow + col + 8 * u);
          if (p.accumulate) {
            const uint4 old = *dst;
            const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
              v[2 * e] += f.x;
              v[2 * e + 1] += f.y;
            }
          }
          *dst = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    // unwinding: shared memory stays with this CTA until the loads already issued into
    // it have landed (every armed phase had all of its loads issued)
    for (int s = 0; s < kStages; ++s) {
      const int armed = ring_phases(issued, s, kStages);
      if (armed > 0) mbar_wait_settle(&sm.full[s], (armed - 1) & 1, p.status);
    }
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  return n;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  GemmParams p;
  // A: K-major [M][K] -> box {64 k, 128 rows}; MN-major [K][M] -> box {64 m, 64 k}
  const bool ok_a = a.a_mn ? encode_2d_bf16_map(&p.ta, a.a, a.M, a.K, a.lda, 64, 64)
                           : encode_2d_bf16_map(&p.ta, a.a, a.K, a.M, a.lda, 64, kBM);
  const bool ok_b = a.b_mn ? encode_2d_bf16_map(&p.tb, a.b, a.N, a.K, a.ldb, 64, 64)
                           : encode_2d_bf16_map(&p.tb, a.b, a.K, a.N, a.ldb, 64, kBN);
  if (!ok_a || !ok_b) return cudaErrorInvalidValue;
  p.c = static_cast<__nv_bfloat16*>(a.c);
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.tiles_m = (a.M + kBM - 1) / kBM;
  p.tiles_n = (a.N + kBN - 1) / kBN;
  p.accumulate = a.accumulate ? 1 : 0;
  p.status = a.status;
  const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  if (sms == 0) return cudaErrorNoDevice;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, sms));
  const size_t smem = sizeof(GemmSmem);
  auto launch = [&](auto kernel) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  };
  if (!a.a_mn && !a.b_mn) return launch(gemm_kernel<false, false>);
  if (!a.a_mn && a.b_mn) return launch(gemm_kernel<false, true>);
  if (a.a_mn && a.b_mn) return launch(gemm_kernel<true, true>);
  return launch(gemm_kernel<true, false>);
}

}  // namespace sp
