// attn_bwd.cu -- backward of the attention forward, on tcgen05.
//
// The pages give no backward formulas; this is the textbook derivative of
// out_i = sum_j P_ij v_j with P_ij = exp(scale q_i.k_j - lse_i) over visible keys:
//     D_i   = sum_c dout_ic out_ic
//     dP_ij = dout_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
//     dq_i  = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dout_i
//
// Three launches:
//   1. bwd_prep: per query row D_i and -lse_i*log2(e) into the workspace (padded
//      and empty rows get -inf, D = 0 so they contribute nothing), and zero the fp32
//      dQ accumulator.  Skipped by a call that continues an accumulation over key
//      chunks: its rows, o, lse and dout are the previous call's.  Bandwidth bound.
//   2. bwd_main: one CTA per (batch entry, head, 128-key block), looping over the
//      128-row query tiles that can see it (causal: from the diagonal down).  Two
//      compute warpgroups each own 64 of a tile's query columns.  P is kept in fp32
//      registers between the P pass and the dS pass.
//        S^T = K Q_i^T, dP^T = V dO_i^T        (A, B from shared memory, K-major;
//                                               N = 128: an N = 64 product takes
//                                               as long as an N = 128 one)
//        dV += P^T dO_i                        (P^T from TMEM, dO MN-major in smem)
//        dK += dS^T Q_i                        (dS^T K-major in smem, Q MN-major)
//        dQ_i^T = K^T dS^T  (d = 128)          (K and the dS tile, both read MN-major)
//        dQ_i   = dS K      (d = 64)
//      dQ_i is read out of TMEM at once by a drain warpgroup (so the next tile's dP^T
//      can reuse the columns) and added into the fp32 workspace: for d = 128 straight
//      from registers (TMEM lanes are head-dim indices, so a warp's 32 lanes add one
//      contiguous 128-byte piece of a dQ row); for d = 64 by 16-byte vector reductions
//      into an accumulator laid out [16][rows][4] per head (TMEM lanes are queries, so
//      a warp's 32 lanes add 512 contiguous bytes).
//   3. bwd_dq_convert: dq = bf16(scale * accumulator).  Bandwidth bound.
#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace sp {
namespace {

constexpr int kRows = 128;   // query rows per tile
constexpr int kKeys = 128;   // keys per CTA
// warp 0 TMA, warp 1 MMA (warps 2, 3 idle), warps 4..11 two compute warpgroups, warps
// 12..15 the dQ drain warpgroup
constexpr int kThreads = 512;
// Registers per thread after the split (launched with 65536 / 512 = 128 each).  Each
// SM sub-partition holds one warp of every warpgroup: 72 + 152 + 152 + 136 = 512
// registers per lane slot, its whole 16384-entry file; the 56 x 128 registers the first
// warpgroup gives back are exactly the 24 x 256 + 8 x 128 the others take.
constexpr uint32_t kRegsControl = 72, kRegsCompute = 152, kRegsDrain = 136;
static_assert(kRegsControl + 2 * kRegsCompute + kRegsDrain == 4 * 128, "register split");
constexpr float kLog2e = 1.4426950408889634f;
// Sleep between pairs of 128-byte dQ reductions (d = 128), and twice that between
// 512-byte ones (d = 64): the same rate of bytes per drain warp.
constexpr unsigned kDrainPaceNs = 30;

// ---------------------------------------------------------------- 1. row statistics

template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const RowAddr ao,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ stats,
                                                       float* __restrict__ dq_acc, int B, int H,
                                                       int sq, int64_t rows) {
  // one warp per kRowsPerWarp consecutive (batch entry, head, padded row) rows: all of
  // their loads are issued before any reduction, so that a warp waits for memory once
  constexpr int kRowsPerWarp = 4;
  constexpr int kPer = D / 32;   // elements per lane
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int64_t total = static_cast<int64_t>(B) * H * rows;
  const int64_t first = wid * kRowsPerWarp;
  if (first >= total) return;
  // rows is a multiple of 128, so the kRowsPerWarp rows share one (batch entry, head)
  const int64_t bh = first / rows;
  const int64_t i0 = first % rows;
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  float x[kRowsPerWarp][kPer], y[kRowsPerWarp][kPer];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) x[r][k] = y[r][k] = 0.0f;
    const int64_t i = i0 + r;
    if (i < sq) {
      const int64_t off = ao.off(b, static_cast<int>(i), h) + lane * kPer;
      if constexpr (kPer == 4) {
        const uint2 a2 = *reinterpret_cast<const uint2*>(o + off);
        const uint2 c2 = *reinterpret_cast<const uint2*>(dout + off);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a2);
        const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c2);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float2 fa = __bfloat1622float2(pa[k]), fc = __bfloat1622float2(pc[k]);
          x[r][2 * k] = fa.x;
          x[r][2 * k + 1] = fa.y;
          y[r][2 * k] = fc.x;
          y[r][2 * k + 1] = fc.y;
        }
      } else {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + off));
        const float2 fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dout + off));
        x[r][0] = fa.x;
        x[r][1] = fa.y;
        y[r][0] = fc.x;
        y[r][1] = fc.y;
      }
    }
  }
  float* srow = stats + bh * 2 * rows;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc = fmaf(x[r][k], y[r][k], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int64_t i = i0 + r;
    if (lane == 0) {
      float nl2 = -INFINITY;   // padded or empty row: P = exp2(x - inf) = 0
      if (i < sq) {
        const float v = lse[bh * sq + i];
        if (v != -INFINITY) nl2 = -v * kLog2e;
      }
      srow[i] = nl2;
      srow[rows + i] = (i < sq) ? acc : 0.0f;
    }
  }
  if (dq_acc != nullptr) {   // null: keep the previous call's accumulator
    // the kRowsPerWarp rows are contiguous in the accumulator
    float4* z = reinterpret_cast<float4*>(dq_acc + (bh * rows + i0) * D);
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = lane; c < kRowsPerWarp * D / 4; c += 32) z[c] = zero;
  }
}

// ---------------------------------------------------------------- 3. dQ convert

template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ dq_acc,
                                                             __nv_bfloat16* __restrict__ dq,
                                                             const RowAddr aq, int B, int H, int sq,
                                                             int64_t rows, float scale) {
  // thread = 8 consecutive elements of one row
  constexpr int kVec = D / 8;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(B) * H * sq * kVec;
  if (t >= total) return;
  const int c = static_cast<int>(t % kVec);
  const int64_t row = t / kVec;   // (b, h, i) with i fastest
  const int64_t i = row % sq;
  const int64_t bh = row / sq;
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  const float4* src = reinterpret_cast<const float4*>(dq_acc + (bh * rows + i) * D + c * 8);
  const float4 x = src[0], y = src[1];
  uint4 out;
  out.x = pack_bf16x2(x.x * scale, x.y * scale);
  out.y = pack_bf16x2(x.z * scale, x.w * scale);
  out.z = pack_bf16x2(y.x * scale, y.y * scale);
  out.w = pack_bf16x2(y.z * scale, y.w * scale);
  *reinterpret_cast<uint4*>(dq + aq.off(b, static_cast<int>(i), h) + c * 8) = out;
}

// d = 64: the accumulator holds each head as [16][rows][4] (four consecutive head-dim
// entries of a row side by side).  Thread = one row: 16 loads of 16 bytes, adjacent
// threads on adjacent rows.
__global__ void __launch_bounds__(256) bwd_dq_convert_d4_kernel(const float* __restrict__ dq_acc,
                                                                __nv_bfloat16* __restrict__ dq,
                                                                const RowAddr aq, int B, int H,
                                                                int sq, int64_t rows, float scale) {
  constexpr int D = 64;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= static_cast<int64_t>(B) * H * sq) return;
  const int64_t i = t % sq;
  const int64_t bh = t / sq;
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  const float4* src = reinterpret_cast<const float4*>(dq_acc + bh * rows * D) + i;
  __nv_bfloat16* out = dq + aq.off(b, static_cast<int>(i), h);
#pragma unroll
  for (int g = 0; g < D / 8; ++g) {
    const float4 x = src[(2 * g) * rows], y = src[(2 * g + 1) * rows];
    *reinterpret_cast<uint4*>(out + g * 8) =
        make_uint4(pack_bf16x2(x.x * scale, x.y * scale), pack_bf16x2(x.z * scale, x.w * scale),
                   pack_bf16x2(y.x * scale, y.y * scale), pack_bf16x2(y.z * scale, y.w * scale));
  }
}

// ---------------------------------------------------------------- 2. main kernel

template <int D>
struct BwdSmem {
  static constexpr int kTileBytes = kRows * D * 2;
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t dout[2][kTileBytes];
  // dS as [key][query]: chunk h holds query columns [64h, 64h+64) of the tile
  alignas(1024) uint8_t ds[kKeys * kRows * 2];
  alignas(16) float stats[2][2][kRows];            // [stage][-lse*log2e | D][row]
  // q_full: Q tile + row statistics (needed first, by S^T); do_full: dO tile (dP^T, dV).
  // do_empty frees a dO stage as soon as dV has read it, q_empty a Q stage after dK: the
  // next dO load then starts half a tile earlier than the Q load of the same stage
  uint64_t kv_full, q_full[2], do_full[2], q_empty[2], do_empty[2], s_full, dp_full, p_full[2],
      pds[2],
      ds_empty, dq_full, dq_empty, dkv_full, drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdKernelParams {
  CUtensorMap tq, tk, tv, tdo;
  const float* stats;     // [B][H][2][rows]: -lse*log2(e), D
  float* dq_acc;          // [B][H] blocks of rows * D: [rows][D] (d = 128), [D/4][rows][4] (d = 64)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  RowAddr aq, ak, av;     // row layouts of q and dO (TMA), k/dk, v/dv
  AttnGeom g;
  int64_t rows;
  int num_kv_tiles;
  int group_shift;       // CTAs ordered heaviest first within groups of 2^group_shift heads
  uint32_t* status;
};

// Valid keys of batch entry b: key_len[b] clamped into [0, sk].  A length outside that
// range is also reported in the status word (once per CTA), so that the host learns of
// it from sp_get_device_status while the results stay those of the clamped length.
__device__ __forceinline__ int kv_limit(const AttnGeom& g, int b, uint32_t* status) {
  int n = g.sk;
  if (g.key_len != nullptr) {
    const int kl = __ldg(g.key_len + b);
    if ((kl < 0 || kl > g.sk) && threadIdx.x == 0) raise_status(status, kStatusBadKeyLen);
    n = min(n, max(kl, 0));
  }
  return n;
}

// Threads: warp 0 TMA, warp 1 MMA (+ TMEM), warps 4..7 and 8..11 = compute warpgroups
// WG0 / WG1, each owning 64 of the 128 query columns of every tile, warps 12..15 = the
// dQ drain (a warp reaches the TMEM lanes 32 * (warp % 4) .. + 31, so any four
// consecutive warps cover all 128).  The drain has its own warps because adding a dQ
// tile into the L2-resident accumulator takes longer than computing P and dS for it
// (the reductions run at the L2's reduction rate whatever the instruction width); with
// their own warps they overlap the next tile's P and dS instead of delaying them.
//
// TMEM columns (128 lanes = the CTA's 128 keys):
//   [0,128)   S^T (query half h in [64h, 64h+64)); each warpgroup writes its P^T (bf16)
//             over the first 32 columns of the S^T half it has read
//   [128,256) dP^T; once both halves are read, dQ^T (d = 128: lanes = head-dim
//             indices, columns = queries) or dQ (d = 64: lanes = queries, columns = d)
//   [256,256+D) dK accumulator, [256+D,256+2D) dV accumulator
// Per query tile i the MMA thread issues
//   (dQ_{i-1} read out) dP^T_i | (P^T_i half h in TMEM) dV += P^T_h dO_h, h = 0, 1 |
//   S^T_{i+1} | (dS_i in shared memory) dQ_i, dK += dS^T Q_i
// Each compute warpgroup, per tile, computes P from S^T (while dP^T runs), writes P^T and
// signals it, then computes dS from dP^T (while dV and the next S^T run); the drain
// warpgroup reads dQ_i out of TMEM (while dK runs), which frees the columns for the next
// dP^T, and adds it to the accumulator while the next tile proceeds.  The tensor core thus
// works on one product or another while the warpgroups compute, instead of waiting for
// both halves of P and dS before any dV, dK or next-tile product can start.  A dO stage is
// released as soon as dV has read it, so the dO of tile i + 2 is already loading while
// tile i's S^T, dQ and dK products run (measured on B300: a dO wait of about 300 cycles
// per tile before; 70B-shaped backward 44.5 -> 43.8 ms at a lower clock).  The next
// S^T overwrites the P^T columns only after the dV products that read them (tcgen05 MMAs
// of one thread run in issue order), and the warpgroups write the next dS only after
// the dK and dQ products of this tile have finished reading the dS tile.
//
// d = 64: the dQ product keeps queries as lanes (dQ^T would have only 64 lanes), and
// the accumulator holds each head as [16][rows][4], so that a lane's four consecutive
// head-dim entries are one 16-byte reduction and a warp's 32 rows 512 contiguous bytes.
// (Staging dQ through the freed dS tile and adding it with TMA reduce-adds instead made
// the compute warpgroups wait for the tile: padded workload's backward 0.638 ms, against
// 0.549 with these reductions.)
// kGrouped: CTAs ordered heaviest first across groups of heads (a separate instantiation:
// the mapping costs the d = 128 kernel a few spilled registers, so launches that keep one
// head at a time use the plain one).
template <int D, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdKernelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  constexpr int kChunks = D / 64;
  constexpr uint32_t kTileBytes = BwdSmem<D>::kTileBytes;
  constexpr uint32_t kColDP = 128, kColDQ = 128;
  constexpr uint32_t kColDK = 256, kColDV = 256 + D;
  constexpr int kHalf = kRows / 2;                 // query columns per warpgroup

  const AttnGeom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // key blocks in order of work (small n = most query tiles under the causal mask),
  // heaviest first across a group of heads whose Q, dO and dQ accumulator fit in L2
  int bh, n;
  if constexpr (kGrouped) {
    cta_order(blockIdx.x, p.num_kv_tiles, p.group_shift, &bh, &n);
  } else {
    bh = blockIdx.x / p.num_kv_tiles;
    n = blockIdx.x % p.num_kv_tiles;
  }
  const int b = bh / g.H, h = bh % g.H;
  const int kv0 = n * kKeys;
  const int kvlen = kv_limit(g, b, p.status);
  const int m_start = g.causal ? max(0, kv0 - g.q_offset) / kRows : 0;
  const int m_end = (g.sq + kRows - 1) / kRows;
  // key mask: does the block hold a masked key below kvlen, and a visible one at all?
  // (every thread computes the same answer from the same 128 bytes)
  bool block_masked = false, block_visible = kv0 < kvlen;
  if (g.key_mask != nullptr && kv0 < kvlen) {
    const uint8_t* mask_row = g.key_mask + b * g.key_mask_stride;
    uint32_t masked = 0, visible = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 z = key_mask_zero16(mask_row, kv0 + 16 * u, g.sk);
      const uint32_t zw[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t valid = key_lanes_below(kv0 + 16 * u + 4 * w, kvlen);
        masked |= zw[w] & valid;
        visible |= ~zw[w] & valid;
      }
    }
    block_masked = masked != 0;
    block_visible = visible != 0;
  }
  // a block with no visible key has zero dK, dV and adds nothing to dQ
  const int nq = block_visible ? max(0, m_end - m_start) : 0;

  if (threadIdx.x == 0) {
    if ((smem_u32(smem_raw) & 1023u) != 0) raise_status(p.status, kStatusBadSmem);
    mbar_init(&sm.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.do_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
      mbar_init(&sm.do_empty[s], 1);
      mbar_init(&sm.p_full[s], kKeys);
      mbar_init(&sm.pds[s], kKeys);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.ds_empty, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, kKeys);
    mbar_init(&sm.dkv_full, 1);
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
  int q_issued = 0;    // producer: query tiles whose Q and statistics loads were issued
  int do_issued = 0;   // producer: query tiles whose dO load was issued

  // Every CTA takes the same register split, whatever work it has; each warpgroup sets
  // its limit at the top of its own branch.
  if (warp < 4) {
  setmaxnreg_dec<kRegsControl>();
  if (warp == 0 && lane == 0 && nq > 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    tma_prefetch_desc(&p.tdo);
    mbar_expect_tx(&sm.kv_full, 2 * kTileBytes);
    const TmaRow rk = tma_row(p.ak, b, kv0, h);
    for (int c = 0; c < kChunks; ++c) {
      tma_load_5d(sm.k + c * 16384, &p.tk, &sm.kv_full, c * 64, rk.head, rk.row, rk.batch,
                  rk.shard);
      tma_load_5d(sm.v + c * 16384, &p.tv, &sm.kv_full, c * 64, rk.head, rk.row, rk.batch,
                  rk.shard);
    }
    const float* st_base = p.stats + static_cast<int64_t>(bh) * 2 * p.rows;
    for (int it = 0; it < nq; ++it) {
      const int s = it & 1;
      const int q0 = (m_start + it) * kRows;
      // (q and dout share their row geometry, so one set of coordinates serves both)
      const TmaRow rq = tma_row(p.aq, b, q0, h);
      // dO first: its stage is free once dV of tile it - 2 has read it, before Q's stage
      // (free after dK of that tile)
      if (it >= 2 && !mbar_wait(&sm.do_empty[s], ((it >> 1) - 1) & 1, p.status, abort_flag)) break;
      mbar_expect_tx(&sm.do_full[s], kTileBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_5d(sm.dout[s] + c * 16384, &p.tdo, &sm.do_full[s], c * 64, rq.head, rq.row,
                    rq.batch, rq.shard);
      do_issued = it + 1;
      if (it >= 2 && !mbar_wait(&sm.q_empty[s], ((it >> 1) - 1) & 1, p.status, abort_flag)) break;
      mbar_expect_tx(&sm.q_full[s], kTileBytes + 2 * kRows * 4);
      for (int c = 0; c < kChunks; ++c)
        tma_load_5d(sm.q[s] + c * 16384, &p.tq, &sm.q_full[s], c * 64, rq.head, rq.row,
                    rq.batch, rq.shard);
      bulk_load(sm.stats[s][0], st_base + q0, kRows * 4, &sm.q_full[s]);
      bulk_load(sm.stats[s][1], st_base + p.rows + q0, kRows * 4, &sm.q_full[s]);
      q_issued = it + 1;
    }
  } else if (warp == 1 && lane == 0 && nq > 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16(kKeys, kRows, false, false);   // [keys x queries]
    constexpr uint32_t kIdKV = idesc_bf16(kKeys, D, false, true);       // dK, dV: N = d
    constexpr uint32_t kIdQ = idesc_bf16(kRows, D, true, true);         // dQ: M = queries, N = d
    constexpr uint32_t kIdQT = idesc_bf16(D, kRows, true, true);        // dQ^T: M = d, N = queries
    const uint32_t k_addr = smem_u32(sm.k), v_addr = smem_u32(sm.v), ds_addr = smem_u32(sm.ds);
    // S^T = K Q^T: K [keys x d] times a tile's 128 query rows, contracting over d
    auto issue_s = [&](uint32_t q_addr) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
        mma_ss(tmem, sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(q_addr + off, 16, 1024),
               kIdS, kk > 0);
      }
    };
    bool ok = mbar_wait(&sm.kv_full, 0, p.status, abort_flag);
    ok = ok && mbar_wait(&sm.q_full[0], 0, p.status, abort_flag);
    if (ok) {
      tc_fence_after();
      issue_s(smem_u32(sm.q[0]));
      mma_commit(&sm.s_full);
    }
    for (int it = 0; it < nq && ok; ++it) {
      const int s = it & 1;
      const uint32_t q_addr = smem_u32(sm.q[s]), do_addr = smem_u32(sm.dout[s]);
      // dP^T overwrites the previous tile's dQ: wait until it has been read out of TMEM
      if (it > 0 && !(ok = mbar_wait(&sm.dq_empty, (it - 1) & 1, p.status, abort_flag))) break;
      if (!(ok = mbar_wait(&sm.do_full[s], (it >> 1) & 1, p.status, abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
        mma_ss(tmem + kColDP, sdesc_sw128(v_addr + off, 16, 1024),
               sdesc_sw128(do_addr + off, 16, 1024), kIdS, kk > 0);
      }
      mma_commit(&sm.dp_full);
      // dV += P^T dO over query half hf (K = 64 queries), as soon as that P^T is in TMEM
      for (int hf = 0; hf < 2; ++hf) {
        if (!(ok = mbar_wait(&sm.p_full[hf], it & 1, p.status, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          mma_ts(tmem + kColDV, tmem + hf * kHalf + kk * 8,
                 sdesc_sw128(do_addr + hf * 8192 + kk * 2048, 16384, 1024), kIdKV,
                 (it > 0 || hf > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      mma_commit(&sm.do_empty[s]);   // dO_i has no reader left
      // the next tile's S^T: its columns are free once the dV products above have read
      // P^T (tcgen05 MMAs of one thread run in issue order); it runs while the
      // warpgroups compute dS
      if (it + 1 < nq) {
        if (!(ok = mbar_wait(&sm.q_full[s ^ 1], ((it + 1) >> 1) & 1, p.status, abort_flag))) break;
        tc_fence_after();
        issue_s(smem_u32(sm.q[s ^ 1]));
        mma_commit(&sm.s_full);
      }
      if (!(ok = mbar_wait(&sm.pds[0], it & 1, p.status, abort_flag))) break;
      if (!(ok = mbar_wait(&sm.pds[1], it & 1, p.status, abort_flag))) break;
      tc_fence_after();
      // dK += dS^T Q over both query halves (K = 128 queries)
      auto issue_dk = [&]() {
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk)
          mma_ss(tmem + kColDK, sdesc_sw128(ds_addr + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                 sdesc_sw128(q_addr + kk * 2048, 16384, 1024), kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
      };
      // dQ, contracting over the 128 keys; K and the dS tile are both read MN-major
      if constexpr (D == 128) {
        // dQ^T = K^T dS^T: A = K^T (head-dim contiguous), B = dS^T (queries contiguous).
        // Issued before dK so that its read-out and reductions overlap the dK products.
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ss(tmem + kColDQ, sdesc_sw128(k_addr + kk * 2048, 16384, 1024),
                 sdesc_sw128(ds_addr + kk * 2048, 16384, 1024), kIdQT, kk > 0);
        mma_commit(&sm.dq_full);
        issue_dk();
      } else {
        // dQ = dS K: A = dS (queries contiguous), B = K (head-dim contiguous).  Issued
        // before dK so that its read-out and reductions overlap the dK products.
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ss(tmem + kColDQ, sdesc_sw128(ds_addr + kk * 2048, 16384, 1024),
                 sdesc_sw128(k_addr + kk * 2048, 16384, 1024), kIdQ, kk > 0);
        mma_commit(&sm.dq_full);
        issue_dk();
      }
      // the dS tile and Q_i have no reader left
      mma_commit(&sm.ds_empty);
      mma_commit(&sm.q_empty[s]);
    }
    mma_commit(&sm.dkv_full);
    if (!ok) {
      // unwinding: let every issued MMA finish before TMEM is released
      mma_commit(&sm.drain);
      mbar_wait_settle(&sm.drain, 0, p.status);
    }
  }
  } else if (warp < 12) {
    setmaxnreg_inc<kRegsCompute>();
    // ------------------------------------------------------------ P / dS, epilogue
    const int wg = (warp - 4) / 4;                   // query half owned by this warpgroup
    const int quad = warp % 4;
    const int jj = quad * 32 + lane;                 // key row in tile == TMEM lane
    const int key = kv0 + jj;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t s_col = wg * kHalf;
    const uint32_t dp_col = kColDP + wg * kHalf;
    uint8_t* ds_row = sm.ds + wg * 16384 + jj * 128; // row jj of this half's dS chunk
    const int swz = jj & 7;
    const bool key_ok = key < kvlen && (g.key_mask == nullptr ||
                                        g.key_mask[b * g.key_mask_stride + key] != 0);
    bool ok = true;
    for (int it = 0; it < nq; ++it) {
      const int s = it & 1;
      const int q0 = (m_start + it) * kRows;
      ok = mbar_wait(&sm.q_full[s], (it >> 1) & 1, p.status, abort_flag);
      ok = ok && mbar_wait(&sm.s_full, it & 1, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* nlse2 = sm.stats[s][0] + wg * kHalf;   // -lse * log2(e)
      const float* Dv = sm.stats[s][1] + wg * kHalf;
      const int qh0 = q0 + wg * kHalf;               // first query row of this half
      const bool need_mask = block_masked || (kv0 + kKeys > kvlen) ||
                             (g.causal && kv0 + kKeys - 1 > g.q_offset + qh0);
      // first query column (relative to the half) that sees this key under the causal mask
      const int first_q = g.causal ? key - g.q_offset - qh0 : -(1 << 30);
      const float4* nl4 = reinterpret_cast<const float4*>(nlse2);
      const float4* D4 = reinterpret_cast<const float4*>(Dv);
      const uint64_t scale2 = f2_pack(g.scale_log2, g.scale_log2);
      // P of this half's 64 columns, fp32 column pairs, kept for dS
      uint64_t p2[kHalf / 2];
      // one copy of each loop per masking case, chosen once per tile (need_mask is
      // uniform across the warpgroup): no branches inside, so column pairs interleave
      auto p_half = [&](auto masked) {
        constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          // 32 columns of S^T per round trip to TMEM
          uint32_t sraw[32];
          tmem_ld32(lane_base + s_col + ch * 32, sraw);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 l4 = nl4[ch * 8 + i4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int cc = i4 * 4 + h2 * 2;          // column pair within the chunk
              // x = S * scale * log2(e) - lse * log2(e), two columns per instruction
              const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sraw[cc]),
                                                 __uint_as_float(sraw[cc + 1])),
                                         scale2, h2 ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y));
              float x0, x1;
              f2_unpack(x2, x0, x1);
              float p0 = ex2(x0), p1 = ex2(x1);
              if constexpr (kMasked) {
                const int c = ch * 32 + cc;
                p0 = (key_ok && c >= first_q) ? p0 : 0.0f;
                p1 = (key_ok && c + 1 >= first_q) ? p1 : 0.0f;
              }
              p2[ch * 16 + i4 * 2 + h2] = f2_pack(p0, p1);
              pk[i4 * 2 + h2] = pack_bf16x2(p0, p1);
            }
          }
          tmem_st16(lane_base + s_col + ch * 16, pk);   // over S^T columns already read
        }
      };
      if (need_mask)
        p_half(std::true_type{});
      else
        p_half(std::false_type{});
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[wg]);
      // dS = P (dP - D) once dP^T is in TMEM and the MMAs of the previous tile have
      // finished reading the dS tile
      ok = mbar_wait(&sm.dp_full, it & 1, p.status, abort_flag);
      if (it > 0)
        ok = ok && mbar_wait(&sm.ds_empty, (it - 1) & 1, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t draw[32];
        tmem_ld32(lane_base + dp_col + ch * 32, draw);
        tmem_ld_wait();
        uint32_t dk2[16];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 d4 = D4[ch * 8 + i4];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int cc = i4 * 4 + h2 * 2;
            const uint64_t ds2 = f2_mul(
                p2[ch * 16 + i4 * 2 + h2],
                f2_sub(f2_pack(__uint_as_float(draw[cc]), __uint_as_float(draw[cc + 1])),
                       h2 ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y)));
            float d0, d1;
            f2_unpack(ds2, d0, d1);
            dk2[i4 * 2 + h2] = pack_bf16x2(d0, d1);
          }
        }
        // dS row into the swizzled [key][query] chunk of this half: 4 x 16-byte units
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4* dst = reinterpret_cast<uint4*>(ds_row + (((ch * 4 + u) ^ swz) * 16));
          *dst = make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.pds[wg]);
    }
    // epilogue: dK = scale * acc, dV = acc (zero when no query row sees this key block);
    // each warpgroup writes its half of the d columns
    const bool have = nq > 0;
    if (have && ok) {
      ok = mbar_wait(&sm.dkv_full, 0, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) tc_fence_after();
    }
    const bool store = key < g.sk;
    __nv_bfloat16* dk_row = p.dk + p.ak.off(b, key, h) + wg * (D / 2);
    __nv_bfloat16* dv_row = p.dv + p.av.off(b, key, h) + wg * (D / 2);
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = (which == 0 ? kColDK : kColDV) + wg * (D / 2);
      const float mul = which == 0 ? g.scale : 1.0f;
      __nv_bfloat16* row = which == 0 ? dk_row : dv_row;
#pragma unroll
      for (int c = 0; c < D / 2; c += 32) {
        uint32_t r[32];
        if (have && ok) {
          tmem_ld32(lane_base + col + c, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        if (store) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
          uint4* o = reinterpret_cast<uint4*>(row + c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  } else {
    setmaxnreg_inc<kRegsDrain>();
    // ------------------------------------------------------------ dQ drain
    const int quad = warp % 4;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    for (int it = 0; it < nq; ++it) {
      const int q0 = (m_start + it) * kRows;
      ok = mbar_wait(&sm.dq_full, it & 1, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if constexpr (D == 128) {
        // dQ^T: lane = head-dim index quad * 32 + lane, columns = the tile's 128 queries.
        // All of it leaves TMEM before the release (the next dP^T waits for it); then it
        // is added row by row: a warp's lanes cover 32 consecutive head-dim entries of one
        // query row, one 128-byte piece
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + kColDQ + c * 32, r[c]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        float* dst = p.dq_acc + (static_cast<int64_t>(bh) * p.rows + q0) * D + quad * 32 + lane;
        // The reductions leave two at a time with a short sleep between pairs: issued back
        // to back, 512 of them per tile fill the memory-instruction queue that the MMA
        // thread's barrier waits and the compute warps' shared-memory stores also go
        // through, and those then wait behind them.  (Measured on B300, 70B-shaped
        // backward, three runs each: 43.25-43.45 -> 41.29-41.54 ms, at a clock 130 MHz lower
        // under the power cap, i.e. 12% fewer cycles.  One pair per 20-30 ns is the setting
        // that held; 4 per 20 ns did nothing; 1 per 10 ns or 4 per 80 ns let the drain fall
        // behind the tiles; pacing all tiles but the last of a CTA, or spreading the
        // reductions over the measured tile period with clock reads, gave nothing.)
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            red_add(dst + (c * 32 + i) * D, __uint_as_float(r[c][i]));
            if ((i % 2) == 1) __nanosleep(kDrainPaceNs);
          }
      } else {
        // dQ: lane = query row q0 + quad * 32 + lane, columns = the 64 head-dim entries.
        // The accumulator holds each head as [d / 4][rows][4]: a lane's four consecutive
        // head-dim entries are 16 bytes, and the warp's 32 rows 512 contiguous bytes.
        uint32_t r[2][32];
        tmem_ld32(lane_base + kColDQ, r[0]);
        tmem_ld32(lane_base + kColDQ + 32, r[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        float* dst = p.dq_acc + static_cast<int64_t>(bh) * p.rows * D +
                     (static_cast<int64_t>(q0) + quad * 32 + lane) * 4;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            red_add_v4(dst + static_cast<int64_t>(c * 8 + j) * p.rows * 4,
                       __uint_as_float(r[c][4 * j]), __uint_as_float(r[c][4 * j + 1]),
                       __uint_as_float(r[c][4 * j + 2]), __uint_as_float(r[c][4 * j + 3]));
            __nanosleep(2 * kDrainPaceNs);
          }
      }
    }
    // the drain warps meet here before the common exit (without this reconvergence
    // point ptxas spills registers in every instantiation of the kernel)
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (warp == 0 && lane == 0 && nq > 0 && *abort_flag) {
    // unwinding: shared memory stays with this CTA until the loads already issued into
    // it have landed (every armed phase had all of its loads issued)
    mbar_wait_settle(&sm.kv_full, 0, p.status);
    for (int s = 0; s < 2; ++s) {
      const int armed_q = ring_phases(q_issued, s, 2), armed_do = ring_phases(do_issued, s, 2);
      if (armed_q > 0) mbar_wait_settle(&sm.q_full[s], (armed_q - 1) & 1, p.status);
      if (armed_do > 0) mbar_wait_settle(&sm.do_full[s], (armed_do - 1) & 1, p.status);
    }
  }
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  const AttnGeom& g = a.g;
  const int64_t rows = padded_rows(g.sq);
  const int64_t bh = static_cast<int64_t>(g.B) * g.H;
  if (bh == 0 || (g.sq == 0 && g.sk == 0)) return cudaSuccess;
  cudaError_t e;
  // 1. statistics + zero the dQ accumulator; a call that continues an accumulation
  //    over key chunks reuses both (same o, lse and dout as the previous call)
  if (!a.dq_accumulate) {
    const int64_t warps = bh * rows / 4;   // four rows per warp (rows is a multiple of 128)
    const int64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > 0) {
      if (g.d == 128)
        bwd_prep_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout),
            a.ao, a.lse, a.row_stats,
            a.dq_accumulate ? nullptr : a.dq_acc, g.B, g.H,
            g.sq, rows);
      else
        bwd_prep_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout),
            a.ao, a.lse, a.row_stats,
            a.dq_accumulate ? nullptr : a.dq_acc, g.B, g.H,
            g.sq, rows);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  // 2. main kernel
  {
    BwdKernelParams p;
    p.tq = a.tq;
    p.tk = a.tk;
    p.tv = a.tv;
    p.tdo = a.tdo;
    p.stats = a.row_stats;
    p.dq_acc = a.dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.aq = a.aq;
    p.ak = a.ak;
    p.av = a.av;
    p.g = g;
    p.rows = rows;
    p.num_kv_tiles = (g.sk + kKeys - 1) / kKeys;
    // Up to eight heads per group, as many as keep their Q, dO and fp32 dQ rows within
    // half of L2: the re-read tensors stay there, and the heavy key blocks of several
    // heads start first (measured on B300: 32 heads x 4096 tokens 0.52 -> 0.49 ms;
    // 8 heads x 32768 tokens, where a group would overflow L2, keeps one head at a time).
    {
      const int64_t per_head = std::max<int64_t>(1, rows * g.d * (2 + 2 + 4));   // 0 rows: sq = 0
      const int64_t l2 = device_l2_bytes();
      const int64_t cap = l2 > 0 ? std::min<int64_t>(8, (l2 / 2) / per_head) : 1;
      p.group_shift = group_shift(bh, cap);
    }
    p.status = a.status;
    const int64_t nblocks = bh * p.num_kv_tiles;
    if (nblocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if (nblocks > 0) {
      auto launch = [&](auto kernel, size_t smem) -> cudaError_t {
        cudaError_t err =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        kernel<<<static_cast<unsigned>(nblocks), kThreads, smem, stream>>>(p);
        return cudaGetLastError();
      };
      const bool grouped = p.group_shift > 0;
      if (g.d == 128)
        e = grouped ? launch(attn_bwd_kernel<128, true>, sizeof(BwdSmem<128>))
                    : launch(attn_bwd_kernel<128, false>, sizeof(BwdSmem<128>));
      else
        e = grouped ? launch(attn_bwd_kernel<64, true>, sizeof(BwdSmem<64>))
                    : launch(attn_bwd_kernel<64, false>, sizeof(BwdSmem<64>));
      if (e != cudaSuccess) return e;
    }
  }
  // 3. dQ convert
  {
    const int64_t threads = bh * g.sq * (g.d / 8);
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0) {
      if (g.d == 128)
        bwd_dq_convert_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), a.aq, g.B, g.H, g.sq, rows, g.scale);
      else
        bwd_dq_convert_d4_kernel<<<static_cast<unsigned>((bh * g.sq + 255) / 256), 256, 0,
                                   stream>>>(
            a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), a.aq, g.B, g.H, g.sq, rows, g.scale);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace sp

