// attn_fwd.cu -- causal / key-padded multi-head attention forward on tcgen05.
//
// What it computes ("adv07: Sequence Parallel" tutorial, section 3 Q4 and
// section 4; "Parallel multi-head attention", section 3.2):
//     out[i] = softmax(scale * q[i] K^T + mask) V,   lse[i] = log sum_j exp(scale q[i].k_j)
// over the visible keys j (j <= q_offset + i when causal, q_offset being query row
// 0's position relative to key row 0; j < key_len[b]).
//
// Design (one CTA = two 128-row query tiles of one (batch entry, head)):
//   warp 0        TMA producer: Q tiles once, then K/V blocks through a 2-stage ring
//   warp 1        MMA issuer (one thread) and TMEM owner
//   warps 4..7    softmax for query tile 0, warps 8..11 for query tile 1
//                 (thread = one query row = one TMEM lane)
// TMEM (512 columns): S0 | S1 | O0 | O1.  S_t = Q_t K_j^T lands in fp32; the
// softmax warps overwrite its first half with P_t in bf16, which feeds
// O_t += P_t V_j as the TMEM A operand.  The MMA thread interleaves the two
// tiles (PV0, next S0, PV1, next S1) so the tensor core works on one tile
// while the softmax warps of the other tile run.
// Online softmax in base 2 with fp32 running max m and sum l; O is rescaled
// in TMEM only when the max grows by more than 2^8 (the stale max keeps P <= 256,
// and O, l share it, so the final O / l is unchanged).
// KV blocks past the causal diagonal or past key_len are never loaded; only
// the blocks that straddle a boundary are masked element-wise.
#include "internal.h"
#include "ptx.cuh"

namespace sp {
namespace {

constexpr int kRows = 128;      // query rows per tile (TMEM lanes)
constexpr int kKeys = 128;      // keys per KV block
constexpr int kStages = 2;
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// With a key mask, key blocks whose keys are all masked are skipped; visibility of the
// first kVisBlocks blocks (4M keys) is kept as a bitmap, later blocks are never skipped.
constexpr int kVisWords = 1024;
constexpr int kVisBlocks = kVisWords * 32;

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = kRows * D * 2;     // D/64 chunks of [128][64] bf16
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t k[kStages][kTileBytes];
  alignas(1024) uint8_t v[kStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full, drain;
  uint32_t vis[kVisWords];      // bit j: key block j has a key the key mask lets through
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdKernelParams {
  CUtensorMap tq, tk, tv;
  __nv_bfloat16* o;
  RowAddr aq, ak, ao;     // row layouts of q, k/v and o
  float* lse;
  AttnGeom g;
  int num_pairs;      // ceil(sq / 256)
  int group_shift;       // CTAs ordered heaviest first within groups of 2^group_shift heads
  uint32_t* status;
};

struct TileInfo {
  int q0;        // first query row of the tile
  int nblocks;   // KV blocks it needs
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

__device__ __forceinline__ TileInfo tile_info(const AttnGeom& g, int kvlen, int q0) {
  TileInfo t{q0, 0};
  if (q0 >= g.sq) return t;
  int end = kvlen;
  if (g.causal) end = min(end, g.q_offset + q0 + kRows);
  t.nblocks = end > 0 ? (end + kKeys - 1) / kKeys : 0;
  return t;
}

// Heads whose CTAs are dispatched together, heaviest first across the group: the largest
// power of two up to 8 that divides `heads`, so that every group is full.  With one head at a time, a
// whole wave of CTAs streams the same K and V blocks in step; spread over eight heads it
// draws on eight, and under the causal mask the heavy tiles of eight heads start first.
// (Measured on B300: 32 heads x 4096 tokens, forward 742 -> 907 TFLOP/s; 8 heads x
// 32768 tokens, 1232 -> 1288.)
int heads_group_shift(int64_t heads) { return group_shift(heads, 8); }

// kKeyMask: the problem has a general key mask (a separate instantiation, so that the
// common case carries none of the block-skipping bookkeeping).
template <int D, bool kKeyMask>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdKernelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(smem_raw);
  constexpr int kChunks = D / 64;
  constexpr uint32_t kTileBytes = FwdSmem<D>::kTileBytes;
  constexpr uint32_t kOCol0 = 256;   // O_t at column 256 + t*D

  const AttnGeom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // query-tile pairs in order of work (the late ones see the most keys under the causal
  // mask), heaviest first across a group of heads whose K and V fit in L2
  int bh, cls;
  cta_order(blockIdx.x, p.num_pairs, p.group_shift, &bh, &cls);
  const int pair = p.num_pairs - 1 - cls;   // causal: the last query tiles carry most work
  const int b = bh / g.H, h = bh % g.H;
  const int kvlen = kv_limit(g, b, p.status);
  const TileInfo ti[2] = {tile_info(g, kvlen, pair * 2 * kRows),
                          tile_info(g, kvlen, pair * 2 * kRows + kRows)};
  const int nmax = max(ti[0].nblocks, ti[1].nblocks);

  if (threadIdx.x == 0) {
    if ((smem_u32(smem_raw) & 1023u) != 0) raise_status(p.status, kStatusBadSmem);
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], kRows);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  // key mask: which key blocks hold a visible key (all threads share the loads)
  constexpr bool use_vis = kKeyMask;
  const int nvis = min(nmax, kVisBlocks);
  if constexpr (use_vis)
    for (int w = threadIdx.x; w < (nvis + 31) / 32; w += blockDim.x) sm.vis[w] = 0u;
  __syncthreads();
  if constexpr (use_vis) {
    const uint8_t* mask_row = g.key_mask + b * g.key_mask_stride;
    for (int j = threadIdx.x; j < nvis; j += blockDim.x) {
      uint32_t visible = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 z = key_mask_zero16(mask_row, j * kKeys + 16 * u, g.sk);
        const uint32_t zw[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
        for (int w = 0; w < 4; ++w)
          visible |= ~zw[w] & key_lanes_below(j * kKeys + 16 * u + 4 * w, kvlen);
      }
      if (visible != 0u) atomicOr(&sm.vis[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
  }
  // the next key block at or after j that is not skipped (nmax when none is left)
  auto next_vis = [&](int j) -> int {
    if constexpr (!use_vis) return j;
    while (j < nmax) {
      if (j >= kVisBlocks) return j;
      const uint32_t w = sm.vis[j >> 5] >> (j & 31);
      if (w != 0u) return min(j + __ffs(static_cast<int>(w)) - 1, nmax);
      j = (j | 31) + 1;
    }
    return nmax;
  };
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  int kv_issued = 0;   // producer: key blocks whose K and V loads were issued

  if (warp == 0 && lane == 0 && nmax > 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    const int ntiles = ti[1].nblocks > 0 ? 2 : 1;
    mbar_expect_tx(&sm.q_full, kTileBytes * ntiles);
    for (int t = 0; t < ntiles; ++t)
      for (int c = 0; c < kChunks; ++c) {
        const TmaRow r = tma_row(p.aq, b, ti[t].q0, h);
        tma_load_5d(sm.q[t] + c * 16384, &p.tq, &sm.q_full, c * 64, r.head, r.row, r.batch,
                    r.shard);
      }
    // n counts the key blocks visited (stages and phases follow it)
    for (int j = next_vis(0), n = 0; j < nmax; j = next_vis(j + 1), ++n) {
      const int s = n % kStages;
      if (n >= kStages && !mbar_wait(&sm.kv_empty[s], ((n / kStages) - 1) & 1, p.status, abort_flag))
        break;
      const TmaRow r = tma_row(p.ak, b, j * kKeys, h);
      mbar_expect_tx(&sm.k_full[s], kTileBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_5d(sm.k[s] + c * 16384, &p.tk, &sm.k_full[s], c * 64, r.head, r.row, r.batch,
                    r.shard);
      mbar_expect_tx(&sm.v_full[s], kTileBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_5d(sm.v[s] + c * 16384, &p.tv, &sm.v_full[s], c * 64, r.head, r.row, r.batch,
                    r.shard);
      kv_issued = n + 1;
    }
  } else if (warp == 1 && lane == 0 && nmax > 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16(kRows, kKeys, false, false);
    constexpr uint32_t kIdO = idesc_bf16(kRows, D, false, true);
    const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
    int k_ready = -1;   // visited KV blocks whose K tile has been waited for
    bool ok = mbar_wait(&sm.q_full, 0, p.status, abort_flag);
    // n: index of a key block among the visited ones (its ring stage and phase)
    auto ensure_k = [&](int n) -> bool {
      if (k_ready >= n) return true;
      k_ready = n;
      const bool r = mbar_wait(&sm.k_full[n % kStages], (n / kStages) & 1, p.status, abort_flag);
      tc_fence_after();
      return r;
    };
    auto issue_s = [&](int t, int n) {
      const uint32_t k_addr = smem_u32(sm.k[n % kStages]);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
        mma_ss(tmem + t * kKeys, sdesc_sw128(q_addr[t] + off, 16, 1024),
               sdesc_sw128(k_addr + off, 16, 1024), kIdS, kk > 0);
      }
      mma_commit(&sm.s_full[t]);
    };
    auto issue_pv = [&](int t, int n) {
      const uint32_t v_addr = smem_u32(sm.v[n % kStages]);
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)
        mma_ts(tmem + kOCol0 + t * D, tmem + t * kKeys + kk * 8,
               sdesc_sw128(v_addr + kk * 2048, 16384, 1024), kIdO, (n > 0 || kk > 0) ? 1u : 0u);
    };
    const int j0 = next_vis(0);
    if (ok && j0 < nmax) {
      tc_fence_after();
      ok = ensure_k(0);
      for (int t = 0; t < 2 && ok; ++t)
        if (j0 < ti[t].nblocks) issue_s(t, 0);
    }
    for (int j = j0, n = 0; j < nmax && ok; ++n) {
      const int jn = next_vis(j + 1);   // the next visited block
      const int s = n % kStages;
      if (!(ok = mbar_wait(&sm.v_full[s], (n / kStages) & 1, p.status, abort_flag))) break;
      tc_fence_after();
      // tile 0
      if (j < ti[0].nblocks) {
        if (!(ok = mbar_wait(&sm.p_full[0], n & 1, p.status, abort_flag))) break;
        tc_fence_after();
        issue_pv(0, n);
      }
      if (jn < ti[0].nblocks) {
        if (!(ok = ensure_k(n + 1))) break;
        issue_s(0, n + 1);
      }
      // tile 1
      if (j < ti[1].nblocks) {
        if (!(ok = mbar_wait(&sm.p_full[1], n & 1, p.status, abort_flag))) break;
        tc_fence_after();
        issue_pv(1, n);
      }
      mma_commit(&sm.kv_empty[s]);
      if (jn < ti[1].nblocks) {
        if (!(ok = ensure_k(n + 1))) break;
        issue_s(1, n + 1);
      }
      j = jn;
    }
    mma_commit(&sm.o_full);
    if (!ok) {
      // unwinding: let every issued MMA finish before TMEM is released
      mma_commit(&sm.drain);
      mbar_wait_settle(&sm.drain, 0, p.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = (warp - 4) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;                  // row in tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t s_col = t * kKeys;
    const uint32_t o_col = kOCol0 + t * D;
    const TileInfo tile = ti[t];
    const int qrow = tile.q0 + r;                    // local query row
    const int gq = g.q_offset + qrow;                // position relative to key row 0
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    int visited = 0;   // key blocks of this tile that were computed (skipped ones excluded)
    for (int j = next_vis(0); j < tile.nblocks; j = next_vis(j + 1), ++visited) {
      const int n = visited;
      if (!(ok = mbar_wait(&sm.s_full[t], n & 1, p.status, abort_flag))) break;
      tc_fence_after();
      // the score row in two round trips to TMEM of 64 columns each
      float sv[kKeys];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t raw[2][32];
        tmem_ld32(lane_base + s_col + h2 * 64, raw[0]);
        tmem_ld32(lane_base + s_col + h2 * 64 + 32, raw[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[h2 * 64 + c] = __uint_as_float(raw[c / 32][c % 32]);
      }
      const int key0 = j * kKeys;
      bool need_mask = (key0 + kKeys > kvlen) ||
                       (g.causal && key0 + kKeys - 1 > g.q_offset + tile.q0);
      const uint8_t* mask_row = kKeyMask ? g.key_mask + b * g.key_mask_stride : nullptr;
      if (kKeyMask && !need_mask) {
        // a block whose keys all pass the key mask needs no element-wise masking
        uint32_t any = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 z = key_mask_zero16(mask_row, key0 + 16 * u, g.sk);
          any |= z.x | z.y | z.z | z.w;
        }
        need_mask = any != 0;
      }
      if (need_mask) {
        const int lim = g.causal ? min(kvlen, gq + 1) : kvlen;   // visible keys: key < lim
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4 z = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (kKeyMask) z = key_mask_zero16(mask_row, key0 + 16 * u, g.sk);
          const uint32_t zw[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 16 * u + e;
            if (key0 + c >= lim || ((zw[e / 4] >> (8 * (e % 4))) & 1u)) sv[c] = -INFINITY;
          }
        }
      }
      // row maximum over eight independent chains (a single chain is 127 dependent steps)
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = sv[k];
#pragma unroll
      for (int c = 8; c < kKeys; ++c) mx8[c % 8] = fmaxf(mx8[c % 8], sv[c]);
#pragma unroll
      for (int k = 0; k < 4; ++k) mx8[k] = fmaxf(mx8[k], mx8[k + 4]);
      const float mx = fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3]));
      const float m_blk = mx * g.scale_log2;
      float m_use = m;
      float alpha = 1.0f;
      bool rescale = false;
      if (n == 0) {
        m_use = m_blk;
      } else if (m_blk > m + kRescaleThreshold) {
        m_use = m_blk;
        alpha = ex2(m - m_blk);
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_t += P V of block j-1 has completed (it precedes this S in issue order)
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t ov[16];
          tmem_ld16(lane_base + o_col + c * 16, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st16(lane_base + o_col + c * 16, ov);
        }
        tmem_st_wait();
      }
      l *= alpha;
      m = m_use;
      // P = exp2(S * scale * log2(e) - m), two columns per instruction; the row sum
      // goes into two independent pair accumulators.  A row that sees no key of this
      // tile so far keeps m = -inf; its P must be 0.
      const float nm = (m == -INFINITY) ? 0.0f : -m;
      const uint64_t sc2 = f2_pack(g.scale_log2, g.scale_log2);
      const uint64_t nm2 = f2_pack(nm, nm);
      uint64_t lsum[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(sv[c * 32 + 2 * i], sv[c * 32 + 2 * i + 1]), sc2, nm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          lsum[i & 1] = f2_add(lsum[i & 1], f2_pack(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(lane_base + s_col + c * 16, pk);
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(lsum[0], a0, a1);
        f2_unpack(lsum[1], b0, b1);
        l += (a0 + b0) + (a1 + b1);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[t]);
    }
    // epilogue: O / l -> bf16, lse = (m + log2 l) * ln 2
    if (qrow < g.sq) {
      __nv_bfloat16* orow = p.o + p.ao.off(b, qrow, h);
      float* lse_out = p.lse + (static_cast<int64_t>(b) * g.H + h) * g.sq + qrow;
      if (visited == 0 || !ok) {
        uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        *lse_out = -INFINITY;
      }
    }
    if (visited > 0 && ok) {
      ok = mbar_wait(&sm.o_full, 0, p.status, abort_flag);
      tc_fence_after();
      const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_base + o_col + c * 32, ov);
        tmem_ld_wait();
        if (qrow < g.sq && ok) {
          __nv_bfloat16* orow = p.o + p.ao.off(b, qrow, h);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                __uint_as_float(ov[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (qrow < g.sq && ok) {
        float* lse_out = p.lse + (static_cast<int64_t>(b) * g.H + h) * g.sq + qrow;
        *lse_out = (m + __log2f(l)) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (warp == 0 && lane == 0 && nmax > 0 && *abort_flag) {
    // unwinding: shared memory stays with this CTA until the loads already issued into
    // it have landed (every armed phase had all of its loads issued)
    mbar_wait_settle(&sm.q_full, 0, p.status);
    for (int s = 0; s < kStages; ++s) {
      const int armed = ring_phases(kv_issued, s, kStages);
      if (armed > 0) {
        mbar_wait_settle(&sm.k_full[s], (armed - 1) & 1, p.status);
        mbar_wait_settle(&sm.v_full[s], (armed - 1) & 1, p.status);
      }
    }
  }
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t stream) {
  FwdKernelParams p;
  p.tq = a.tq;
  p.tk = a.tk;
  p.tv = a.tv;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.aq = a.aq;
  p.ak = a.ak;
  p.ao = a.ao;
  p.lse = a.lse;
  p.g = a.g;
  p.num_pairs = (a.g.sq + 2 * kRows - 1) / (2 * kRows);
  p.group_shift = heads_group_shift(static_cast<int64_t>(a.g.B) * a.g.H);
  p.status = a.status;
  const int64_t nblocks = static_cast<int64_t>(p.num_pairs) * a.g.B * a.g.H;
  if (nblocks == 0) return cudaSuccess;
  if (nblocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  auto launch = [&](auto kernel, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<static_cast<unsigned>(nblocks), kThreads, smem, stream>>>(p);
    return cudaSuccess;
  };
  const bool masked = a.g.key_mask != nullptr;
  cudaError_t e;
  if (a.g.d == 128)
    e = masked ? launch(attn_fwd_kernel<128, true>, sizeof(FwdSmem<128>))
               : launch(attn_fwd_kernel<128, false>, sizeof(FwdSmem<128>));
  else
    e = masked ? launch(attn_fwd_kernel<64, true>, sizeof(FwdSmem<64>))
               : launch(attn_fwd_kernel<64, false>, sizeof(FwdSmem<64>));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sp
