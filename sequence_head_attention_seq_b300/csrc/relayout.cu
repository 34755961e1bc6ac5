// relayout.cu -- the Ulysses all-to-all of one GPU: sequence shards <-> head groups.
//
// Pages: long-context-attention issue "关于数据分割和合并" (the all-to-all acts
// like a transpose so that each rank holds the full sequence for a subset of
// heads, and a second one brings the heads back); transformers PR 31525
// "Support deepspeed sequence parallel" (shard r = rows [r*s/N, (r+1)*s/N));
// "Parallel multi-head attention" section 2.2 (contiguous head blocks).
//
//   shard buffer  [N][b][s/N][h][d]      (shard r, batch bb, local row u, head, c)
//   group buffer  [N][b][s][h/N][d]      (group g, batch bb, row t, local head j, c)
//   with t = r*(s/N) + u and head = g*(h/N) + j.
//
// Both buffers consist of "runs" of R = (h/N)*d contiguous elements (one local
// head block of one sequence row), so the permutation moves whole runs.  A CTA
// owns a tile of T consecutive sequence rows of one (group, batch): in the group
// buffer the tile is one contiguous span of T*R elements, in the shard buffer it
// is T runs at a stride of h*d.  Threads walk the tile in 16-byte vectors
// (or narrower when R is not a multiple of 8 elements), with all loads of a
// batch issued before the stores.  Purely bandwidth bound: no arithmetic on data.
#include "internal.h"

namespace sp {

namespace {

// Division by a runtime-invariant divisor by multiply-high and shift (Granlund &
// Montgomery, "Division by invariant integers using multiplication", 1994):
// q = (umulhi(n, m) + n) >> s with s = ceil(log2 D), m = floor(2^32 (2^s - D) / D) + 1.
struct FastDiv {
  uint32_t d, m, s;
  __host__ FastDiv(uint32_t divisor = 1) : d(divisor) {
    s = 0;
    while ((1ull << s) < divisor) ++s;
    m = static_cast<uint32_t>(((1ull << 32) * ((1ull << s) - divisor)) / divisor + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint64_t hi = __umulhi(n, m);
    return static_cast<uint32_t>((hi + n) >> s);
  }
};

struct RelayoutArgs {
  const uint8_t* in[kMaxRelayoutTensors];
  uint8_t* out[kMaxRelayoutTensors];
  uint32_t N, b, s, sl, h, hl, d;
  uint32_t run_vecs;       // R / vector width
  uint32_t shard_row_vecs; // shard-side row pitch in vectors: h*d, or 3*h*d for packed Q/K/V
  uint64_t shard_row;      // the same pitch in elements
  uint32_t tile_rows;      // T
  uint32_t tiles_per_shard;
  FastDiv run_div;         // divide a vector index by run_vecs
};

template <typename Vec, int kUnroll>
__device__ __forceinline__ void copy_tile(const Vec* __restrict__ src_base, Vec* __restrict__ dst_base,
                                          uint32_t nvec, const RelayoutArgs& a, bool to_heads) {
  // Vector w of the tile: run = w / run_vecs, k = w % run_vecs.
  //   group side offset  : w                       (contiguous span)
  //   shard side offset  : run * (h*d/vec) + k     (runs at stride h*d)
  const uint32_t shard_stride = a.shard_row_vecs;   // shard-side row pitch
  for (uint32_t w0 = threadIdx.x; w0 < nvec; w0 += blockDim.x * kUnroll) {
    Vec v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w = w0 + u * blockDim.x;
      if (w < nvec) {
        const uint32_t run = a.run_div.div(w);
        const uint32_t k = w - run * a.run_vecs;
        const size_t shard_off = static_cast<size_t>(run) * shard_stride + k;
        v[u] = to_heads ? __ldcs(src_base + shard_off) : __ldcs(src_base + w);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w = w0 + u * blockDim.x;
      if (w < nvec) {
        const uint32_t run = a.run_div.div(w);
        const uint32_t k = w - run * a.run_vecs;
        const size_t shard_off = static_cast<size_t>(run) * shard_stride + k;
        if (to_heads)
          __stcs(dst_base + w, v[u]);
        else
          __stcs(dst_base + shard_off, v[u]);
      }
    }
  }
}

// grid.x: tiles over (group g, batch bb, shard r, tile-in-shard); grid.y: tensor index.
template <typename Vec>
__global__ void __launch_bounds__(256) relayout_kernel(RelayoutArgs a, int to_heads) {
  constexpr uint32_t kElemsPerVec = sizeof(Vec) / 2;
  uint32_t x = blockIdx.x;
  const uint32_t tile = x % a.tiles_per_shard;
  x /= a.tiles_per_shard;
  const uint32_t r = x % a.N;
  x /= a.N;
  const uint32_t bb = x % a.b;
  const uint32_t g = x / a.b;
  const uint32_t u0 = tile * a.tile_rows;
  const uint32_t rows = min(a.tile_rows, a.sl - u0);
  const uint32_t t0 = r * a.sl + u0;
  const size_t R = static_cast<size_t>(a.hl) * a.d;
  // element offsets of the tile's first run on each side
  const size_t group_off = ((static_cast<size_t>(g) * a.b + bb) * a.s + t0) * R;
  const size_t shard_off = ((static_cast<size_t>(r) * a.b + bb) * a.sl + u0) * a.shard_row + g * R;
  const uint32_t nvec = rows * a.run_vecs;
  const int t = blockIdx.y;
  if (to_heads) {
    const Vec* src = reinterpret_cast<const Vec*>(a.in[t] + shard_off * 2);
    Vec* dst = reinterpret_cast<Vec*>(a.out[t] + group_off * 2);
    copy_tile<Vec, 4>(src, dst, nvec, a, true);
  } else {
    const Vec* src = reinterpret_cast<const Vec*>(a.in[t] + group_off * 2);
    Vec* dst = reinterpret_cast<Vec*>(a.out[t] + shard_off * 2);
    copy_tile<Vec, 4>(src, dst, nvec, a, false);
  }
  (void)kElemsPerVec;
}

}  // namespace

cudaError_t launch_relayout(const void* const* in, void* const* out, int ntensors, int N, int b,
                            int s, int h, int d, bool to_heads, cudaStream_t stream,
                            int64_t shard_row) {
  RelayoutArgs a{};
  for (int t = 0; t < ntensors; ++t) {
    a.in[t] = static_cast<const uint8_t*>(in[t]);
    a.out[t] = static_cast<uint8_t*>(out[t]);
  }
  a.N = N;
  a.b = b;
  a.s = s;
  a.sl = s / N;
  a.h = h;
  a.hl = h / N;
  a.d = d;
  const uint64_t R = static_cast<uint64_t>(a.hl) * d;
  a.shard_row = shard_row > 0 ? static_cast<uint64_t>(shard_row) : static_cast<uint64_t>(h) * d;
  // widest vector that divides a run and keeps every run 16/8/4-byte aligned
  int vec_elems = (R % 8 == 0) ? 8 : (R % 4 == 0) ? 4 : (R % 2 == 0) ? 2 : 1;
  a.run_vecs = static_cast<uint32_t>(R / vec_elems);
  a.shard_row_vecs = static_cast<uint32_t>(a.shard_row / vec_elems);
  // tile of about 32 KiB per (group, batch, shard) span
  uint64_t rows = (32768 / 2 + R - 1) / R;
  if (rows < 1) rows = 1;
  if (rows > a.sl) rows = a.sl;
  a.tile_rows = static_cast<uint32_t>(rows);
  a.tiles_per_shard = (a.sl + a.tile_rows - 1) / a.tile_rows;
  a.run_div = FastDiv(a.run_vecs);
  const uint64_t nblocks = static_cast<uint64_t>(N) * b * N * a.tiles_per_shard;
  if (nblocks == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(nblocks), ntensors);
  switch (vec_elems) {
    case 8: relayout_kernel<uint4><<<grid, 256, 0, stream>>>(a, to_heads); break;
    case 4: relayout_kernel<uint2><<<grid, 256, 0, stream>>>(a, to_heads); break;
    case 2: relayout_kernel<uint32_t><<<grid, 256, 0, stream>>>(a, to_heads); break;
    default: relayout_kernel<uint16_t><<<grid, 256, 0, stream>>>(a, to_heads); break;
  }
  return cudaGetLastError();
}

}  // namespace sp
