// sp_abi.cu -- the extern "C" boundary of libsp (declared in include/sp.h).
//
// Every entry point validates its arguments on the host and returns before
// launching anything when they are wrong.  The only library-held device state
// is a 4-byte status word that kernels OR error codes into (read and cleared by
// sp_get_device_status).
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace sp {

__device__ uint32_t g_device_status;

namespace {

ContextAddressCache g_status_addr;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sp_status check_relayout(const void* const* in, void* const* out, int ntensors, int N, int b,
                         int s, int h, int d) {
  if (in == nullptr || out == nullptr) return SP_ERR_INVALID_ARG;
  if (ntensors < 1 || ntensors > SP_MAX_RELAYOUT_TENSORS) return SP_ERR_INVALID_ARG;
  if (N < 1 || b < 1 || s < 1 || h < 1 || d < 1) return SP_ERR_INVALID_ARG;
  if (s % N != 0 || h % N != 0) return SP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(b) * s * h * d > (int64_t(1) << 40)) return SP_ERR_UNSUPPORTED;
  for (int t = 0; t < ntensors; ++t) {
    if (in[t] == nullptr || out[t] == nullptr) return SP_ERR_INVALID_ARG;
    if (!aligned16(in[t]) || !aligned16(out[t])) return SP_ERR_MISALIGNED;
  }
  return SP_OK;
}

sp_status relayout(const void* const* in, void* const* out, int ntensors, int N, int b, int s,
                   int h, int d, bool to_heads, void* stream, int64_t shard_row = 0) {
  const sp_status st = check_relayout(in, out, ntensors, N, b, s, h, d);
  if (st != SP_OK) return st;
  if (launch_relayout(in, out, ntensors, N, b, s, h, d, to_heads,
                      static_cast<cudaStream_t>(stream), shard_row) != cudaSuccess)
    return SP_ERR_CUDA;
  return SP_OK;
}

// The three tensors of a packed [N][b][s/N][3][h][d] buffer: tensor t starts t*h*d
// elements into every row of 3*h*d.
void packed_parts(const void* qkv, int h, int d, const void* part[3]) {
  const size_t step = static_cast<size_t>(h) * d * 2;
  for (int t = 0; t < 3; ++t)
    part[t] = qkv == nullptr ? nullptr : static_cast<const uint8_t*>(qkv) + t * step;
}

bool strides_ok(const int64_t st[3]) {
  for (int i = 0; i < 3; ++i)
    if (st[i] < 0 || (st[i] % 8) != 0) return false;
  return true;
}

sp_status check_attn(const sp_attn_params* p, AttnGeom* g) {
  if (p == nullptr) return SP_ERR_INVALID_ARG;
  if (p->B < 0 || p->H < 0 || p->sq < 0 || p->sk < 0) return SP_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return SP_ERR_INVALID_ARG;
  if (p->dq_accumulate != 0 && p->dq_accumulate != 1) return SP_ERR_INVALID_ARG;
  if (p->q_offset < 0 || p->kv_offset < 0) return SP_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->q_offset) + p->sq > (int64_t(1) << 30) ||
      static_cast<int64_t>(p->kv_offset) + p->sk > (int64_t(1) << 30))
    return SP_ERR_UNSUPPORTED;
  // A tensor without elements may be a null pointer (PyTorch allocates none for it): q
  // when there are no query rows, k and v when there are no keys.
  const bool none = p->B == 0 || p->H == 0;
  if ((p->q == nullptr && !(none || p->sq == 0)) ||
      ((p->k == nullptr || p->v == nullptr) && !(none || p->sk == 0)))
    return SP_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v)) return SP_ERR_MISALIGNED;
  if (!strides_ok(p->q_stride) || !strides_ok(p->k_stride) || !strides_ok(p->v_stride) ||
      !strides_ok(p->o_stride))
    return SP_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(p->key_len) & 3u) != 0) return SP_ERR_MISALIGNED;
  if (p->key_mask != nullptr) {
    if (!aligned16(p->key_mask) || p->key_mask_stride % 16 != 0) return SP_ERR_MISALIGNED;
    if (p->key_mask_stride < p->sk) return SP_ERR_INVALID_ARG;
  }
  if (p->seq_shards < 0) return SP_ERR_INVALID_ARG;
  if (p->seq_shards > 1) {
    // tensors in the sequence-shard layout: B = N * b entries, the full sequence on
    // both sides, whole 128-row tiles per shard
    const int N = p->seq_shards;
    if (p->B % N != 0 || p->sq != p->sk || p->sq % N != 0) return SP_ERR_INVALID_ARG;
    if ((p->sq / N) % 128 != 0) return SP_ERR_UNSUPPORTED;
  }
  g->B = p->B;
  g->H = p->H;
  g->sq = p->sq;
  g->sk = p->sk;
  g->d = p->d;
  g->causal = p->causal;
  // the kernels mask by the query position relative to key row 0 (may be negative:
  // query rows before a key chunk's start see none of its keys)
  g->q_offset = p->q_offset - p->kv_offset;
  g->key_len = p->key_len;
  g->key_mask = p->key_mask;
  g->key_mask_stride = p->key_mask != nullptr ? p->key_mask_stride : 0;
  g->seq_shards = p->seq_shards > 1 ? p->seq_shards : 1;
  float scale = p->softmax_scale;
  if (!(scale > 0.0f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(p->d));
  g->scale = scale;
  g->scale_log2 = scale * 1.4426950408889634f;
  return SP_OK;
}

bool empty_problem(const AttnGeom& g) { return g.B == 0 || g.H == 0 || g.sq == 0; }

struct WorkspaceLayout {
  size_t dq_off, stats_off, total;
};

WorkspaceLayout workspace_layout(const AttnGeom& g) {
  const size_t bh = static_cast<size_t>(g.B) * g.H;
  const size_t rows = static_cast<size_t>(padded_rows(g.sq));
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  WorkspaceLayout w;
  w.dq_off = 0;
  w.stats_off = up(bh * rows * g.d * sizeof(float));
  w.total = w.stats_off + up(bh * 2 * rows * sizeof(float));
  return w;
}

}  // namespace

void* current_context() {
  PFN_cuCtxGetCurrent_v4000 get = ctx_get_current_fn();
  if (get == nullptr) return nullptr;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return nullptr;
  if (ctx == nullptr) {
    // nothing current yet on this thread: cudaSetDevice makes the device's primary
    // context current (and creates it if needed)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return nullptr;
  }
  return ctx;
}

// Device address of the status word in the current context (looked up once per context).
uint32_t* status_word() {
  return static_cast<uint32_t*>(g_status_addr.get([]() -> void* {
    void* p = nullptr;
    return cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess ? p : nullptr;
  }));
}

bool encode_2d_bf16_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                        int64_t pitch, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr || inner < 1 || outer < 1) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t elem[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

RowAddr plain_rows(const int64_t stride[3], int B, int S) {
  RowAddr a;
  a.group = 0;
  a.batch = stride[0];
  a.shard = 0;
  a.row = stride[1];
  a.head = stride[2];
  a.bi = B > 0 ? B : 1;
  a.sl = S > 0 ? S : 1;
  a.group_heads = 0;
  return a;
}

RowAddr shard_rows(int N, int b, int S, int H, int d) {
  const int64_t sl = S / N, heads = static_cast<int64_t>(N) * H;
  RowAddr a;
  a.head = d;
  a.row = heads * d;
  a.batch = sl * a.row;
  a.shard = b * a.batch;
  a.group = static_cast<int64_t>(H) * d;
  a.bi = b;
  a.sl = static_cast<int>(sl);
  a.group_heads = H;
  return a;
}

bool encode_rows_map(CUtensorMap* map, const void* base, int d, int heads_total, int shards,
                     const RowAddr& a) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  // strides of size-1 dimensions are never used: any legal value (a 16-byte multiple)
  const cuuint64_t legal = static_cast<cuuint64_t>(d) * 2;
  const int heads = heads_total > 0 ? heads_total : 1;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(a.sl), static_cast<cuuint64_t>(a.bi),
                        static_cast<cuuint64_t>(shards > 0 ? shards : 1)};
  cuuint64_t strides[4] = {heads > 1 ? static_cast<cuuint64_t>(a.head) * 2 : legal,
                           a.sl > 1 ? static_cast<cuuint64_t>(a.row) * 2 : legal,
                           a.bi > 1 ? static_cast<cuuint64_t>(a.batch) * 2 : legal,
                           shards > 1 ? static_cast<cuuint64_t>(a.shard) * 2 : legal};
  cuuint32_t box[5] = {64, 1, 128, 1, 1};
  cuuint32_t elem[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// Row layouts of the attention tensors: plain strided [B][S][H][d], or all eight in the
// sequence-shard layout [N][B/N][S/N][N*H][d].
struct Layouts {
  RowAddr q, k, v, o;
  int heads_total, shards;
};

Layouts layouts_of(const sp_attn_params* p, const AttnGeom& g) {
  Layouts L;
  if (g.seq_shards > 1) {
    const int N = g.seq_shards;
    L.q = L.k = L.v = L.o = shard_rows(N, g.B / N, g.sq, g.H, g.d);
    L.heads_total = N * g.H;
    L.shards = N;
  } else {
    L.q = plain_rows(p->q_stride, g.B, g.sq);
    L.k = plain_rows(p->k_stride, g.B, g.sk);
    L.v = plain_rows(p->v_stride, g.B, g.sk);
    L.o = plain_rows(p->o_stride, g.B, g.sq);
    L.heads_total = g.H;
    L.shards = 1;
  }
  return L;
}

}  // namespace sp

using namespace sp;

namespace sp {
namespace {

// The failure path of every kernel's waits, on its own: one warp waits for phase 0 of an
// mbarrier that nothing arrives on.  The bounded wait gives up after SP_WAIT_LIMIT_NS,
// records kStatusTimeout in the status word and the kernel returns normally.
__global__ void wait_timeout_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, status, reinterpret_cast<volatile int*>(&abort_flag));
}

}  // namespace
}  // namespace sp

namespace sp {

int group_shift(int64_t heads, int64_t cap) {
  int shift = 0;
  while ((int64_t(2) << shift) <= cap && heads % (int64_t(2) << shift) == 0) ++shift;
  return shift;
}

int64_t device_l2_bytes() {
  constexpr int kMaxDev = 64;
  static std::atomic<int64_t> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int64_t l2 = cache[dev].load(std::memory_order_relaxed);
  if (l2 == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0) return 0;
    l2 = v;
    cache[dev].store(l2, std::memory_order_relaxed);
  }
  return l2;
}

}  // namespace sp

extern "C" {

sp_status sp_relayout_seq2head(const void* const* in, void* const* out, int ntensors, int N,
                               int b, int s, int h, int d, void* stream) {
  return relayout(in, out, ntensors, N, b, s, h, d, true, stream);
}

sp_status sp_relayout_head2seq(const void* const* in, void* const* out, int ntensors, int N,
                               int b, int s, int h, int d, void* stream) {
  return relayout(in, out, ntensors, N, b, s, h, d, false, stream);
}

sp_status sp_relayout(const void* in, void* out, int N, const int64_t shape[4], int scatter_dim,
                      int gather_dim, void* stream) {
  if (shape == nullptr) return SP_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (shape[i] < 1 || shape[i] > INT32_MAX) return SP_ERR_INVALID_ARG;
  if (N < 1) return SP_ERR_INVALID_ARG;
  const int b = static_cast<int>(shape[0]), d = static_cast<int>(shape[3]);
  const void* src[1] = {in};
  void* dst[1] = {out};
  if (scatter_dim == 2 && gather_dim == 1) {
    // per-rank input [b][s/N][h][d]: heads scattered, sequence gathered
    const int64_t s = shape[1] * N;
    if (s > INT32_MAX) return SP_ERR_INVALID_ARG;
    return relayout(src, dst, 1, N, b, static_cast<int>(s), static_cast<int>(shape[2]), d, true,
                    stream);
  }
  if (scatter_dim == 1 && gather_dim == 2) {
    // per-rank input [b][s][h/N][d]: sequence scattered, heads gathered
    const int64_t h = shape[2] * N;
    if (h > INT32_MAX) return SP_ERR_INVALID_ARG;
    return relayout(src, dst, 1, N, b, static_cast<int>(shape[1]), static_cast<int>(h), d, false,
                    stream);
  }
  return SP_ERR_UNSUPPORTED;
}

sp_status sp_relayout_seq2head_packed(const void* qkv, void* const* out, int N, int b, int s,
                                      int h, int d, void* stream) {
  if (h < 1 || d < 1) return SP_ERR_INVALID_ARG;
  const void* in[3];
  packed_parts(qkv, h, d, in);
  return relayout(in, out, 3, N, b, s, h, d, true, stream, static_cast<int64_t>(3) * h * d);
}

sp_status sp_relayout_head2seq_packed(const void* const* in, void* qkv, int N, int b, int s,
                                      int h, int d, void* stream) {
  if (h < 1 || d < 1) return SP_ERR_INVALID_ARG;
  const void* part[3];
  packed_parts(qkv, h, d, part);
  void* out[3] = {const_cast<void*>(part[0]), const_cast<void*>(part[1]),
                  const_cast<void*>(part[2])};
  return relayout(in, out, 3, N, b, s, h, d, false, stream, static_cast<int64_t>(3) * h * d);
}

sp_status sp_attn_fwd(const sp_attn_params* p, void* o, float* lse, void* stream) {
  AttnGeom g;
  sp_status st = check_attn(p, &g);
  if (st != SP_OK) return st;
  if (!aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return SP_ERR_MISALIGNED;
  if (empty_problem(g)) return SP_OK;   // o and lse have no elements (may be null)
  if (o == nullptr || lse == nullptr) return SP_ERR_INVALID_ARG;
  FwdArgs a{};
  const Layouts L = layouts_of(p, g);
  if (!encode_rows_map(&a.tq, p->q, g.d, L.heads_total, L.shards, L.q)) return SP_ERR_CUDA;
  // no keys: every row gets out = 0 and lse = -inf, and no K or V tile is ever loaded
  if (g.sk > 0 && (!encode_rows_map(&a.tk, p->k, g.d, L.heads_total, L.shards, L.k) ||
                   !encode_rows_map(&a.tv, p->v, g.d, L.heads_total, L.shards, L.v)))
    return SP_ERR_CUDA;
  a.aq = L.q;
  a.ak = L.k;
  a.o = o;
  a.ao = L.o;
  a.lse = lse;
  a.g = g;
  a.status = status_word();
  if (a.status == nullptr) return SP_ERR_CUDA;
  return launch_attn_fwd(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

size_t sp_attn_bwd_workspace_size(const sp_attn_params* p) {
  AttnGeom g;
  if (check_attn(p, &g) != SP_OK) return 0;
  return workspace_layout(g).total;
}

sp_status sp_attn_bwd(const sp_attn_params* p, const void* o, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                      void* stream) {
  AttnGeom g;
  sp_status st = check_attn(p, &g);
  if (st != SP_OK) return st;
  // as for q, k, v: the tensors of the query rows may be null when there are none, dk
  // and dv when there are no keys
  const bool none = g.B == 0 || g.H == 0;
  if (((o == nullptr || lse == nullptr || dout == nullptr || dq == nullptr) &&
       !(none || g.sq == 0)) ||
      ((dk == nullptr || dv == nullptr) && !(none || g.sk == 0)))
    return SP_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return SP_ERR_MISALIGNED;
  if (g.B == 0 || g.H == 0) return SP_OK;
  const WorkspaceLayout w = workspace_layout(g);
  // the dQ accumulator is addressed by 32-bit TMA row coordinates
  if (static_cast<int64_t>(g.B) * g.H * padded_rows(g.sq) > INT32_MAX) return SP_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < w.total) return SP_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SP_ERR_MISALIGNED;
  BwdArgs a{};
  const Layouts L = layouts_of(p, g);
  if (g.sq > 0 && g.sk > 0) {
    if (!encode_rows_map(&a.tq, p->q, g.d, L.heads_total, L.shards, L.q) ||
        !encode_rows_map(&a.tk, p->k, g.d, L.heads_total, L.shards, L.k) ||
        !encode_rows_map(&a.tv, p->v, g.d, L.heads_total, L.shards, L.v) ||
        !encode_rows_map(&a.tdo, dout, g.d, L.heads_total, L.shards, L.o))
      return SP_ERR_CUDA;
  }
  a.aq = L.q;
  a.ak = L.k;
  a.av = L.v;
  a.ao = L.o;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.dq_off);
  a.row_stats = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.stats_off);
  a.dq_accumulate = p->dq_accumulate != 0;
  a.g = g;
  a.status = status_word();
  if (a.status == nullptr) return SP_ERR_CUDA;
  return launch_attn_bwd(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

sp_status sp_attn_merge(const sp_merge_params* p, void* stream) {
  if (p == nullptr) return SP_ERR_INVALID_ARG;
  if (p->B < 0 || p->H < 0 || p->sq < 0) return SP_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SP_ERR_UNSUPPORTED;
  // with no rows every tensor is empty and may be null
  const bool none = p->B == 0 || p->H == 0 || p->sq == 0;
  if (!none && (p->o_part == nullptr || p->lse_part == nullptr || p->o_acc == nullptr ||
                p->lse_acc == nullptr))
    return SP_ERR_INVALID_ARG;
  if (!aligned16(p->o_part) || !aligned16(p->o_acc) || !strides_ok(p->part_stride) ||
      (reinterpret_cast<uintptr_t>(p->lse_part) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(p->lse_acc) & 3u) != 0)
    return SP_ERR_MISALIGNED;
  if (p->o_out != nullptr && (!aligned16(p->o_out) || !strides_ok(p->out_stride)))
    return SP_ERR_MISALIGNED;
  if (p->B == 0 || p->H == 0 || p->sq == 0) return SP_OK;
  MergeArgs a;
  a.B = p->B;
  a.H = p->H;
  a.sq = p->sq;
  a.d = p->d;
  a.init = p->init != 0;
  a.o_part = p->o_part;
  a.lse_part = p->lse_part;
  a.o_acc = p->o_acc;
  a.lse_acc = p->lse_acc;
  a.o_out = p->o_out;
  for (int i = 0; i < 3; ++i) {
    a.part_stride[i] = p->part_stride[i];
    a.out_stride[i] = p->out_stride[i];
  }
  return launch_attn_merge(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SP_OK
                                                                                 : SP_ERR_CUDA;
}

sp_status sp_selftest_wait_timeout(void* stream) {
  uint32_t* st = status_word();
  if (st == nullptr) return SP_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

sp_status sp_get_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SP_ERR_CUDA;
  uint32_t* addr = status_word();
  if (addr == nullptr) return SP_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, addr, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SP_ERR_CUDA;
  if (cudaMemsetAsync(addr, 0, sizeof word, s) != cudaSuccess) return SP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SP_ERR_CUDA;
  if (word & kStatusTimeout) return SP_ERR_TIMEOUT;
  if (word == kStatusBadKeyLen) return SP_ERR_INVALID_ARG;
  if (word != 0) return SP_ERR_CUDA;
  return SP_OK;
}

const char* sp_status_string(sp_status s) {
  switch (s) {
    case SP_OK: return "ok";
    case SP_ERR_INVALID_ARG: return "invalid argument";
    case SP_ERR_UNSUPPORTED: return "unsupported problem";
    case SP_ERR_MISALIGNED: return "misaligned pointer or stride";
    case SP_ERR_CUDA: return "CUDA error";
    case SP_ERR_TIMEOUT: return "device-side wait timed out";
    case SP_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

}  // extern "C"
