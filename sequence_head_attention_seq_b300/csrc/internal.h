// internal.h -- declarations shared by the library's translation units only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "sp.h"

namespace sp {

// The calling thread's current CUDA context (the device's primary context when the
// runtime made it current), or null when none is current or the driver is unreachable.
void* current_context();

// Device address of one of the library's __device__ variables, cached per CUDA
// context: every context that loads the library holds its own copy of each such
// variable, so an address looked up in one context is not valid in another (a caller
// may run in its own driver-API context instead of the device's primary one).
// `lookup` runs with the context current and returns the address (null on failure).
class ContextAddressCache {
 public:
  template <class Lookup>
  void* get(Lookup lookup) {
    void* ctx = current_context();
    if (ctx == nullptr) return nullptr;
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < n_; ++i)
      if (entries_[i].ctx == ctx) return entries_[i].addr;
    void* addr = lookup();
    if (addr != nullptr && n_ < kEntries) entries_[n_++] = Entry{ctx, addr};
    return addr;
  }

 private:
  static constexpr int kEntries = 256;
  struct Entry {
    void* ctx;
    void* addr;
  };
  std::mutex mu_;
  Entry entries_[kEntries];
  int n_ = 0;
};

// Device address of the status word that kernels OR error codes into, in the current
// context (null if it cannot be found).
uint32_t* status_word();

constexpr int kMaxRelayoutTensors = SP_MAX_RELAYOUT_TENSORS;

// shard_row: element pitch of a shard-side row (0: h*d; 3*h*d for packed Q/K/V, whose
// tensor t starts t*h*d elements into each row).
cudaError_t launch_relayout(const void* const* in, void* const* out, int ntensors, int N, int b,
                            int s, int h, int d, bool to_heads, cudaStream_t stream,
                            int64_t shard_row = 0);

// Problem geometry after validation (see sp_attn_params).
struct AttnGeom {
  int B, H, sq, sk, d;
  int causal;
  int q_offset;               // query row 0's position relative to key row 0 (may be < 0)
  const int32_t* key_len;     // device, may be null
  const uint8_t* key_mask;    // device [B][key_mask_stride] bytes, may be null
  int64_t key_mask_stride;
  int seq_shards;             // 1: plain strided tensors; N > 1: sequence-shard layout
  float scale;                // softmax scale
  float scale_log2;           // scale * log2(e)
};

// log2 of the largest power of two that divides `heads` and is at most `cap` (0 when cap
// < 2): a group size with no partial last group.
int group_shift(int64_t heads, int64_t cap);
// L2 bytes of the current device (0 if unknown), queried once per device.
int64_t device_l2_bytes();

// CTA -> (batch entry x head, work class) for a launch of heads x `classes` CTAs in groups
// of 2^gshift heads (which divides the head count): within a group, class 0 (the
// heaviest) of every head first.
__device__ __forceinline__ void cta_order(int cta, int classes, int gshift, int* bh, int* cls) {
  const int per_group = classes << gshift;
  const int g = cta / per_group;
  const int r = cta - g * per_group;
  *cls = r >> gshift;
  *bh = (g << gshift) + (r & ((1 << gshift) - 1));
}

// Rows of the per-head statistics arrays in the backward workspace (sq rounded to 128).
inline int64_t padded_rows(int sq) { return (static_cast<int64_t>(sq) + 127) / 128 * 128; }

// Where head j of sequence row t of attention batch entry e sits in a bf16 tensor with
// head_dim contiguous (element offsets):
//     off = (e / bi) * group + (e % bi) * batch + (t / sl) * shard + (t % sl) * row + j * head
// The plain layout [B][S][H][d] with strides (s0, s1, s2) has bi = B, sl = S,
// group = shard = 0.  The sequence-shard layout of the Ulysses step,
// [N][b][s/N][N*H][d], read as N*b entries (entry g*b + bb = head group g of batch row
// bb) has bi = b, sl = s/N, group = H*d (the group's first head), batch = (s/N)*N*H*d,
// shard = b*(s/N)*N*H*d, row = N*H*d.  The tensor map of such a tensor is 5-D:
// (d, heads, sl, bi, shards) with head coordinate (e / bi) * group_heads + j.
struct RowAddr {
  int64_t group, batch, shard, row, head;
  int bi, sl;
  int group_heads;          // group / head: the head coordinate of a group's first head
  __host__ __device__ __forceinline__ int64_t off(int e, int t, int j) const {
    return static_cast<int64_t>(e / bi) * group + static_cast<int64_t>(e % bi) * batch +
           static_cast<int64_t>(t / sl) * shard + static_cast<int64_t>(t % sl) * row +
           static_cast<int64_t>(j) * head;
  }
};

// TMA coordinates (after the d chunk) of head j, row t of batch entry e.
struct TmaRow {
  int head, row, batch, shard;
};
__device__ __forceinline__ TmaRow tma_row(const RowAddr& a, int e, int t, int j) {
  return TmaRow{(e / a.bi) * a.group_heads + j, t % a.sl, e % a.bi, t / a.sl};
}

// RowAddr of a plain [B][S][H][d] tensor with element strides (batch, seq, head).
RowAddr plain_rows(const int64_t stride[3], int B, int S);
// RowAddr of a sequence-shard tensor [N][b][S/N][N*H][d], contiguous.
RowAddr shard_rows(int N, int b, int S, int H, int d);

// 5-D TMA map over a bf16 tensor described by `a` (heads_total heads, `shards` sequence
// shards), box = 64 columns of d x 128 rows of one shard, 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, const void* base, int d, int heads_total, int shards,
                     const RowAddr& a);


// 2-D TMA map over a bf16 matrix of `outer` rows of `inner` elements at a pitch of
// `pitch` elements, box = box_inner x box_outer, 128-byte swizzle (box_inner = 64).
bool encode_2d_bf16_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                        int64_t pitch, uint32_t box_inner, uint32_t box_outer);

// C[M][N] (+)= sum_k A[m][k] B[n][k] in bf16 with fp32 accumulation (gemm.cu).  A is
// K-major ([M][K], pitch lda) or, with a_mn, MN-major ([K][M]); B likewise ([N][K] or
// [K][N], pitch ldb); C row-major with pitch ldc.  All pitches and N multiples of 8
// elements, all pointers 16-byte aligned.
struct GemmArgs {
  const void* a;
  const void* b;
  void* c;
  int64_t lda, ldb, ldc;
  int M, N, K;
  bool a_mn, b_mn;
  bool accumulate;
  uint32_t* status;
};
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream);

struct FwdArgs {
  CUtensorMap tq, tk, tv;
  RowAddr aq, ak;       // layouts of q (and o's row coordinates) and k/v
  void* o;
  RowAddr ao;
  float* lse;
  AttnGeom g;
  uint32_t* status;
};
cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t stream);

struct BwdArgs {
  CUtensorMap tq, tk, tv, tdo;
  RowAddr aq, ak, av, ao;   // layouts of q/dq, k/dk, v/dv, o/dout
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;      // workspace: fp32, [B][H] blocks of rows * d (layout per d in attn_bwd.cu)
  float* row_stats;   // workspace: [B][H][2][rows] fp32 (-lse*log2e, D)
  bool dq_accumulate; // keep dq_acc from the previous call instead of zeroing it
  AttnGeom g;
  uint32_t* status;
};
cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream);

// Merge of one key chunk's attention result into a running accumulator (sp_attn_merge).
struct MergeArgs {
  int B, H, sq, d;
  int init;
  const void* o_part;
  int64_t part_stride[3];
  const float* lse_part;
  float* o_acc;
  float* lse_acc;
  void* o_out;            // may be null
  int64_t out_stride[3];
};
cudaError_t launch_attn_merge(const MergeArgs& a, cudaStream_t stream);

}  // namespace sp
