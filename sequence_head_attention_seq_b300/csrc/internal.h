// internal.h -- declarations shared by the library's translation units only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sp.h"

namespace sp {

constexpr int kMaxRelayoutTensors = SP_MAX_RELAYOUT_TENSORS;

cudaError_t launch_relayout(const void* const* in, void* const* out, int ntensors, int N, int b,
                            int s, int h, int d, bool to_heads, cudaStream_t stream);

// Problem geometry after validation (see sp_attn_params).
struct AttnGeom {
  int B, H, sq, sk, d;
  int causal;
  int q_offset;               // query row 0's position relative to key row 0 (may be < 0)
  const int32_t* key_len;     // device, may be null
  const uint8_t* key_mask;    // device [B][key_mask_stride] bytes, may be null
  int64_t key_mask_stride;
  float scale;                // softmax scale
  float scale_log2;           // scale * log2(e)
};

// Rows of the per-head statistics arrays in the backward workspace (sq rounded to 128).
inline int64_t padded_rows(int sq) { return (static_cast<int64_t>(sq) + 127) / 128 * 128; }

// 4-D TMA map over a [B][S][H][d] bf16 tensor (element strides for batch, seq,
// head), box = 64 columns of d x 128 rows of S, 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, const void* base, int d, int S, int H, int B,
                     const int64_t stride[3]);

// 2-D TMA map over the fp32 dQ accumulator viewed as [rows_total][d], box = 32
// columns x 32 rows, 128-byte swizzle (the backward reduces dQ tiles into it).
bool encode_acc_map(CUtensorMap* map, const float* base, int d, int64_t rows_total);

struct FwdArgs {
  CUtensorMap tq, tk, tv;
  void* o;
  int64_t o_stride[3];
  float* lse;
  AttnGeom g;
  uint32_t* status;
};
cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t stream);

struct BwdArgs {
  CUtensorMap tq, tk, tv, tdo;
  CUtensorMap tdq;     // over dq_acc (encode_acc_map)
  const void* o;
  const void* dout;
  int64_t o_stride[3];
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int64_t q_stride[3], k_stride[3], v_stride[3];
  float* dq_acc;      // workspace: [B][H][rows][d] fp32
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
