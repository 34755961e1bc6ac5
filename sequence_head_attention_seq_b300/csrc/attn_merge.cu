// attn_merge.cu -- ring / blockwise attention: merge one key chunk's (o, lse) into a
// running fp32 accumulator.
//
// "adv07: Sequence Parallel", sections 5 and 7: Ring Attention passes the K/V blocks
// around a ring and every device attends to one block at a time, like a distributed
// chunked prefill.  The pages do not spell out how the per-block results combine; for
// a softmax split over disjoint key sets the combination is exact:
//     lse = log(exp(lse_acc) + exp(lse_part))
//     o   = exp(lse_acc - lse) * o_acc + exp(lse_part - lse) * o_part
// A side with lse = -inf (no visible key) has weight 0; both -inf leaves o = 0.
//
// Bandwidth bound: per element, 2 bytes of o_part read, 4 bytes of o_acc read (not on
// the first chunk) and 4 written, plus 2 bytes of o_out on the last chunk.  One thread
// moves 8 consecutive head-dim elements (16-byte bf16 and 32-byte fp32 vectors);
// the d/8 threads of one row sit in the same warp, which lets one of them update the
// row's lse after all of them have read the old value.  All loads are issued before
// any arithmetic, so each thread waits for memory once.
#include "internal.h"
#include "ptx.cuh"

namespace sp {
namespace {

template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const MergeArgs a) {
  constexpr int kVec = D / 8;                    // threads per row
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(a.B) * a.sq * a.H * kVec;
  const bool active = t < total;
  const int c = static_cast<int>(t % kVec);
  int64_t row = t / kVec;                        // (bb, i, h), h fastest
  const int h = static_cast<int>(row % a.H);
  row /= a.H;
  const int i = static_cast<int>(row % a.sq);
  const int bb = static_cast<int>(row / a.sq);
  const int64_t lse_at = (static_cast<int64_t>(bb) * a.H + h) * a.sq + i;
  float lse_new = -INFINITY;
  if (active) {
    // every load first (they do not depend on each other), so that a thread waits for
    // memory once rather than for the statistics and then for the accumulator
    const float lp = __ldg(a.lse_part + lse_at);
    const float la = a.init ? -INFINITY : a.lse_acc[lse_at];
    const uint4 part = __ldg(reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(a.o_part) + bb * a.part_stride[0] +
        static_cast<int64_t>(i) * a.part_stride[1] + h * a.part_stride[2] + c * 8));
    float4* acc = reinterpret_cast<float4*>(a.o_acc + ((static_cast<int64_t>(bb) * a.sq + i) *
                                                           a.H + h) * D + c * 8);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
    if (!a.init) {   // uniform across the launch
      x = acc[0];
      y = acc[1];
    }
    const float m = fmaxf(lp, la);
    float wa = 0.0f, wp = 0.0f;
    if (m != -INFINITY) {
      const float ea = expf(la - m), ep = expf(lp - m);
      const float sum = ea + ep;
      lse_new = m + logf(sum);
      wa = ea / sum;
      wp = ep / sum;
    }
    // a side with weight 0 is left out (not multiplied by 0): the accumulator of a
    // row that has seen no key yet is never used, whatever it holds
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&part);
    const float xa[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
    float o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(p2[k]);
      o[2 * k] = wa != 0.0f ? fmaf(wa, xa[2 * k], wp * f.x) : wp * f.x;
      o[2 * k + 1] = wa != 0.0f ? fmaf(wa, xa[2 * k + 1], wp * f.y) : wp * f.y;
    }
    acc[0] = make_float4(o[0], o[1], o[2], o[3]);
    acc[1] = make_float4(o[4], o[5], o[6], o[7]);
    if (a.o_out != nullptr) {
      uint4 out;
      out.x = pack_bf16x2(o[0], o[1]);
      out.y = pack_bf16x2(o[2], o[3]);
      out.z = pack_bf16x2(o[4], o[5]);
      out.w = pack_bf16x2(o[6], o[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o_out) + bb * a.out_stride[0] +
                                static_cast<int64_t>(i) * a.out_stride[1] +
                                h * a.out_stride[2] + c * 8) = out;
    }
  }
  // every thread of the row has read the old lse before it is replaced
  __syncwarp();
  if (active && c == 0) a.lse_acc[lse_at] = lse_new;
}

}  // namespace

cudaError_t launch_attn_merge(const MergeArgs& a, cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(a.B) * a.sq * a.H * (a.d / 8);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  if (a.d == 128)
    attn_merge_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  else
    attn_merge_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace sp
