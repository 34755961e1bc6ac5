// host_step.cu -- one Ulysses attention step on HOST-resident shards, with the
// host<->device traffic overlapped with the attention kernels.
//
// The regrouping of "Parallel multi-head attention" section 2.2 and the long-context-
// attention issue "关于数据分割和合并" (every head group needs its heads from every
// sequence shard) is, for one head group, a strided gather: N*b runs of s/N rows of
// (h/N)*d contiguous elements at a pitch of h*d.  A 2-D copy does exactly that, so the
// copy engines move each head group between the host shard layout and a head-major
// device buffer while they transfer it, and no relayout kernel runs on this path.
//
// Per unit u, a head group or half of one (slot = u % 3: unit u+1's inputs move in and
// unit u-1's results move out while u computes, and the third slot lets the inputs run
// a whole unit ahead):
//   h2d stream     : Q, K, V of u into the slot            -> qkv_ready[slot]
//                    dO of u                               -> do_ready[slot]
//   compute stream : attention forward of u (waits qkv_ready, and out_free of u-3)
//                                                          -> o_ready[slot]
//                    attention backward of u (waits do_ready) -> grads_ready[slot]
//   d2h stream     : O of u to the host (waits o_ready), then dQ, dK, dV (waits
//                    grads_ready)                          -> out_free[slot]
// The h2d stream refills a slot only after the backward that last read it
// (grads_ready of u-3).  (Measured on B300, 70B-shaped step from host memory: two slots
// 61.44-61.75 ms, three 60.97-61.40 ms: with the host link about as fast as the kernels,
// the inputs of the next unit no longer wait for the backward two units back.)  The first and the last head group go as two halves of their
// heads: only the first unit's inputs and the last unit's results are not overlapped
// with kernels, so halving those units halves the exposed transfer time.  Events are created for the call and released at its end
// (their pending records complete on their own); no device memory is allocated.
#include <cuda_runtime.h>

#include <vector>

#include "internal.h"

namespace sp {
namespace {

constexpr size_t kAlign = 256;
constexpr int kSlots = 3;   // device buffer slots the units cycle through

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct HostGeom {
  int N, b, s, h, d, H, sl;   // H = heads per group, sl = rows per shard
  size_t elems;               // elements of one group's tensor: b * s * H * d
};

bool host_geom(int N, int b, int s, int h, int d, HostGeom* g) {
  if (N < 1 || b < 1 || s < 1 || h < 1 || (d != 64 && d != 128)) return false;
  if (s % N != 0 || h % N != 0) return false;
  g->N = N;
  g->b = b;
  g->s = s;
  g->h = h;
  g->d = d;
  g->H = h / N;
  g->sl = s / N;
  g->elems = static_cast<size_t>(b) * s * g->H * d;
  return true;
}

// The attention problem of `nh` heads of one head group in their head-major slot
// buffers [b][s][nh][d].
sp_attn_params group_params(const HostGeom& g, int nh, const void* q, const void* k,
                            const void* v, int causal, const int32_t* key_len, float scale) {
  sp_attn_params p{};
  p.q = q;
  p.k = k;
  p.v = v;
  const int64_t st[3] = {static_cast<int64_t>(g.s) * nh * g.d, static_cast<int64_t>(nh) * g.d,
                         g.d};
  for (int i = 0; i < 3; ++i) p.q_stride[i] = p.k_stride[i] = p.v_stride[i] = p.o_stride[i] = st[i];
  p.B = g.b;
  p.H = nh;
  p.sq = p.sk = g.s;
  p.d = g.d;
  p.causal = causal;
  p.key_len = key_len;
  p.softmax_scale = scale;
  p.seq_shards = 1;
  return p;
}

struct Layout {
  size_t tensor;      // one slot tensor (bf16)
  size_t lse;         // one slot's lse (fp32 [b][H][s])
  size_t slot;        // 8 tensors + lse
  size_t bwd;         // backward workspace, shared by the slots
  size_t total;
};

Layout layout_of(const HostGeom& g, int causal) {
  Layout l;
  l.tensor = align_up(g.elems * 2);
  l.lse = align_up(static_cast<size_t>(g.b) * g.H * g.s * 4);
  l.slot = 8 * l.tensor + l.lse;
  // only the geometry matters for the size: any 16-byte-aligned stand-in pointer will do
  const void* stand_in = reinterpret_cast<const void*>(static_cast<uintptr_t>(kAlign));
  const sp_attn_params p = group_params(g, g.H, stand_in, stand_in, stand_in, causal, nullptr,
                                       0.0f);
  l.bwd = align_up(sp_attn_bwd_workspace_size(&p));
  l.total = kSlots * l.slot + l.bwd;
  return l;
}

// A unit of work: heads j0 .. j0+nh-1 of head group grp.
struct Unit {
  int grp, j0, nh;
};

// Copy one unit of one tensor between the host shard layout [N][b][s/N][h][d] and a
// head-major device buffer [b][s][nh][d].  For b = 1 the shards follow each other at
// the same host pitch, so one 2-D copy moves the whole unit.
cudaError_t copy_unit(const HostGeom& g, const Unit& u, void* host, void* dev, bool to_device,
                      cudaStream_t st) {
  const size_t e = 2;   // bf16
  const size_t width = static_cast<size_t>(u.nh) * g.d * e;
  const size_t hpitch = static_cast<size_t>(g.h) * g.d * e;
  const int runs_n = g.b == 1 ? 1 : g.N;
  const int rows = g.b == 1 ? g.s : g.sl;
  for (int n = 0; n < runs_n; ++n)
    for (int bb = 0; bb < g.b; ++bb) {
      // host row (n, bb, 0) and device row (bb, n * s/N)
      const size_t hrow = (static_cast<size_t>(n) * g.b + bb) * g.sl;
      const size_t drow = static_cast<size_t>(bb) * g.s + static_cast<size_t>(n) * g.sl;
      char* hp = static_cast<char*>(host) + hrow * hpitch +
                 (static_cast<size_t>(u.grp) * g.H + u.j0) * g.d * e;
      char* dp = static_cast<char*>(dev) + drow * width;
      const cudaError_t err =
          to_device ? cudaMemcpy2DAsync(dp, width, hp, hpitch, width, rows, cudaMemcpyHostToDevice, st)
                    : cudaMemcpy2DAsync(hp, hpitch, dp, width, width, rows, cudaMemcpyDeviceToHost, st);
      if (err != cudaSuccess) return err;
    }
  return cudaSuccess;
}

bool pinned_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

struct Events {
  static constexpr int kCount = 2 + 5 * kSlots;
  cudaEvent_t e[kCount] = {};
  bool create() {
    for (auto& x : e)
      if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
  ~Events() {
    for (auto& x : e)
      if (x) cudaEventDestroy(x);
  }
};

}  // namespace
}  // namespace sp

using namespace sp;

extern "C" {

size_t sp_ulysses_host_workspace_size(int N, int b, int s, int h, int d, int causal) {
  HostGeom g;
  if (!host_geom(N, b, s, h, d, &g) || (causal != 0 && causal != 1)) return 0;
  const Layout lay = layout_of(g, causal);
  return lay.bwd == 0 ? 0 : lay.total;
}

sp_status sp_ulysses_step_host(const sp_ulysses_host_params* p, void* workspace,
                               size_t workspace_bytes, void* stream, void* h2d_stream,
                               void* d2h_stream) {
  if (p == nullptr) return SP_ERR_INVALID_ARG;
  HostGeom g;
  if (p->N < 1 || p->b < 1 || p->s < 1 || p->h < 1 || p->s % p->N != 0 || p->h % p->N != 0 ||
      (p->causal != 0 && p->causal != 1))
    return SP_ERR_INVALID_ARG;
  if (!host_geom(p->N, p->b, p->s, p->h, p->d, &g)) return SP_ERR_UNSUPPORTED;
  const void* in[4] = {p->q, p->k, p->v, p->dout};
  void* out[4] = {p->o, p->dq, p->dk, p->dv};
  for (const void* x : in)
    if (x == nullptr) return SP_ERR_INVALID_ARG;
  for (const void* x : out)
    if (x == nullptr) return SP_ERR_INVALID_ARG;
  if (workspace == nullptr || h2d_stream == nullptr || d2h_stream == nullptr ||
      h2d_stream == stream || d2h_stream == stream || h2d_stream == d2h_stream)
    return SP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return SP_ERR_MISALIGNED;
  // key lengths are int32: checked here so that nothing is queued before a refusal
  if ((reinterpret_cast<uintptr_t>(p->key_len) & 3u) != 0) return SP_ERR_MISALIGNED;
  const Layout lay = layout_of(g, p->causal);
  if (lay.bwd == 0) return SP_ERR_UNSUPPORTED;   // a group problem the kernels refuse
  if (workspace_bytes < lay.total) return SP_ERR_WORKSPACE;
  for (const void* x : in)
    if (!pinned_host(x)) return SP_ERR_INVALID_ARG;
  for (const void* x : out)
    if (!pinned_host(x)) return SP_ERR_INVALID_ARG;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t hs = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ds = static_cast<cudaStream_t>(d2h_stream);
  Events ev;
  if (!ev.create()) return SP_ERR_CUDA;
  cudaEvent_t start = ev.e[0], done = ev.e[1];
  cudaEvent_t qkv_ready[kSlots], do_ready[kSlots], o_ready[kSlots], grads_ready[kSlots],
      out_free[kSlots];
  for (int i = 0; i < kSlots; ++i) {
    qkv_ready[i] = ev.e[2 + i];
    do_ready[i] = ev.e[2 + kSlots + i];
    o_ready[i] = ev.e[2 + 2 * kSlots + i];
    grads_ready[i] = ev.e[2 + 3 * kSlots + i];
    out_free[i] = ev.e[2 + 4 * kSlots + i];
  }

  char* ws = static_cast<char*>(workspace);
  auto slot_tensor = [&](int slot, int t) { return ws + slot * lay.slot + t * lay.tensor; };
  auto slot_lse = [&](int slot) { return reinterpret_cast<float*>(ws + slot * lay.slot + 8 * lay.tensor); };
  void* bwd_ws = ws + kSlots * lay.slot;

#define SP_CHECK(x)                            \
  do {                                         \
    if ((x) != cudaSuccess) return SP_ERR_CUDA; \
  } while (0)
  // the copy streams start after whatever the caller queued before this call
  SP_CHECK(cudaEventRecord(start, cs));
  SP_CHECK(cudaStreamWaitEvent(hs, start, 0));
  SP_CHECK(cudaStreamWaitEvent(ds, start, 0));
  // the first and the last head group in two halves of their heads
  std::vector<Unit> units;
  const int half = g.H / 2;
  for (int grp = 0; grp < g.N; ++grp) {
    if (half > 0 && (grp == 0 || grp == g.N - 1)) {
      units.push_back({grp, 0, half});
      units.push_back({grp, half, g.H - half});
      if (g.N == 1) break;
    } else {
      units.push_back({grp, 0, g.H});
    }
  }
  // Queue every unit.  A failure part-way leaves copies queued on hs and ds: the
  // caller's stream is then joined to both before the error is returned, so that
  // synchronising the caller's stream also waits for every copy that touches the host
  // buffers (the caller may free or reuse them after that).
  auto enqueue_units = [&]() -> sp_status {
    for (size_t ui = 0; ui < units.size(); ++ui) {
      const Unit& u = units[ui];
      const int slot = static_cast<int>(ui % kSlots);
      // slot tensors: 0 q, 1 k, 2 v, 3 dout, 4 o, 5 dq, 6 dk, 7 dv
      if (ui >= kSlots) SP_CHECK(cudaStreamWaitEvent(hs, grads_ready[slot], 0));
      for (int t = 0; t < 3; ++t)
        SP_CHECK(copy_unit(g, u, const_cast<void*>(in[t]), slot_tensor(slot, t), true, hs));
      SP_CHECK(cudaEventRecord(qkv_ready[slot], hs));
      SP_CHECK(copy_unit(g, u, const_cast<void*>(in[3]), slot_tensor(slot, 3), true, hs));
      SP_CHECK(cudaEventRecord(do_ready[slot], hs));

      SP_CHECK(cudaStreamWaitEvent(cs, qkv_ready[slot], 0));
      if (ui >= kSlots) SP_CHECK(cudaStreamWaitEvent(cs, out_free[slot], 0));
      const sp_attn_params ap = group_params(g, u.nh, slot_tensor(slot, 0), slot_tensor(slot, 1),
                                             slot_tensor(slot, 2), p->causal, p->key_len,
                                             p->softmax_scale);
      sp_status st = sp_attn_fwd(&ap, slot_tensor(slot, 4), slot_lse(slot), cs);
      if (st != SP_OK) return st;
      SP_CHECK(cudaEventRecord(o_ready[slot], cs));
      SP_CHECK(cudaStreamWaitEvent(cs, do_ready[slot], 0));
      st = sp_attn_bwd(&ap, slot_tensor(slot, 4), slot_lse(slot), slot_tensor(slot, 3),
                       slot_tensor(slot, 5), slot_tensor(slot, 6), slot_tensor(slot, 7), bwd_ws,
                       lay.bwd, cs);
      if (st != SP_OK) return st;
      SP_CHECK(cudaEventRecord(grads_ready[slot], cs));

      SP_CHECK(cudaStreamWaitEvent(ds, o_ready[slot], 0));
      SP_CHECK(copy_unit(g, u, out[0], slot_tensor(slot, 4), false, ds));
      SP_CHECK(cudaStreamWaitEvent(ds, grads_ready[slot], 0));
      for (int t = 1; t < 4; ++t)
        SP_CHECK(copy_unit(g, u, out[t], slot_tensor(slot, 4 + t), false, ds));
      SP_CHECK(cudaEventRecord(out_free[slot], ds));
    }
    return SP_OK;
  };
  const sp_status queued = enqueue_units();
  if (queued != SP_OK) {
    if (cudaEventRecord(qkv_ready[0], hs) == cudaSuccess) cudaStreamWaitEvent(cs, qkv_ready[0], 0);
    if (cudaEventRecord(done, ds) == cudaSuccess) cudaStreamWaitEvent(cs, done, 0);
    return queued;
  }
  // the caller's stream resumes once every result has reached the host
  SP_CHECK(cudaEventRecord(done, ds));
  SP_CHECK(cudaStreamWaitEvent(cs, done, 0));
#undef SP_CHECK
  return SP_OK;
}

}  // extern "C"
