/*
 * sp.h -- C ABI of libsp: causal multi-head attention on the Ulysses
 * sequence/head layout, forward and backward, for NVIDIA B300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are bf16 in DEVICE memory, owned by the caller; the library never
 *    allocates, frees or keeps a pointer after a call returns.  Each buffer must hold
 *    every element that its shape and strides address: the library cannot see
 *    allocation sizes and does not check them.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call only
 *    enqueues work on it: no host synchronisation, no allocation.
 *  - Argument errors are detected on the host and returned BEFORE anything is
 *    launched (SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_MISALIGNED).
 *  - A failed launch returns SP_ERR_CUDA.  Faults found while the kernels run
 *    (a device wait that gave up, a key length outside [0, sk] read from device
 *    memory) are reported by sp_get_device_status().
 *  - Calls are thread-safe; the library holds no per-call state.
 */
#ifndef SP_H
#define SP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sp_status {
    SP_OK = 0,
    SP_ERR_INVALID_ARG = 1,  /* a size, count, flag or pointer is out of range */
    SP_ERR_UNSUPPORTED = 2,  /* valid in principle, not implemented (e.g. head_dim not 64/128) */
    SP_ERR_MISALIGNED = 3,   /* a pointer or stride breaks the 16-byte rule */
    SP_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    SP_ERR_TIMEOUT = 5,      /* a device-side wait exceeded its limit; results are invalid */
    SP_ERR_WORKSPACE = 6     /* the workspace passed to sp_attn_bwd is too small */
} sp_status;

#define SP_MAX_RELAYOUT_TENSORS 8

/*
 * Ulysses regrouping: sequence shards -> head groups.
 *
 * Defined by: long-context-attention issue "关于数据分割和合并" (each rank
 * starts with 1/N of the sequence of Q/K/V, an all-to-all that works like a
 * transpose gives every rank the full sequence for a subset of the heads);
 * transformers PR 31525 "Support deepspeed sequence parallel" (shard r holds
 * rows [r*s/N, (r+1)*s/N), inputs of the all-to-all are [b, s/p, n, h]);
 * "Parallel multi-head attention", section 2.2 (heads are assigned to devices
 * in contiguous blocks).  On one GPU the all-to-all is this local permutation.
 *
 *   in[t]  : [N][b][s/N][h][d]   shard r = sequence rows r*s/N .. (r+1)*s/N-1
 *   out[t] : [N][b][s][h/N][d]   group g = heads g*h/N .. (g+1)*h/N-1
 *   out[t][g][bb][r*s/N+u][j][c] = in[t][r][bb][u][g*h/N+j][c]
 *
 * in, out : HOST arrays of `ntensors` DEVICE pointers (1 <= ntensors <= 8), so
 *           Q, K and V (or dQ, dK, dV) move in one launch.  Elements are copied
 *           as opaque 16-bit words: the result is bit-exact.  in[t] and out[t]
 *           must not overlap.  Pointers 16-byte aligned.
 * Errors  : N < 1, b/s/h/d < 1, s % N or h % N != 0 -> SP_ERR_INVALID_ARG;
 *           a NULL pointer -> SP_ERR_INVALID_ARG; misalignment -> SP_ERR_MISALIGNED.
 */
sp_status sp_relayout_seq2head(const void* const* in, void* const* out, int ntensors,
                               int N, int b, int s, int h, int d, void* stream);

/*
 * Inverse regrouping: head groups -> sequence shards (the all-to-all after
 * attention in the same pages; each rank's output is (b, s/N, hidden)).
 *
 *   in[t]  : [N][b][s][h/N][d],  out[t] : [N][b][s/N][h][d]
 * Arguments and errors as sp_relayout_seq2head.
 */
sp_status sp_relayout_head2seq(const void* const* in, void* const* out, int ntensors,
                               int N, int b, int s, int h, int d, void* stream);

/*
 * The regrouping in the form of the sequence-parallel all-to-all of transformers PR
 * 31525 ("Support deepspeed sequence parallel"): every rank's tensor is 4-D, one
 * dimension is split across the N ranks (scatter_dim) and another is concatenated
 * from them (gather_dim).  On one GPU the N ranks' tensors are stacked along a leading
 * dimension of size N, in and out.
 *
 *   shape          : the per-rank INPUT shape [b][x][y][d] (4 entries, each >= 1)
 *   scatter 2, gather 1 : in [N][b][s/N][h][d] -> out [N][b][s][h/N][d]  (x = s/N, y = h;
 *                         the same as sp_relayout_seq2head with one tensor)
 *   scatter 1, gather 2 : in [N][b][s][h/N][d] -> out [N][b][s/N][h][d]  (x = s, y = h/N;
 *                         the same as sp_relayout_head2seq with one tensor)
 * Other (scatter_dim, gather_dim) pairs -> SP_ERR_UNSUPPORTED.  A NULL shape, an entry
 * below 1 or N < 1 -> SP_ERR_INVALID_ARG; otherwise arguments and errors as
 * sp_relayout_seq2head.
 */
sp_status sp_relayout(const void* in, void* out, int N, const int64_t shape[4], int scatter_dim,
                      int gather_dim, void* stream);

/*
 * Packed Q/K/V (the long-context-attention issue names a packed-QKV variant of its
 * attention, LongContextAttentionQKVPacked): one sequence-shard buffer holding all
 * three, [N][b][s/N][3][h][d], regrouped into three head-group buffers in one launch.
 *
 *   qkv    : DEVICE bf16 [N][b][s/N][3][h][d]; Q, K, V at index 0, 1, 2 of each row
 *   out[t] : DEVICE bf16 [N][b][s][h/N][d] for t = Q, K, V (HOST array of 3 pointers)
 * Bit-exact copy, as sp_relayout_seq2head; errors as sp_relayout_seq2head (the three
 * parts of qkv must be 16-byte aligned: h*d a multiple of 8).
 */
sp_status sp_relayout_seq2head_packed(const void* qkv, void* const* out, int N, int b, int s,
                                      int h, int d, void* stream);

/*
 * Inverse: three head-group buffers (e.g. dQ, dK, dV) into one packed sequence-shard
 * buffer [N][b][s/N][3][h][d].  in: HOST array of 3 DEVICE pointers.
 */
sp_status sp_relayout_head2seq_packed(const void* const* in, void* qkv, int N, int b, int s,
                                      int h, int d, void* stream);

/*
 * One attention problem.  Sources: "adv07: Sequence Parallel" (mini-vllm
 * tutorial), section 3 Q4: out[i] = softmax(q[i] K^T / sqrt(d)) V with a causal
 * mask that hides only future keys (j > i), a query shard masking by its GLOBAL
 * row position; section 4: a query shard attends to the full K/V prefix.
 * "Parallel multi-head attention", section 3.2: scores / sqrt(head_dim), an
 * additive mask, softmax in fp32.  transformers PR 31525: a key-padding mask
 * from (input_ids != pad).
 *
 * Key j is visible from query row i of batch entry bb iff
 *     (!causal || kv_offset + j <= q_offset + i)  &&  (key_len == NULL || j < key_len[bb])
 *     &&  (key_mask == NULL || key_mask[bb * key_mask_stride + j] != 0).
 * key_mask is a general per-key mask (transformers PR 31525: attention_mask =
 * input_ids != pad_token_id, pads anywhere); key_len is the right-padding special case.
 * q_offset and kv_offset are the global sequence positions of query row 0 and key
 * row 0: a query shard (split-Q) sets q_offset, a key chunk of ring / blockwise
 * attention sets kv_offset ("adv07: Sequence Parallel", sections 5 and 7: K/V blocks
 * passed around a ring, each device attending to one block at a time).
 * A row with no visible key returns out = 0, lse = -inf and no gradient.
 *
 * Layout: q, o, dout, dq are [B][sq][H][d]; k, v, dk, dv are [B][sk][H][d];
 * d is contiguous and the other strides (in ELEMENTS) are given per tensor.
 * Strides must be multiples of 8 elements and pointers 16-byte aligned.
 */
typedef struct sp_attn_params {
    const void* q;            /* bf16, device */
    const void* k;            /* bf16, device */
    const void* v;            /* bf16, device */
    int64_t q_stride[3];      /* batch, seq, head strides of q and dq */
    int64_t k_stride[3];      /* ... of k and dk */
    int64_t v_stride[3];      /* ... of v and dv */
    int64_t o_stride[3];      /* ... of o and dout */
    int B, H;                 /* batch entries (e.g. N*b head groups) and heads per entry */
    int sq, sk;               /* query rows and key rows */
    int d;                    /* head_dim: 64 or 128 */
    int causal;               /* 0 or 1 */
    int q_offset;             /* global sequence position of query row 0 (>= 0) */
    int kv_offset;            /* global sequence position of key row 0 (>= 0) */
    const int32_t* key_len;   /* NULL, or DEVICE [B] valid-key counts in [0, sk]; a count
                                 outside that range is clamped into it and reported by
                                 sp_get_device_status as SP_ERR_INVALID_ARG */
    float softmax_scale;      /* <= 0 selects 1/sqrt(d) */
    int dq_accumulate;        /* sp_attn_bwd only, 0 or 1: see sp_attn_bwd */
    const uint8_t* key_mask;  /* NULL, or DEVICE bytes [B][key_mask_stride]: key j of batch
                                 entry bb takes part iff key_mask[bb*stride + j] != 0;
                                 16-byte aligned */
    int64_t key_mask_stride;  /* bytes between batch rows: a multiple of 16, >= sk */
    int seq_shards;           /* 0 or 1: q, k, v, o, dout, dq, dk, dv use the strides above.
                                 N >= 2: all eight are in the Ulysses sequence-shard layout
                                 [N][B/N][sq/N][N*H][d] (contiguous; strides ignored), read
                                 as B = N*b batch entries, entry g*b + bb being head group g
                                 (heads g*H .. g*H+H-1) of batch row bb; needs sq == sk,
                                 B % N == 0, sq % N == 0 and (sq/N) % 128 == 0 */
} sp_attn_params;

/*
 * Forward: o = softmax(scale * q k^T + mask) v per (batch entry, head), and
 * lse = log(sum_j exp(scale * q.k_j)) over the visible keys (natural log),
 * both from fp32 accumulation; o is rounded to bf16 (nearest even).
 *
 * o   : DEVICE bf16, layout of q with o_stride.
 * lse : DEVICE fp32 [B][H][sq], contiguous.  Needed by sp_attn_bwd.
 * Empty sizes: B, H or sq equal to 0 leaves nothing to do (SP_OK, nothing launched);
 *         sk = 0 leaves every row without a visible key (o = 0, lse = -inf).  A tensor
 *         without elements may be NULL: q, o and lse when sq = 0, k and v when sk = 0,
 *         all of them when B or H is 0.
 * Errors: B, H, sq, sk < 0, q_offset < 0, kv_offset < 0, causal not 0/1, any other
 *         NULL pointer -> SP_ERR_INVALID_ARG; key_mask_stride < sk with a key_mask ->
 *         SP_ERR_INVALID_ARG; d not 64/128, q_offset + sq or kv_offset + sk above
 *         2^30 -> SP_ERR_UNSUPPORTED; pointer/stride alignment (key_mask and its
 *         stride included) -> SP_ERR_MISALIGNED.
 */
sp_status sp_attn_fwd(const sp_attn_params* p, void* o, float* lse, void* stream);

/*
 * Bytes of device workspace sp_attn_bwd needs for `p` (fp32 dQ accumulator and
 * per-row statistics, rounded up to 128-row tiles).  0 on invalid arguments.
 */
size_t sp_attn_bwd_workspace_size(const sp_attn_params* p);

/*
 * Backward of sp_attn_fwd given dout (no formulas on the pages; the textbook
 * derivative of the forward definition, recomputing P from the saved lse):
 *     D_i   = sum_c dout_ic o_ic
 *     dS_ij = P_ij (dout_i . v_j - D_i)
 *     dq_i  = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dout_i
 * dq, dk, dv are written (not accumulated) in bf16 with the strides of q, k, v.
 *
 * o, lse     : the forward's outputs for the same p.
 * workspace  : DEVICE, >= sp_attn_bwd_workspace_size(p) bytes, 256-byte aligned,
 *              owned by the caller; its contents on entry do not matter unless
 *              p->dq_accumulate is set.
 * dq_accumulate = 1 (ring / blockwise attention, one call per key chunk with that
 *              chunk's k, v and kv_offset, and the merged o and lse): this call's dq
 *              contribution is added to the fp32 accumulator the previous call left in
 *              the same workspace (same B, H, sq, d), and dq receives the running sum.
 *              The per-row statistics of that call are reused too, so o, lse and dout
 *              must be the previous call's.  The first chunk's call uses
 *              dq_accumulate = 0.  dk and dv are always this call's (this chunk's)
 *              gradients.
 * Empty sizes as sp_attn_fwd: with sk = 0, dq = 0 (dk, dv have no elements and may be
 * NULL); with sq = 0 and sk > 0, dk = dv = 0 (o, lse, dout and dq may be NULL).
 * Errors as sp_attn_fwd, plus SP_ERR_WORKSPACE when workspace_bytes is too small.
 */
sp_status sp_attn_bwd(const sp_attn_params* p, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Ring / blockwise attention: merge the result of one key chunk into a running
 * accumulator.  "adv07: Sequence Parallel", section 5 (Ring Attention passes K/V
 * blocks around a ring, each device computing attention against one block at a time,
 * "like a distributed chunked prefill") and section 7.  The pages give no formula for
 * combining the blocks; this is the plain identity for a softmax split over disjoint
 * key sets, with per-chunk results (o_c, lse_c) from sp_attn_fwd (kv_offset = chunk
 * start):
 *     lse = log(exp(lse_acc) + exp(lse_part))
 *     o   = exp(lse_acc - lse) * o_acc + exp(lse_part - lse) * o_part
 * (a side with lse = -inf, no visible key, has weight 0; both -inf gives o = 0,
 * lse = -inf).  fp32 arithmetic.
 *
 * All pointers are DEVICE memory owned by the caller; rows are (bb, i, h) for
 * bb < B, i < sq, h < H, with head_dim d in {64, 128} contiguous:
 *   o_part   : bf16, element (bb, i, h, c) at bb*part_stride[0] + i*part_stride[1]
 *              + h*part_stride[2] + c (strides in elements, multiples of 8)
 *   lse_part : fp32 [B][H][sq] contiguous
 *   o_acc    : fp32 [B][sq][H][d] contiguous, updated in place
 *   lse_acc  : fp32 [B][H][sq] contiguous, updated in place
 *   o_out    : NULL, or bf16 with out_stride: also receives the merged output
 *              rounded to bf16 (nearest even), for the last chunk
 * init != 0 starts a new accumulation: o_acc and lse_acc are overwritten with the
 * partial (their contents on entry are not read).
 * B, H or sq equal to 0: nothing to merge (SP_OK; the tensors, all empty, may be NULL).
 * Errors: sizes < 0, d not 64/128 -> SP_ERR_INVALID_ARG / SP_ERR_UNSUPPORTED; NULL
 * required pointers -> SP_ERR_INVALID_ARG; pointers not 16-byte aligned or strides
 * not multiples of 8 -> SP_ERR_MISALIGNED.
 */
typedef struct sp_merge_params {
    int B, H, sq, d;
    int init;
    const void* o_part;
    int64_t part_stride[3];
    const float* lse_part;
    float* o_acc;
    float* lse_acc;
    void* o_out;
    int64_t out_stride[3];
} sp_merge_params;

sp_status sp_attn_merge(const sp_merge_params* p, void* stream);

/*
 * The projections around attention, as nn.Linear products with W [out][in] (row-major,
 * contiguous): "Parallel multi-head attention", sections 2.1-2.3 and 3.1, projects the
 * input with ColumnParallelLinear wq, wk, wv and the attention output with a
 * RowParallelLinear wo.  On one GPU the full weights are local; a single [3*h*d][dim]
 * weight gives the packed [..][3][h][d] layout that sp_relayout_seq2head_packed takes.
 *
 *   sp_linear_fwd : y[M][out] = x[M][in] . W^T
 *   sp_linear_bwd : dx[M][in] = dy[M][out] . W          (skipped when dx is NULL)
 *                   dW[out][in] = dy^T . x, or += with accumulate_dw = 1 (skipped when
 *                   dw is NULL)
 * bf16 in and out, fp32 accumulation, on the library's own tcgen05 GEMM (128 x 256 tiles,
 * TMA-fed, persistent); nothing is allocated.
 * M = 0: x, y, dy and dx have no elements (nothing is written, and they may be NULL);
 * dy^T . x is then the zero matrix, so dW is cleared (kept with accumulate_dw = 1).
 * All pointers DEVICE, 16-byte aligned.  Errors: M < 0, in or out < 1, accumulate_dw
 * not 0/1, required pointers NULL -> SP_ERR_INVALID_ARG; in or out not a multiple of 8,
 * misaligned pointers -> SP_ERR_MISALIGNED; a failed GEMM -> SP_ERR_CUDA.
 */
sp_status sp_linear_fwd(const void* x, const void* w, void* y, int M, int in, int out,
                        void* stream);
sp_status sp_linear_bwd(const void* dy, const void* x, const void* w, void* dx, void* dw, int M,
                        int in, int out, int accumulate_dw, void* stream);

/* Size of the device scratch array that sp_attn_bwd_noalloc uses (32 MiB). */
#define SP_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * sp_attn_bwd for callers that cannot allocate device memory: code running inside a
 * framework or runtime that owns all device memory (no cudaMalloc/cudaFree allowed on
 * its threads), or code bound to a fixed memory plan.  None of the cited pages has one.
 *
 * Instead of a caller-supplied workspace it uses a library-owned device array of
 * SP_NOALLOC_SCRATCH_BYTES, created on every GPU that loads the library and kept
 * until the process exits.  It never calls cudaMalloc, cudaFree or any allocating
 * routine.  Arguments, outputs and results are those of sp_attn_bwd.
 *
 *  - Problems whose workspace (sp_attn_bwd_workspace_size) exceeds
 *    SP_NOALLOC_SCRATCH_BYTES are rejected with SP_ERR_WORKSPACE before any launch.
 *  - dq_accumulate must be 0 (SP_ERR_INVALID_ARG otherwise): the shared scratch does
 *    not carry an accumulation from one call to the next.
 *  - Every CUDA context that loads the library holds its own copy of the array (the
 *    device's primary context, or a caller's own driver-API context).  The first call
 *    in a context looks up the array's device address with that context current and
 *    caches it per context; make that first call before capturing any stream.
 *  - All calls share the one array per device and it keeps whatever the last call
 *    left in it (every byte is rewritten before it is read, so nothing needs
 *    clearing).  Calls whose kernels overlap on the GPU (different streams without
 *    ordering between them) race on it: serialise them.
 */
sp_status sp_attn_bwd_noalloc(const sp_attn_params* p, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, void* stream);

/*
 * One Ulysses attention step (forward and backward) on HOST-resident shards, with the
 * host<->device transfers overlapped with the attention kernels.  "Parallel multi-head
 * attention", section 2.2, and the long-context-attention issue "关于数据分割和合并":
 * each head group needs its heads from every sequence shard.  Here the copy engines
 * perform that regrouping: head group g of a tensor is moved by 2-D copies (N*b runs of
 * s/N rows of (h/N)*d elements at a pitch of h*d; one copy when b = 1) between the host
 * shard layout and a head-major device buffer, and back for the results.  Group g's
 * copies in, its forward and backward on `stream`, and its copies out run on three
 * streams with group g+1's transfers overlapping group g's kernels (three buffer slots);
 * the first and the last group go as two halves of their heads, which halves the
 * transfers that no kernel can hide.
 *
 * The results equal those of sp_relayout_seq2head, sp_attn_fwd, sp_relayout_head2seq,
 * sp_relayout_seq2head (dout), sp_attn_bwd and sp_relayout_head2seq on the same data:
 * every head group is the independent attention problem [b][s][h/N][d].
 *
 * q, k, v, dout   : HOST bf16 [N][b][s/N][h][d] (shard r = sequence rows r*s/N ..),
 *                   PAGE-LOCKED (cudaHostAlloc / cudaHostRegister), read only.
 * o, dq, dk, dv   : HOST bf16, same layout, page-locked; written.  Valid once `stream`
 *                   has reached the point this call enqueued up to.
 * key_len         : NULL or DEVICE int32 [b] (keys of batch row bb: j < key_len[bb]).
 * softmax_scale   : <= 0 selects 1/sqrt(d).
 * workspace       : DEVICE, >= sp_ulysses_host_workspace_size(...) bytes, 256-byte
 *                   aligned, owned by the caller (three slots of eight group tensors, the
 *                   lse, and the backward workspace).
 * stream          : the kernels run on it, and it waits for the last result to reach
 *                   the host.  h2d_stream, d2h_stream: two further streams, distinct from
 *                   each other and from `stream`, non-blocking (cudaStreamNonBlocking)
 *                   for the transfers to overlap; both first wait for the work already
 *                   queued on `stream`.
 * The call creates a few CUDA events and releases them before it returns (their
 * pending records complete on their own); it allocates no memory and does not
 * synchronise the host.
 * Errors: N, b, s, h < 1, s % N or h % N != 0, causal not 0/1, a NULL pointer or
 *         stream, repeated streams, a host pointer that is not page-locked host memory
 *         -> SP_ERR_INVALID_ARG; d not 64/128 -> SP_ERR_UNSUPPORTED; workspace too
 *         small -> SP_ERR_WORKSPACE; workspace or key_len misaligned ->
 *         SP_ERR_MISALIGNED; all of these before anything is queued.  A failed CUDA
 *         call or a refusal by a kernel entry point part-way -> its status (SP_ERR_CUDA
 *         for a failed CUDA call); copies already queued by this call then still run,
 *         and `stream` is made to wait for both transfer streams before the call
 *         returns, so synchronising `stream` is enough before the host buffers are
 *         freed or reused.
 */
typedef struct sp_ulysses_host_params {
    int N, b, s, h, d;        /* shards, batch rows, full sequence, heads, head_dim */
    int causal;               /* 0 or 1 */
    float softmax_scale;
    const int32_t* key_len;   /* NULL or DEVICE [b] */
    const void* q;            /* HOST, page-locked: inputs */
    const void* k;
    const void* v;
    const void* dout;
    void* o;                  /* HOST, page-locked: results */
    void* dq;
    void* dk;
    void* dv;
} sp_ulysses_host_params;

/* Device workspace bytes of sp_ulysses_step_host; 0 on invalid arguments. */
size_t sp_ulysses_host_workspace_size(int N, int b, int s, int h, int d, int causal);

sp_status sp_ulysses_step_host(const sp_ulysses_host_params* p, void* workspace,
                               size_t workspace_bytes, void* stream, void* h2d_stream,
                               void* d2h_stream);

/*
 * Self-test of the failure path that every device-side wait shares: enqueues a
 * one-warp kernel that waits on an mbarrier nothing arrives on.  The wait gives up
 * after its limit (2 s), records the timeout in the device status word and the kernel
 * returns, so the context stays usable; sp_get_device_status then returns
 * SP_ERR_TIMEOUT (and clears the word).  SP_ERR_CUDA if the launch fails.
 */
sp_status sp_selftest_wait_timeout(void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word that the
 * kernels set since the last read: SP_ERR_TIMEOUT when a bounded device-side wait
 * gave up; SP_ERR_INVALID_ARG when the only event was a key_len entry outside
 * [0, sk] (the kernels clamped it, so their results are those of the clamped
 * length); SP_ERR_CUDA for a failed launch-time invariant inside a kernel or a
 * stream that reports an error.
 */
sp_status sp_get_device_status(void* stream);

/* Static, human-readable name of a status code. */
const char* sp_status_string(sp_status s);

#ifdef __cplusplus
}
#endif

#endif /* SP_H */
