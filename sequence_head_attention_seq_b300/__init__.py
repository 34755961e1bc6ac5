"""Causal multi-head attention on the Ulysses sequence/head layout, for B300 (sm_103a).

The computation lives in ``libsp.so`` (C ABI in ``include/sp.h``, CUDA kernels in
``csrc/``).  This package is its thin binding:

    sp_relayout_seq2head / sp_relayout_head2seq   sequence shards <-> head groups
    sp_relayout                                   the same as an all-to-all (scatter/gather dims)
    sp_attn_fwd                                   attention forward (out + lse)
    sp_attn_bwd                                   attention backward (dq, dk, dv)
    sp_attn_merge                                 ring / blockwise: merge key-chunk results
    sp_linear_fwd / sp_linear_bwd                 projections around attention (GEMMs)
    UlyssesAttention                              the whole step on shard tensors
    UlyssesHostStep / sp_ulysses_step_host        the step on host shards, transfers overlapped
    ring_attention_fwd / ring_attention_bwd       blockwise attention over key chunks
    AttentionLayer                                projections + regrouping + attention
    attention / seq_all_to_all / ulysses_attention  the same calls as torch.autograd
                                                  Functions (gradients through libsp)

Nothing here computes attention in Python; if the native library is missing the
calls raise.
"""
from .binding import (SpError, sp_attn_bwd, sp_attn_bwd_workspace_size, sp_attn_fwd,
                      sp_attn_merge, sp_get_device_status, sp_linear_bwd, sp_linear_fwd,
                      sp_relayout, sp_relayout_head2seq,
                      sp_relayout_head2seq_packed, sp_relayout_seq2head,
                      sp_relayout_seq2head_packed, sp_status_string,
                      sp_ulysses_host_workspace_size, sp_ulysses_step_host)
from .autograd import attention, seq_all_to_all, ulysses_attention
from .pipeline import (AttentionLayer, UlyssesAttention, UlyssesHostStep, ring_attention_bwd,
                       ring_attention_fwd)

__all__ = ["SpError", "sp_attn_bwd", "sp_attn_bwd_workspace_size", "sp_attn_fwd", "sp_attn_merge",
           "sp_get_device_status", "sp_relayout", "sp_relayout_head2seq", "sp_relayout_seq2head",
           "sp_relayout_seq2head_packed", "sp_relayout_head2seq_packed", "sp_linear_fwd",
           "sp_linear_bwd",
           "sp_status_string", "sp_ulysses_host_workspace_size", "sp_ulysses_step_host",
           "UlyssesAttention", "UlyssesHostStep", "AttentionLayer", "ring_attention_fwd",
           "ring_attention_bwd", "attention", "seq_all_to_all", "ulysses_attention"]
