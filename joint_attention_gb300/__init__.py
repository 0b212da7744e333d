"""GB300-native MM-DiT joint attention with QK-RMSNorm (forward and backward).

The compute path is libjattn.so (hand-written sm_103a CUDA kernels behind a C
ABI, declared in include/jattn.h); this package is its thin ctypes binding
plus small conveniences that allocate the output tensors with torch.
"""
from __future__ import annotations

from ._binding import (KERNEL_KINDS, STATUS, STATUS_CODE, JattnError, declared_symbols, jattn_bwd, jattn_fwd,
                       jattn_fwd_noalloc, jattn_fwd_varlen, jattn_bwd_varlen, jattn_selftest_wait_timeout, jattn_set_sm_limit,
                       jattn_set_deterministic, jattn_kernel_name, jattn_last_device_error, jattn_last_error_message, jattn_profile_enable, jattn_profile_read,
                       jattn_profile_reset, jattn_status_string, jattn_version, load_library, profile_snapshot,
                       jattn_saved_bytes, jattn_saved_bytes_varlen, jattn_fwd_train, jattn_bwd_train,
                       jattn_fwd_train_varlen, jattn_bwd_train_varlen, jattn_qkv_norm, jattn_fwd_saved)

__all__ = ["STATUS", "STATUS_CODE", "JattnError", "declared_symbols", "jattn_bwd", "jattn_fwd",
           "jattn_last_device_error", "jattn_status_string", "jattn_version", "load_library", "forward",
           "backward", "KERNEL_KINDS", "jattn_kernel_name", "jattn_profile_enable", "jattn_profile_read",
           "jattn_profile_reset", "profile_snapshot", "jattn_last_error_message", "jattn_fwd_noalloc",
           "jattn_fwd_varlen", "jattn_bwd_varlen", "forward_varlen", "backward_varlen",
           "jattn_selftest_wait_timeout", "jattn_set_sm_limit", "jattn_set_deterministic", "jattn_saved_bytes",
           "jattn_saved_bytes_varlen", "jattn_fwd_train", "jattn_bwd_train", "jattn_fwd_train_varlen",
           "jattn_bwd_train_varlen", "forward_train", "backward_train", "jattn_qkv_norm", "jattn_fwd_saved",
           "qkv_norm"]


def forward(q, k, v, gq, gk, n_txt: int, stream=None):
    """out, lse = joint attention of [B, H, N, d] bf16 CUDA tensors (text rows first)."""
    import torch

    B, H, N, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    jattn_fwd(q, k, v, gq, gk, B, H, N - n_txt, n_txt, d, out, lse, stream)
    return out, lse


def backward(q, k, v, gq, gk, out, lse, dout, n_txt: int, stream=None):
    """dq, dk, dv, dgq, dgk for the upstream gradient dout."""
    import torch

    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dgq = torch.empty_like(gq)
    dgk = torch.empty_like(gk)
    jattn_bwd(q, k, v, gq, gk, out, lse, dout, dq, dk, dv, dgq, dgk, B, H, N - n_txt, n_txt, d, stream)
    return dq, dk, dv, dgq, dgk


def forward_varlen(q, k, v, gq, gk, cu_seqlens, stream=None):
    """out, lse for packed sequences: q, k, v [H, T, d] bf16 CUDA tensors, sequence s in rows
    cu_seqlens[s] .. cu_seqlens[s+1]-1 of every head (cu_seqlens: host ints)."""
    import torch

    H, T, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    jattn_fwd_varlen(q, k, v, gq, gk, cu_seqlens, H, d, out, lse, stream)
    return out, lse


def backward_varlen(q, k, v, gq, gk, out, lse, dout, cu_seqlens, stream=None):
    """dq, dk, dv, dgq, dgk for packed sequences (layouts as forward_varlen)."""
    import torch

    H, T, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dgq = torch.empty_like(gq)
    dgk = torch.empty_like(gk)
    jattn_bwd_varlen(q, k, v, gq, gk, out, lse, dout, dq, dk, dv, dgq, dgk, cu_seqlens, H, d, stream)
    return dq, dk, dv, dgq, dgk


def forward_train(q, k, v, gq, gk, n_txt: int, stream=None):
    """out, lse, saved: a training forward of [B, H, N, d] bf16 CUDA tensors that keeps the
    normalised q / k in `saved` (a uint8 CUDA tensor) for backward_train."""
    import torch

    B, H, N, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    saved = torch.empty(jattn_saved_bytes(B, H, N - n_txt, n_txt, d), dtype=torch.uint8, device=q.device)
    jattn_fwd_train(q, k, v, gq, gk, B, H, N - n_txt, n_txt, d, out, lse, saved, stream)
    return out, lse, saved


def backward_train(q, k, v, gq, gk, out, lse, dout, saved, n_txt: int, stream=None):
    """dq, dk, dv, dgq, dgk from forward_train's outputs and `saved`."""
    import torch

    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dgq = torch.empty_like(gq)
    dgk = torch.empty_like(gk)
    jattn_bwd_train(q, k, v, gq, gk, out, lse, dout, saved, dq, dk, dv, dgq, dgk, B, H, N - n_txt, n_txt, d, stream)
    return dq, dk, dv, dgq, dgk


def qkv_norm(x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk, H: int, stream=None):
    """q, k, v, saved: the QKV projections of the image tokens x_img [B, N_img, C] and the caption
    tokens x_txt [B, N_txt, C] (bf16 CUDA tensors; weights [3 H d, C] bf16, biases [3 H d] fp32 or
    None) into the joint [B, H, N, d] layout, with q_hat, k_hat and 1/rms in `saved` for
    jattn_fwd_saved / backward_train."""
    import torch

    B, N_img, C = x_img.shape
    N_txt = x_txt.shape[1]
    d = gq.shape[0]
    N = N_img + N_txt
    dev = x_img.device
    q = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    k, v = torch.empty_like(q), torch.empty_like(q)
    saved = torch.empty(jattn_saved_bytes(B, H, N_img, N_txt, d), dtype=torch.uint8, device=dev)
    jattn_qkv_norm(x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk, B, H, N_img, N_txt, d, C, q, k, v, saved,
                   stream)
    return q, k, v, saved
