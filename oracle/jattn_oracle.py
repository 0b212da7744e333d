"""CPU oracle for MM-DiT joint attention with QK-RMSNorm (forward and backward).

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
definition the CUDA path is checked against.  Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the library itself
never does, and this module imports nothing from the library.

What it computes (re-diffusion README):
  * "architecture flowchart": inside each DiT layer the text-stream and
    image-stream Q/K/V are concatenated as ``[c; x]`` (text first), one
    multi-head self-attention runs over the joint sequence, and the result is
    split back per stream.
  * "design notes" table, row "QK norm": RMSNorm is applied to Q and to K
    (not V), with a learned gain.
  * "attention fix" section: the manual attention materialises the full
    B x 12 x N x N score matrix and applies softmax to it; routing the same
    Q/K/V layout ``[B, H, N, d]`` through scaled-dot-product attention gives
    the same function without the matrix.  This oracle is the materialised
    form, in float64.

Readings where the pages are silent (each one listed in the design notes):
  * RMSNorm over the head dim d per (b, h, n): r = (mean_j x_j^2 + eps)^(-1/2),
    x_hat = g * x * r, eps = 1e-6 inside the root, one gain vector of length d
    shared by all heads.
  * Scale 1/sqrt(d) applied to the normalised scores; LSE is the natural log.
  * q_hat and k_hat are bf16 activations (bf16 training, same layout fed to
    SDPA), so they are rounded to bf16 (nearest-even) before the scores; the
    backward treats that rounding as the identity (straight-through).
  * No mask, dropout or causality.

Parity pins (tests): central finite differences of every input, a float64
torch cross-check (``F.rms_norm``, SDPA math path, autograd), closed forms
(all-equal keys, N = 1), and invariants (softmax rows sum to one, token
permutation equivariance, head independence, linearity in V, scale
invariance of the norm, sum_j x_j dx_j = 0 at eps = 0, sum over keys of
dk_hat = 0, sum over keys of dv = sum over queries of dout).
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


# ---------------------------------------------------------------------------
# bf16 rounding of the normalised activations
# ---------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits (7 stored); a float64 keeps 53, so the
    45 low mantissa bits are rounded away directly from the float64 bits
    (one rounding, no float32 detour).  Valid for finite values in the normal
    float32 range and for zero, which is all this workload produces.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    low_bits = np.uint64(45)
    half = np.uint64((1 << 44) - 1)
    lsb = (u >> low_bits) & np.uint64(1)
    u = (u + half + lsb) & ~np.uint64((1 << 45) - 1)
    return u.view(np.float64)


# ---------------------------------------------------------------------------
# QK-RMSNorm ("design notes" table, row "QK norm")
# ---------------------------------------------------------------------------
def rmsnorm_fwd(x: np.ndarray, g: np.ndarray, eps: float = EPS):
    """x_hat = g * x * r with r = (mean over d of x^2 + eps)^(-1/2).

    x: [..., d] float64, g: [d].  Returns (x_hat, r) with r of shape [..., 1].
    """
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return g * x * r, r


def rmsnorm_bwd(x: np.ndarray, g: np.ndarray, r: np.ndarray, dxhat: np.ndarray):
    """Exact gradient of x_hat = g * x * r(x).

    With u = g * dxhat:  dx = r * u - (r^3 / d) * x * sum_j(u_j x_j),
    and dg = sum over all leading axes of dxhat * x * r.
    """
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    d = x.shape[-1]
    u = g * dxhat
    dx = r * u - (r ** 3 / d) * x * np.sum(u * x, axis=-1, keepdims=True)
    dg = np.sum((dxhat * x * r).reshape(-1, d), axis=0)
    return dx, dg


# ---------------------------------------------------------------------------
# Softmax attention with a materialised score matrix ("attention fix" section)
# ---------------------------------------------------------------------------
def attention_fwd_head(qh: np.ndarray, kh: np.ndarray, v: np.ndarray, scale: float):
    """One (b, h): S = scale * qh kh^T, LSE = ln sum_j exp(S_ij), P = exp(S - LSE), O = P v."""
    S = (qh @ kh.T) * scale
    m = S.max(axis=1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(S - m), axis=1, keepdims=True))
    P = np.exp(S - lse)
    O = P @ v
    return O, lse[:, 0], P


def attention_bwd_head(qh, kh, v, P, O, dout, scale):
    """Gradient of L = sum(dout * O) for one (b, h), given the forward's P and O.

    dV = P^T dO;  dP = dO V^T;  D_i = sum_c dO_ic O_ic;  dS = P * (dP - D);
    dqh = scale * dS kh;  dkh = scale * dS^T qh.
    """
    dv = P.T @ dout
    dP = dout @ v.T
    D = np.sum(dout * O, axis=1, keepdims=True)
    dS = P * (dP - D)
    dqh = (dS @ kh) * scale
    dkh = (dS.T @ qh) * scale
    return dqh, dkh, dv


# ---------------------------------------------------------------------------
# Whole path
# ---------------------------------------------------------------------------
def _as64(a):
    return np.asarray(a, dtype=np.float64)


def joint_attention_fwd(q, k, v, gq, gk, eps: float = EPS, round_qk: bool = True, return_state: bool = False):
    """Forward of QK-RMSNorm + softmax attention over [B, H, N, d] inputs.

    Returns (O [B,H,N,d] float64, LSE [B,H,N] float64) and, if
    ``return_state``, a dict with the normalised q_hat/k_hat and the 1/rms
    factors r_q/r_k ([B,H,N]).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    scale = 1.0 / np.sqrt(d)
    qh, rq = rmsnorm_fwd(q, gq, eps)
    kh, rk = rmsnorm_fwd(k, gk, eps)
    if round_qk:
        qh, kh = round_to_bf16(qh), round_to_bf16(kh)
    O = np.empty_like(v)
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], lse[b, h], _ = attention_fwd_head(qh[b, h], kh[b, h], v[b, h], scale)
    if return_state:
        return O, lse, {"qhat": qh, "khat": kh, "rq": rq[..., 0], "rk": rk[..., 0]}
    return O, lse


def joint_attention_bwd(q, k, v, gq, gk, dout, eps: float = EPS, round_qk: bool = True,
                        heads=None, return_state: bool = False):
    """Forward and backward of the whole path.

    Returns dict with O, LSE, dq, dk, dv ([B,H,N,d] float64 / [B,H,N]) and
    dgq, dgk ([d]).  ``heads``: optional list of (b, h) pairs to restrict the
    work to (then dq/dk/dv/O/LSE hold zeros elsewhere and dgq/dgk only sum
    over the listed heads).
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    B, H, N, d = q.shape
    scale = 1.0 / np.sqrt(d)
    qh, rq = rmsnorm_fwd(q, gq, eps)
    kh, rk = rmsnorm_fwd(k, gk, eps)
    if round_qk:
        qh, kh = round_to_bf16(qh), round_to_bf16(kh)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    O = np.zeros_like(v)
    lse = np.zeros((B, H, N))
    dqh = np.zeros_like(q)
    dkh = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, h in heads:
        O[b, h], lse[b, h], P = attention_fwd_head(qh[b, h], kh[b, h], v[b, h], scale)
        dqh[b, h], dkh[b, h], dv[b, h] = attention_bwd_head(qh[b, h], kh[b, h], v[b, h], P, O[b, h],
                                                            dout[b, h], scale)
    mask = np.zeros((B, H, 1, 1))
    for b, h in heads:
        mask[b, h] = 1.0
    dq, dgq = rmsnorm_bwd(q, gq, rq, dqh * mask)
    dk, dgk = rmsnorm_bwd(k, gk, rk, dkh * mask)
    out = {"O": O, "LSE": lse, "dq": dq * mask, "dk": dk * mask, "dv": dv, "dgq": dgq, "dgk": dgk}
    if return_state:
        out.update(qhat=qh, khat=kh, rq=rq[..., 0], rk=rk[..., 0], dqhat=dqh, dkhat=dkh)
    return out


def joint_attention_streams(q_txt, k_txt, v_txt, q_img, k_img, v_img, gq, gk, eps: float = EPS):
    """Per-stream form of the flowchart: concat [c; x] on the token axis, attend, split.

    Inputs are [B, H, N_txt, d] (caption stream) and [B, H, N_img, d] (image
    stream).  Returns (O_txt, O_img, LSE).
    """
    q = np.concatenate([_as64(q_txt), _as64(q_img)], axis=2)
    k = np.concatenate([_as64(k_txt), _as64(k_img)], axis=2)
    v = np.concatenate([_as64(v_txt), _as64(v_img)], axis=2)
    O, lse = joint_attention_fwd(q, k, v, gq, gk, eps)
    n_txt = q_txt.shape[2]
    return O[:, :, :n_txt], O[:, :, n_txt:], lse


# ---------------------------------------------------------------------------
# QKV projection per stream, then QK-RMSNorm ("architecture flowchart":
# adaLN -> QKV per stream -> concat [c; x] -> QK-RMSNorm -> SDPA)
# ---------------------------------------------------------------------------
def qkv_projection(x, w, b, H: int):
    """One stream's QKV projection with that stream's weights.

    x: [B, N_s, C] tokens; w: [3 H d, C], laid out like a linear layer's
    weight (output row j = x . w[j]): rows h d .. h d + d - 1 are head h of q,
    rows H d + h d .. of k, rows 2 H d + h d .. of v; b: [3 H d] or None.
    Returns (Y, Y_bf16), both [3, B, H, N_s, d] (q, k, v stacked): Y = x w^T + b
    exactly in float64, and its single rounding to bf16 (the projection's
    bf16 output in bf16 training).
    """
    x, w = _as64(x), _as64(w)
    B, N_s, _ = x.shape
    d = w.shape[0] // (3 * H)
    Y = x @ w.T
    if b is not None:
        Y = Y + _as64(b)
    Y = Y.reshape(B, N_s, 3, H, d).transpose(2, 0, 3, 1, 4)
    return Y, round_to_bf16(Y)


def qkv_norm_streams(x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk, H: int, eps: float = EPS):
    """Both streams projected, joined caption-first along the token axis, and
    Q, K normalised: what the fused projection call produces.

    Returns a dict: y_exact [3, B, H, N, d] (before rounding), q, k, v
    [B, H, N, d] (bf16 values), qhat, khat (bf16-rounded RMSNorm of q, k) and
    rq, rk [B, H, N] (each row's 1/rms).
    """
    parts = [qkv_projection(x_txt, w_txt, b_txt, H), qkv_projection(x_img, w_img, b_img, H)]
    y_exact = np.concatenate([p[0] for p in parts], axis=3)
    q, k, v = np.concatenate([p[1] for p in parts], axis=3)
    qh, rq = rmsnorm_fwd(q, gq, eps)
    kh, rk = rmsnorm_fwd(k, gk, eps)
    return {"y_exact": y_exact, "q": q, "k": k, "v": v, "qhat": round_to_bf16(qh), "khat": round_to_bf16(kh),
            "rq": rq[..., 0], "rk": rk[..., 0]}


def joint_attention_varlen_bwd(q, k, v, gq, gk, dout, cu_seqlens, eps: float = EPS, round_qk: bool = True):
    """Packed sequences of different lengths (re-diffusion README: the
    aspect-bucketed training data, and multi-resolution training on its
    roadmap): every sequence is its own joint-attention problem.

    Inputs are [H, T, d]; sequence s is rows cu_seqlens[s] .. cu_seqlens[s+1]-1
    of every head.  Each sequence goes through ``joint_attention_bwd`` as a
    batch of one; the gain gradients sum over the sequences.  Returns the same
    keys with O, dq, dk, dv [H, T, d] and LSE [H, T].
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    H, T, d = q.shape
    cu = [int(c) for c in cu_seqlens]
    if cu[0] != 0 or cu[-1] != T or any(b <= a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0, end at T and increase strictly")
    out = {"O": np.zeros_like(v), "LSE": np.zeros((H, T)), "dq": np.zeros_like(q), "dk": np.zeros_like(k),
           "dv": np.zeros_like(v), "dgq": np.zeros(d), "dgk": np.zeros(d)}
    for a, b in zip(cu, cu[1:]):
        r = joint_attention_bwd(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], gq, gk, dout[None, :, a:b],
                                eps=eps, round_qk=round_qk)
        for key in ("O", "dq", "dk", "dv"):
            out[key][:, a:b] = r[key][0]
        out["LSE"][:, a:b] = r["LSE"][0]
        out["dgq"] += r["dgq"]
        out["dgk"] += r["dgk"]
    return out


def attention_one_row(q_row, K, V, gq, gk, eps: float = EPS, round_qk: bool = True):
    """O and LSE of a single query row against the full key/value set of its head.

    Used to check sampled rows of large workloads one by one.
    q_row: [d]; K, V: [N, d].
    """
    d = K.shape[-1]
    qh, _ = rmsnorm_fwd(_as64(q_row)[None, :], gq, eps)
    kh, _ = rmsnorm_fwd(_as64(K), gk, eps)
    if round_qk:
        qh, kh = round_to_bf16(qh), round_to_bf16(kh)
    O, lse, _ = attention_fwd_head(qh, kh, _as64(V), 1.0 / np.sqrt(d))
    return O[0], lse[0]
