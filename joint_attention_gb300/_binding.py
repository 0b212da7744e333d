"""ctypes binding of libjattn (include/jattn.h): argument marshalling only.

Every function here forwards to the C ABI of the same name; torch tensors are
accepted for convenience and passed as raw device pointers (torch provides
device memory and streams, nothing else).  There is no fallback: if the
library is missing the import of a call fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "jattn.h")
LIB_PATH = os.path.join(PKG, "libjattn.so")

STATUS = {
    0: "JATTN_OK",
    1: "JATTN_ERR_INVALID_ARG",
    2: "JATTN_ERR_UNSUPPORTED",
    3: "JATTN_ERR_MISALIGNED",
    4: "JATTN_ERR_ALIAS",
    5: "JATTN_ERR_CUDA",
    6: "JATTN_ERR_TIMEOUT",
    7: "JATTN_ERR_SCRATCH_LIMIT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class JattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = jattn_last_error_message() if status == 5 else ""
        super().__init__(f"{where}: {STATUS.get(status, status)} ({jattn_status_string(status)})"
                         + (f" [{detail}]" if detail else ""))


_lib = None


def load_library(path: str | None = None, build_if_missing: bool = False) -> ctypes.CDLL:
    """Loads libjattn.so (building it first only if asked)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        if build_if_missing:
            from .build import build
            p = build()
        else:
            raise FileNotFoundError(f"{p} not found: run joint_attention_gb300/build.py (or __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.jattn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.jattn_fwd.restype = i32
    lib.jattn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.jattn_fwd_noalloc.restype = i32
    lib.jattn_bwd.argtypes = [vp] * 13 + [i32] * 5 + [vp]
    lib.jattn_bwd.restype = i32
    i32p = ctypes.POINTER(ctypes.c_int)
    lib.jattn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, i32p, i32, i32, i32, vp, vp, vp]
    lib.jattn_fwd_varlen.restype = i32
    lib.jattn_bwd_varlen.argtypes = [vp] * 13 + [i32p, i32, i32, i32, vp]
    lib.jattn_bwd_varlen.restype = i32
    lib.jattn_last_device_error.argtypes = [vp]
    lib.jattn_last_device_error.restype = i32
    lib.jattn_selftest_wait_timeout.argtypes = [vp]
    lib.jattn_selftest_wait_timeout.restype = i32
    lib.jattn_status_string.argtypes = [i32]
    lib.jattn_status_string.restype = ctypes.c_char_p
    lib.jattn_version.argtypes = []
    lib.jattn_version.restype = i32
    lib.jattn_last_error_message.argtypes = []
    lib.jattn_last_error_message.restype = ctypes.c_char_p
    lib.jattn_profile_enable.argtypes = [i32]
    lib.jattn_profile_enable.restype = i32
    lib.jattn_profile_reset.argtypes = []
    lib.jattn_profile_reset.restype = i32
    lib.jattn_profile_read.argtypes = [i32, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]
    lib.jattn_profile_read.restype = i32
    lib.jattn_set_sm_limit.argtypes = [i32]
    lib.jattn_set_sm_limit.restype = i32
    lib.jattn_set_deterministic.argtypes = [i32]
    lib.jattn_set_deterministic.restype = i32
    lib.jattn_kernel_name.argtypes = [i32]
    lib.jattn_kernel_name.restype = ctypes.c_char_p
    sz = ctypes.c_size_t
    lib.jattn_saved_bytes.argtypes = [i32] * 5
    lib.jattn_saved_bytes.restype = sz
    lib.jattn_saved_bytes_varlen.argtypes = [i32p, i32, i32, i32]
    lib.jattn_saved_bytes_varlen.restype = sz
    lib.jattn_fwd_train.argtypes = [vp] * 5 + [i32] * 5 + [vp] * 4
    lib.jattn_fwd_train.restype = i32
    lib.jattn_bwd_train.argtypes = [vp] * 14 + [i32] * 5 + [vp]
    lib.jattn_bwd_train.restype = i32
    lib.jattn_fwd_train_varlen.argtypes = [vp] * 5 + [i32p, i32, i32, i32] + [vp] * 4
    lib.jattn_fwd_train_varlen.restype = i32
    lib.jattn_bwd_train_varlen.argtypes = [vp] * 14 + [i32p, i32, i32, i32, vp]
    lib.jattn_bwd_train_varlen.restype = i32
    lib.jattn_qkv_norm.argtypes = [vp] * 8 + [i32] * 6 + [vp] * 5
    lib.jattn_qkv_norm.restype = i32
    lib.jattn_fwd_saved.argtypes = [vp] + [i32] * 5 + [vp] * 4
    lib.jattn_fwd_saved.restype = i32
    if path is None:
        _lib = lib
    return lib


KERNEL_KINDS = 6


def jattn_profile_enable(on: bool = True) -> int:
    return load_library().jattn_profile_enable(1 if on else 0)


def jattn_profile_reset() -> int:
    return load_library().jattn_profile_reset()


def jattn_profile_read(kind: int) -> tuple[int, float]:
    """(launches, total milliseconds) of one kernel kind since the last reset."""
    n, ms = ctypes.c_int(0), ctypes.c_double(0.0)
    rc = load_library().jattn_profile_read(int(kind), ctypes.byref(n), ctypes.byref(ms))
    if rc != 0:
        raise JattnError(rc, "jattn_profile_read")
    return n.value, ms.value


def jattn_kernel_name(kind: int) -> str:
    return load_library().jattn_kernel_name(int(kind)).decode()


def profile_snapshot() -> dict:
    """{kernel name: (launches, total ms)} for every kernel kind."""
    return {jattn_kernel_name(k): jattn_profile_read(k) for k in range(KERNEL_KINDS)}


def declared_symbols(header: str = HEADER) -> list[str]:
    """Names of the functions include/jattn.h declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(jattn_\w+)\s*\(", text, flags=re.M)))


def _ptr(x, name: str, dtype=None, numel: int | None = None):
    """Raw pointer of a tensor (checked) or an int / None passed through."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch

    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor or an int pointer")
    if not x.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {x.dtype}")
    if numel is not None and x.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {x.numel()}")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def jattn_fwd(q, k, v, gq, gk, B: int, H: int, N_img: int, N_txt: int, d: int, out, lse, stream=None,
              check: bool = True) -> int:
    """C ABI jattn_fwd.  Tensors: q/k/v/out [B,H,N,d] bf16, gq/gk [d] fp32, lse [B,H,N] fp32."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e, r = B * H * N * d, B * H * N
    bf, f32 = torch.bfloat16, torch.float32
    rc = lib.jattn_fwd(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e), _ptr(gq, "gq", f32, d),
                       _ptr(gk, "gk", f32, d), B, H, N_img, N_txt, d, _ptr(out, "out", bf, e),
                       _ptr(lse, "lse", f32, r), _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_fwd")
    return rc


def jattn_fwd_noalloc(q, k, v, gq, gk, B: int, H: int, N_img: int, N_txt: int, d: int, out, lse, stream=None,
                      check: bool = True) -> int:
    """C ABI jattn_fwd_noalloc: jattn_fwd with its scratch in a fixed device array (no allocation)."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e, r = B * H * N * d, B * H * N
    bf, f32 = torch.bfloat16, torch.float32
    rc = lib.jattn_fwd_noalloc(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                               _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), B, H, N_img, N_txt, d,
                               _ptr(out, "out", bf, e), _ptr(lse, "lse", f32, r), _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_fwd_noalloc")
    return rc


def jattn_bwd(q, k, v, gq, gk, out, lse, dout, dq, dk, dv, dgq, dgk, B: int, H: int, N_img: int, N_txt: int,
              d: int, stream=None, check: bool = True) -> int:
    """C ABI jattn_bwd.  Gradients dq/dk/dv [B,H,N,d] bf16 and dgq/dgk [d] fp32 are overwritten."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e, r = B * H * N * d, B * H * N
    bf, f32 = torch.bfloat16, torch.float32
    rc = lib.jattn_bwd(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e), _ptr(gq, "gq", f32, d),
                       _ptr(gk, "gk", f32, d), _ptr(out, "out", bf, e), _ptr(lse, "lse", f32, r),
                       _ptr(dout, "dout", bf, e), _ptr(dq, "dq", bf, e), _ptr(dk, "dk", bf, e),
                       _ptr(dv, "dv", bf, e), _ptr(dgq, "dgq", f32, d), _ptr(dgk, "dgk", f32, d), B, H, N_img,
                       N_txt, d, _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_bwd")
    return rc


def _cu_array(cu_seqlens):
    """Host int array (ctypes) of the sequence offsets, and T and the count."""
    vals = [int(x) for x in cu_seqlens]
    arr = (ctypes.c_int * len(vals))(*vals)
    return arr, vals[-1] if vals else 0, len(vals) - 1


def jattn_fwd_varlen(q, k, v, gq, gk, cu_seqlens, H: int, d: int, out, lse, stream=None,
                     check: bool = True) -> int:
    """C ABI jattn_fwd_varlen.  q/k/v/out [H, T, d] bf16 (sequence s = rows cu[s]..cu[s+1]-1 of every
    head), gq/gk [d] fp32, lse [H, T] fp32; cu_seqlens a host sequence of n + 1 ints."""
    import torch

    lib = load_library()
    arr, T, n = _cu_array(cu_seqlens)
    e, r = H * T * d, H * T
    bf, f32 = torch.bfloat16, torch.float32
    rc = lib.jattn_fwd_varlen(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                              _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), arr, n, H, d,
                              _ptr(out, "out", bf, e), _ptr(lse, "lse", f32, r), _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_fwd_varlen")
    return rc


def jattn_bwd_varlen(q, k, v, gq, gk, out, lse, dout, dq, dk, dv, dgq, dgk, cu_seqlens, H: int, d: int,
                     stream=None, check: bool = True) -> int:
    """C ABI jattn_bwd_varlen (layouts as jattn_fwd_varlen)."""
    import torch

    lib = load_library()
    arr, T, n = _cu_array(cu_seqlens)
    e, r = H * T * d, H * T
    bf, f32 = torch.bfloat16, torch.float32
    rc = lib.jattn_bwd_varlen(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                              _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), _ptr(out, "out", bf, e),
                              _ptr(lse, "lse", f32, r), _ptr(dout, "dout", bf, e), _ptr(dq, "dq", bf, e),
                              _ptr(dk, "dk", bf, e), _ptr(dv, "dv", bf, e), _ptr(dgq, "dgq", f32, d),
                              _ptr(dgk, "dgk", f32, d), arr, n, H, d, _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_bwd_varlen")
    return rc


def jattn_saved_bytes(B: int, H: int, N_img: int, N_txt: int, d: int) -> int:
    """C ABI jattn_saved_bytes: size of the activation buffer of jattn_fwd_train / jattn_bwd_train."""
    return int(load_library().jattn_saved_bytes(B, H, N_img, N_txt, d))


def jattn_saved_bytes_varlen(cu_seqlens, H: int, d: int) -> int:
    """C ABI jattn_saved_bytes_varlen."""
    arr, _, n = _cu_array(cu_seqlens)
    return int(load_library().jattn_saved_bytes_varlen(arr, n, H, d))


def _saved_ptr(saved, nbytes: int):
    import torch

    if isinstance(saved, int) or saved is None:
        return saved
    if not isinstance(saved, torch.Tensor) or not saved.is_cuda or not saved.is_contiguous():
        raise ValueError("saved: expected a contiguous CUDA tensor")
    if saved.numel() * saved.element_size() < nbytes:
        raise ValueError(f"saved: needs {nbytes} bytes, got {saved.numel() * saved.element_size()}")
    return saved.data_ptr()


def jattn_fwd_train(q, k, v, gq, gk, B: int, H: int, N_img: int, N_txt: int, d: int, out, lse, saved,
                    stream=None, check: bool = True) -> int:
    """C ABI jattn_fwd_train: jattn_fwd that also fills `saved` (jattn_saved_bytes bytes) for jattn_bwd_train."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e, r = B * H * N * d, B * H * N
    bf, f32 = torch.bfloat16, torch.float32
    nb = jattn_saved_bytes(B, H, N_img, N_txt, d)
    rc = lib.jattn_fwd_train(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                             _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), B, H, N_img, N_txt, d,
                             _ptr(out, "out", bf, e), _ptr(lse, "lse", f32, r), _saved_ptr(saved, nb),
                             _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_fwd_train")
    return rc


def jattn_bwd_train(q, k, v, gq, gk, out, lse, dout, saved, dq, dk, dv, dgq, dgk, B: int, H: int, N_img: int,
                    N_txt: int, d: int, stream=None, check: bool = True) -> int:
    """C ABI jattn_bwd_train: jattn_bwd reading q_hat, k_hat and 1/rms from the forward's `saved`."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e, r = B * H * N * d, B * H * N
    bf, f32 = torch.bfloat16, torch.float32
    nb = jattn_saved_bytes(B, H, N_img, N_txt, d)
    rc = lib.jattn_bwd_train(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                             _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), _ptr(out, "out", bf, e),
                             _ptr(lse, "lse", f32, r), _ptr(dout, "dout", bf, e), _saved_ptr(saved, nb),
                             _ptr(dq, "dq", bf, e), _ptr(dk, "dk", bf, e), _ptr(dv, "dv", bf, e),
                             _ptr(dgq, "dgq", f32, d), _ptr(dgk, "dgk", f32, d), B, H, N_img, N_txt, d,
                             _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_bwd_train")
    return rc


def jattn_fwd_train_varlen(q, k, v, gq, gk, cu_seqlens, H: int, d: int, out, lse, saved, stream=None,
                           check: bool = True) -> int:
    """C ABI jattn_fwd_train_varlen (layouts as jattn_fwd_varlen)."""
    import torch

    lib = load_library()
    arr, T, n = _cu_array(cu_seqlens)
    e, r = H * T * d, H * T
    bf, f32 = torch.bfloat16, torch.float32
    nb = jattn_saved_bytes_varlen(cu_seqlens, H, d)
    rc = lib.jattn_fwd_train_varlen(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                                    _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), arr, n, H, d,
                                    _ptr(out, "out", bf, e), _ptr(lse, "lse", f32, r), _saved_ptr(saved, nb),
                                    _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_fwd_train_varlen")
    return rc


def jattn_bwd_train_varlen(q, k, v, gq, gk, out, lse, dout, saved, dq, dk, dv, dgq, dgk, cu_seqlens, H: int,
                           d: int, stream=None, check: bool = True) -> int:
    """C ABI jattn_bwd_train_varlen (layouts as jattn_fwd_varlen)."""
    import torch

    lib = load_library()
    arr, T, n = _cu_array(cu_seqlens)
    e, r = H * T * d, H * T
    bf, f32 = torch.bfloat16, torch.float32
    nb = jattn_saved_bytes_varlen(cu_seqlens, H, d)
    rc = lib.jattn_bwd_train_varlen(_ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e),
                                    _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), _ptr(out, "out", bf, e),
                                    _ptr(lse, "lse", f32, r), _ptr(dout, "dout", bf, e), _saved_ptr(saved, nb),
                                    _ptr(dq, "dq", bf, e), _ptr(dk, "dk", bf, e), _ptr(dv, "dv", bf, e),
                                    _ptr(dgq, "dgq", f32, d), _ptr(dgk, "dgk", f32, d), arr, n, H, d,
                                    _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_bwd_train_varlen")
    return rc


def jattn_qkv_norm(x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk, B: int, H: int, N_img: int, N_txt: int,
                   d: int, C: int, q, k, v, saved, stream=None, check: bool = True) -> int:
    """C ABI jattn_qkv_norm.  x_img [B, N_img, C] / x_txt [B, N_txt, C] bf16 tokens, w_* [3 H d, C] bf16,
    b_* [3 H d] fp32 or None, gq/gk [d] fp32; writes q/k/v [B, H, N, d] bf16 and `saved`."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e = B * H * N * d
    bf, f32 = torch.bfloat16, torch.float32
    yc = 3 * H * d
    nb = jattn_saved_bytes(B, H, N_img, N_txt, d)
    rc = lib.jattn_qkv_norm(_ptr(x_img, "x_img", bf, B * N_img * C if N_img else None),
                            _ptr(w_img, "w_img", bf, yc * C if N_img else None), _ptr(b_img, "b_img", f32, yc),
                            _ptr(x_txt, "x_txt", bf, B * N_txt * C if N_txt else None),
                            _ptr(w_txt, "w_txt", bf, yc * C if N_txt else None), _ptr(b_txt, "b_txt", f32, yc),
                            _ptr(gq, "gq", f32, d), _ptr(gk, "gk", f32, d), B, H, N_img, N_txt, d, C,
                            _ptr(q, "q", bf, e), _ptr(k, "k", bf, e), _ptr(v, "v", bf, e), _saved_ptr(saved, nb),
                            _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_qkv_norm")
    return rc


def jattn_fwd_saved(v, B: int, H: int, N_img: int, N_txt: int, d: int, out, lse, saved, stream=None,
                    check: bool = True) -> int:
    """C ABI jattn_fwd_saved: the attention forward from the q_hat / k_hat already in `saved`."""
    import torch

    lib = load_library()
    N = N_img + N_txt
    e, r = B * H * N * d, B * H * N
    bf, f32 = torch.bfloat16, torch.float32
    nb = jattn_saved_bytes(B, H, N_img, N_txt, d)
    rc = lib.jattn_fwd_saved(_ptr(v, "v", bf, e), B, H, N_img, N_txt, d, _ptr(out, "out", bf, e),
                             _ptr(lse, "lse", f32, r), _saved_ptr(saved, nb), _stream(stream))
    if check and rc != 0:
        raise JattnError(rc, "jattn_fwd_saved")
    return rc


def jattn_last_device_error(stream=None) -> int:
    return load_library().jattn_last_device_error(_stream(stream))


def jattn_selftest_wait_timeout(stream=None) -> int:
    """Runs the bounded-wait self-test kernel; the next jattn_last_device_error reports the timeout."""
    rc = load_library().jattn_selftest_wait_timeout(_stream(stream))
    if rc != 0:
        raise JattnError(rc, "jattn_selftest_wait_timeout")
    return rc


def jattn_set_sm_limit(max_sms: int) -> int:
    """C ABI jattn_set_sm_limit: cap the persistent kernels' CTAs (0 = every SM)."""
    rc = load_library().jattn_set_sm_limit(int(max_sms))
    if rc != 0:
        raise JattnError(rc, "jattn_set_sm_limit")
    return rc


def jattn_set_deterministic(on: bool) -> int:
    """C ABI jattn_set_deterministic: bitwise-reproducible backward (fixed dQ accumulation order) or not."""
    rc = load_library().jattn_set_deterministic(1 if on else 0)
    if rc != 0:
        raise JattnError(rc, "jattn_set_deterministic")
    return rc


def jattn_status_string(status: int) -> str:
    return load_library().jattn_status_string(int(status)).decode()


def jattn_last_error_message() -> str:
    return load_library().jattn_last_error_message().decode()


def jattn_version() -> int:
    return load_library().jattn_version()
