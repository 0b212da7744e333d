"""The C ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments before touching the GPU (these calls never reach CUDA, so they
run on a machine without one)."""
import ctypes

import pytest

import joint_attention_gb300 as ja
from joint_attention_gb300 import STATUS_CODE
from joint_attention_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return ja.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = ja.declared_symbols()
    assert {"jattn_fwd", "jattn_bwd", "jattn_last_device_error", "jattn_status_string",
            "jattn_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_kernel_names_and_profile_argument_checks(lib):
    names = [ja.jattn_kernel_name(k) for k in range(ja.KERNEL_KINDS)]
    assert names == ["qk_norm_fwd", "attn_fwd", "bwd_prep", "attn_bwd", "q_norm_bwd", "qkv_norm"]
    assert ja.jattn_kernel_name(ja.KERNEL_KINDS) == "unknown"
    import ctypes
    n, ms = ctypes.c_int(0), ctypes.c_double(0)
    assert lib.jattn_profile_read(-1, ctypes.byref(n), ctypes.byref(ms)) == STATUS_CODE["JATTN_ERR_INVALID_ARG"]
    assert lib.jattn_profile_read(0, None, None) == STATUS_CODE["JATTN_ERR_INVALID_ARG"]


def test_version_and_status_strings(lib):
    assert ja.jattn_version() >= 100
    for code in range(7):
        s = ja.jattn_status_string(code)
        assert isinstance(s, str) and s
    assert ja.jattn_status_string(99) == "unknown status"


# Fake, never-dereferenced device addresses: validation happens first.
A = 0x7F0000000000


def fwd(lib, q=A, k=A + 0x1000000, v=A + 0x2000000, gq=A + 0x3000000, gk=A + 0x3001000, B=1, H=2, N_img=16,
        N_txt=8, d=64, out=A + 0x4000000, lse=A + 0x5000000):
    return lib.jattn_fwd(q, k, v, gq, gk, B, H, N_img, N_txt, d, out, lse, None)


def bwd(lib, **kw):
    p = dict(q=A, k=A + 0x1000000, v=A + 0x2000000, gq=A + 0x3000000, gk=A + 0x3001000, out=A + 0x4000000,
             lse=A + 0x5000000, dout=A + 0x6000000, dq=A + 0x7000000, dk=A + 0x8000000, dv=A + 0x9000000,
             dgq=A + 0xA000000, dgk=A + 0xA001000, B=1, H=2, N_img=16, N_txt=8, d=64)
    p.update(kw)
    return lib.jattn_bwd(p["q"], p["k"], p["v"], p["gq"], p["gk"], p["out"], p["lse"], p["dout"], p["dq"], p["dk"],
                         p["dv"], p["dgq"], p["dgk"], p["B"], p["H"], p["N_img"], p["N_txt"], p["d"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), "JATTN_ERR_INVALID_ARG"),
    (dict(lse=None), "JATTN_ERR_INVALID_ARG"),
    (dict(B=0), "JATTN_ERR_INVALID_ARG"),
    (dict(H=-1), "JATTN_ERR_INVALID_ARG"),
    (dict(N_img=-1), "JATTN_ERR_INVALID_ARG"),
    (dict(N_img=0, N_txt=0), "JATTN_ERR_INVALID_ARG"),
    (dict(d=0), "JATTN_ERR_INVALID_ARG"),
    (dict(d=96), "JATTN_ERR_UNSUPPORTED"),
    (dict(d=256), "JATTN_ERR_UNSUPPORTED"),
    (dict(B=65536, H=2), "JATTN_ERR_INVALID_ARG"),
    (dict(B=1000, H=16, N_img=2000, N_txt=77, d=128), "JATTN_ERR_INVALID_ARG"),
    (dict(q=A + 8), "JATTN_ERR_MISALIGNED"),
    (dict(gk=A + 0x3001004), "JATTN_ERR_MISALIGNED"),
    (dict(out=A + 0x1000000), "JATTN_ERR_ALIAS"),           # out == k
    (dict(lse=A + 0x4000000 + 0x100), "JATTN_ERR_ALIAS"),   # lse inside out
    (dict(out=A + 0x3000000 - 0x10), "JATTN_ERR_ALIAS"),    # out runs into gq
])
def test_fwd_validation(lib, kw, expect):
    assert fwd(lib, **kw) == STATUS_CODE[expect]


@pytest.mark.parametrize("kw,expect", [
    (dict(dout=None), "JATTN_ERR_INVALID_ARG"),
    (dict(dgk=None), "JATTN_ERR_INVALID_ARG"),
    (dict(N_txt=-5), "JATTN_ERR_INVALID_ARG"),
    (dict(d=32), "JATTN_ERR_UNSUPPORTED"),
    (dict(dv=A + 0x9000002), "JATTN_ERR_MISALIGNED"),
    (dict(dq=A), "JATTN_ERR_ALIAS"),                        # dq == q
    (dict(dk=A + 0x7000000 + 0x400), "JATTN_ERR_ALIAS"),    # dk inside dq
    (dict(dgq=A + 0xA001000), "JATTN_ERR_ALIAS"),           # dgq == dgk
    (dict(dgq=A + 0x5000000), "JATTN_ERR_ALIAS"),           # dgq == lse
])
def test_bwd_validation(lib, kw, expect):
    assert bwd(lib, **kw) == STATUS_CODE[expect]


def fwd_varlen(lib, cu=(0, 24, 40), H=2, d=64, **kw):
    p = dict(q=A, k=A + 0x1000000, v=A + 0x2000000, gq=A + 0x3000000, gk=A + 0x3001000, out=A + 0x4000000,
             lse=A + 0x5000000)
    p.update(kw)
    arr = (ctypes.c_int * len(cu))(*cu)
    return lib.jattn_fwd_varlen(p["q"], p["k"], p["v"], p["gq"], p["gk"], arr, len(cu) - 1, H, d, p["out"],
                                p["lse"], None)


def bwd_varlen(lib, cu=(0, 24, 40), H=2, d=64, **kw):
    p = dict(q=A, k=A + 0x1000000, v=A + 0x2000000, gq=A + 0x3000000, gk=A + 0x3001000, out=A + 0x4000000,
             lse=A + 0x5000000, dout=A + 0x6000000, dq=A + 0x7000000, dk=A + 0x8000000, dv=A + 0x9000000,
             dgq=A + 0xA000000, dgk=A + 0xA001000)
    p.update(kw)
    arr = (ctypes.c_int * len(cu))(*cu)
    return lib.jattn_bwd_varlen(p["q"], p["k"], p["v"], p["gq"], p["gk"], p["out"], p["lse"], p["dout"], p["dq"],
                                p["dk"], p["dv"], p["dgq"], p["dgk"], arr, len(cu) - 1, H, d, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), "JATTN_ERR_INVALID_ARG"),
    (dict(cu=(0,)), "JATTN_ERR_INVALID_ARG"),                # no sequence
    (dict(cu=(1, 24)), "JATTN_ERR_INVALID_ARG"),             # does not start at 0
    (dict(cu=(0, 24, 24, 40)), "JATTN_ERR_INVALID_ARG"),     # an empty sequence
    (dict(cu=(0, 30, 20)), "JATTN_ERR_INVALID_ARG"),         # decreasing
    (dict(cu=tuple(range(258))), "JATTN_ERR_UNSUPPORTED"),   # 257 sequences
    (dict(H=0), "JATTN_ERR_INVALID_ARG"),
    (dict(d=96), "JATTN_ERR_UNSUPPORTED"),
    (dict(cu=(0, 1 << 30), H=4), "JATTN_ERR_INVALID_ARG"),   # H*T*d overflows
    (dict(v=A + 0x2000004), "JATTN_ERR_MISALIGNED"),
    (dict(out=A + 0x1000000), "JATTN_ERR_ALIAS"),            # out == k
])
def test_fwd_varlen_validation(lib, kw, expect):
    assert fwd_varlen(lib, **kw) == STATUS_CODE[expect]


@pytest.mark.parametrize("kw,expect", [
    (dict(dout=None), "JATTN_ERR_INVALID_ARG"),
    (dict(cu=(0, 5, 3)), "JATTN_ERR_INVALID_ARG"),
    (dict(d=32), "JATTN_ERR_UNSUPPORTED"),
    (dict(dq=A), "JATTN_ERR_ALIAS"),                         # dq == q
])
def test_bwd_varlen_validation(lib, kw, expect):
    assert bwd_varlen(lib, **kw) == STATUS_CODE[expect]


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(FileNotFoundError):
        ja.load_library(str(tmp_path / "missing.so"))


def test_mode_switches_validate_and_apply_to_later_calls(lib):
    # The CTA cap and the deterministic-backward switch take effect on later
    # calls; only a negative cap is rejected.  Nothing runs on a device here.
    assert ja.jattn_set_sm_limit(0) == 0
    assert ja.jattn_set_sm_limit(7) == 0
    assert ja.jattn_set_sm_limit(0) == 0
    assert lib.jattn_set_sm_limit(-1) == ja.STATUS_CODE["JATTN_ERR_INVALID_ARG"]
    assert ja.jattn_set_deterministic(True) == 0
    assert ja.jattn_set_deterministic(False) == 0


def test_training_pair_sizes_and_validation(lib):
    """jattn_saved_bytes covers q_hat, k_hat and two fp32 values per row (0
    for a shape the calls reject), and the training pair validates like
    jattn_fwd / jattn_bwd plus its `saved` argument, before any CUDA call."""
    B, H, N_img, N_txt, d = 1, 2, 16, 8, 64
    rows, elems = B * H * (N_img + N_txt), B * H * (N_img + N_txt) * d
    nb = ja.jattn_saved_bytes(B, H, N_img, N_txt, d)
    assert nb >= 2 * elems * 2 + 2 * rows * 4 and nb % 256 == 0
    assert ja.jattn_saved_bytes(B, H, N_img, N_txt, 96) == 0
    assert ja.jattn_saved_bytes(0, H, N_img, N_txt, d) == 0
    assert ja.jattn_saved_bytes_varlen([0, 24, 40], 2, 64) >= 2 * 2 * 40 * 64 * 2
    assert ja.jattn_saved_bytes_varlen([0, 24, 24], 2, 64) == 0
    S = A + 0xB000000
    f = lambda **kw: lib.jattn_fwd_train(*[kw.get(n, v) for n, v in (  # noqa: E731
        ("q", A), ("k", A + 0x1000000), ("v", A + 0x2000000), ("gq", A + 0x3000000), ("gk", A + 0x3001000),
        ("B", B), ("H", H), ("N_img", N_img), ("N_txt", N_txt), ("d", d), ("out", A + 0x4000000),
        ("lse", A + 0x5000000), ("saved", S))], None)
    assert f(saved=None) == STATUS_CODE["JATTN_ERR_INVALID_ARG"]
    assert f(saved=S + 8) == STATUS_CODE["JATTN_ERR_MISALIGNED"]
    assert f(saved=A + 0x4000000) == STATUS_CODE["JATTN_ERR_ALIAS"]       # saved == out
    assert f(saved=A + 0x2000000 - 0x100) == STATUS_CODE["JATTN_ERR_ALIAS"]  # saved runs into v
    assert f(d=32) == STATUS_CODE["JATTN_ERR_UNSUPPORTED"]
    g = lambda **kw: lib.jattn_bwd_train(*[kw.get(n, v) for n, v in (  # noqa: E731
        ("q", A), ("k", A + 0x1000000), ("v", A + 0x2000000), ("gq", A + 0x3000000), ("gk", A + 0x3001000),
        ("out", A + 0x4000000), ("lse", A + 0x5000000), ("dout", A + 0x6000000), ("saved", S),
        ("dq", A + 0x7000000), ("dk", A + 0x8000000), ("dv", A + 0x9000000), ("dgq", A + 0xA000000),
        ("dgk", A + 0xA001000), ("B", B), ("H", H), ("N_img", N_img), ("N_txt", N_txt), ("d", d))], None)
    assert g(saved=None) == STATUS_CODE["JATTN_ERR_INVALID_ARG"]
    assert g(saved=A + 0x7000000) == STATUS_CODE["JATTN_ERR_ALIAS"]       # saved == dq
    assert g(dq=None) == STATUS_CODE["JATTN_ERR_INVALID_ARG"]


def test_qkv_norm_and_fwd_saved_validation(lib):
    """jattn_qkv_norm / jattn_fwd_saved refuse bad arguments before any CUDA call."""
    B, H, N_img, N_txt, d, C = 2, 3, 40, 8, 64, 96
    S = A + 0xB000000
    f = lambda **kw: lib.jattn_qkv_norm(*[kw.get(n, v) for n, v in (  # noqa: E731
        ("x_img", A), ("w_img", A + 0x1000000), ("b_img", None), ("x_txt", A + 0x2000000),
        ("w_txt", A + 0x3000000), ("b_txt", A + 0x3100000), ("gq", A + 0x3200000), ("gk", A + 0x3201000),
        ("B", B), ("H", H), ("N_img", N_img), ("N_txt", N_txt), ("d", d), ("C", C), ("q", A + 0x4000000),
        ("k", A + 0x5000000), ("v", A + 0x6000000), ("saved", S))], None)
    code = STATUS_CODE
    assert f(saved=None) == code["JATTN_ERR_INVALID_ARG"]
    assert f(q=None) == code["JATTN_ERR_INVALID_ARG"]
    assert f(x_img=None) == code["JATTN_ERR_INVALID_ARG"]          # image rows need tokens
    assert f(w_txt=None) == code["JATTN_ERR_INVALID_ARG"]          # caption rows need a weight
    assert f(B=0) == code["JATTN_ERR_INVALID_ARG"]
    assert f(C=0) == code["JATTN_ERR_INVALID_ARG"]
    assert f(C=100) == code["JATTN_ERR_UNSUPPORTED"]               # row stride not a multiple of 16 bytes
    assert f(d=32) == code["JATTN_ERR_UNSUPPORTED"]
    assert f(C=1 << 24, H=64) == code["JATTN_ERR_INVALID_ARG"]     # 3 H d C beyond 2^31
    assert f(x_img=A + 2) == code["JATTN_ERR_MISALIGNED"]
    assert f(b_img=A + 0x3300008) == code["JATTN_ERR_MISALIGNED"]
    assert f(q=A + 0x5000000) == code["JATTN_ERR_ALIAS"]           # q == k
    assert f(saved=A + 0x1000000) == code["JATTN_ERR_ALIAS"]       # saved over w_img
    assert f(v=A + 0x3200000 - 0x100) == code["JATTN_ERR_ALIAS"]   # v runs into gq
    # A stream without rows needs no tokens or weight.
    assert f(N_txt=0, x_txt=None, w_txt=None, b_txt=None, d=32) == code["JATTN_ERR_UNSUPPORTED"]
    g = lambda **kw: lib.jattn_fwd_saved(*[kw.get(n, v) for n, v in (  # noqa: E731
        ("v", A), ("B", B), ("H", H), ("N_img", N_img), ("N_txt", N_txt), ("d", d), ("out", A + 0x1000000),
        ("lse", A + 0x2000000), ("saved", S))], None)
    assert g(saved=None) == code["JATTN_ERR_INVALID_ARG"]
    assert g(d=96) == code["JATTN_ERR_UNSUPPORTED"]
    assert g(out=A + 0x1000004) == code["JATTN_ERR_MISALIGNED"]
    assert g(out=S) == code["JATTN_ERR_ALIAS"]
    assert g(lse=A + 0x10) == code["JATTN_ERR_ALIAS"]
