"""Property test of the boundary's argument validation.

Each example draws a valid problem, gives every buffer its own fake,
never-dereferenced, 16-byte aligned address (8 GiB apart, more than any
buffer), and then injects exactly one fault: a null pointer, a misaligned
pointer, an output overlapping another buffer, or a bad size.  The call must
return the status the header documents for that fault.  A call without a
fault is never made (it would launch work on the fake addresses).
"""
import ctypes

import pytest

from joint_attention_gb300 import STATUS_CODE
import joint_attention_gb300 as ja
from joint_attention_gb300.build import build

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings, strategies as st  # noqa: E402

BASE, SPACING = 1 << 44, 1 << 33
MAX_SEQS = 256  # JATTN_MAX_SEQS
FWD_IN, FWD_OUT = ("q", "k", "v", "gq", "gk"), ("out", "lse")
BWD_IN = ("q", "k", "v", "gq", "gk", "out", "lse", "dout")
BWD_OUT = ("dq", "dk", "dv", "dgq", "dgk")


@pytest.fixture(scope="module")
def lib():
    build()
    return ja.load_library()


@st.composite
def problems(draw):
    d = draw(st.sampled_from([64, 128]))
    H = draw(st.integers(1, 48))
    B = draw(st.integers(1, 64))
    n_txt = draw(st.integers(0, 300))
    n_img = draw(st.integers(0 if n_txt else 1, 4096))
    if B * H * (n_img + n_txt) * d >= 1 << 31:
        B = 1
    return dict(B=B, H=H, N_img=n_img, N_txt=n_txt, d=d)


def sizes(p):
    """Bytes of each buffer of the problem."""
    e = p["B"] * p["H"] * (p["N_img"] + p["N_txt"])
    bf, rows, gain = e * p["d"] * 2, e * 4, p["d"] * 4
    return dict(q=bf, k=bf, v=bf, out=bf, dout=bf, dq=bf, dk=bf, dv=bf, lse=rows, gq=gain, gk=gain, dgq=gain,
                dgk=gain)


@st.composite
def faults(draw, ins, outs):
    names = ins + outs
    kind = draw(st.sampled_from(["null", "misalign", "alias", "shape"]))
    if kind == "null":
        return ("null", draw(st.sampled_from(names)))
    if kind == "misalign":
        return ("misalign", draw(st.sampled_from(names)), draw(st.sampled_from([1, 2, 4, 8, 12])))
    if kind == "alias":
        o = draw(st.sampled_from(outs))
        other = draw(st.sampled_from([n for n in names if n != o]))
        return ("alias", o, other, draw(st.floats(0.0, 0.999)))
    return ("shape", draw(st.sampled_from(["B0", "H0", "Nneg", "N0", "d", "heads", "elems"])))


def apply(p, fault, ins, outs):
    """Pointers and sizes with the fault in, and the status it must give."""
    ptr = {n: BASE + i * SPACING for i, n in enumerate(ins + outs)}
    p = dict(p)
    kind = fault[0]
    if kind == "null":
        ptr[fault[1]] = None
        return ptr, p, "JATTN_ERR_INVALID_ARG"
    if kind == "misalign":
        ptr[fault[1]] += fault[2]
        return ptr, p, "JATTN_ERR_MISALIGNED"
    if kind == "alias":
        _, o, other, frac = fault
        size = sizes(p)[other]
        ptr[o] = ptr[other] + (int(frac * size) // 16) * 16  # starts inside `other`
        return ptr, p, "JATTN_ERR_ALIAS"
    what = fault[1]
    if what == "B0":
        p["B"] = 0
    elif what == "H0":
        p["H"] = -p["H"]
    elif what == "Nneg":
        p["N_txt"] = -1 - p["N_txt"]
    elif what == "N0":
        p["N_img"], p["N_txt"] = 0, 0
    elif what == "d":
        p["d"] = {64: 96, 128: 32}[p["d"]]
        return ptr, p, "JATTN_ERR_UNSUPPORTED"
    elif what == "heads":
        p["B"], p["N_img"], p["N_txt"] = 65536 // p["H"] + 1, 1, 0
    else:  # elements >= 2^31
        p["B"], p["H"] = 1024, 48
        p["N_img"] = max(p["N_img"], (1 << 31) // (1024 * 48 * p["d"]) + 1)
    return ptr, p, "JATTN_ERR_INVALID_ARG"


SETTINGS = settings(max_examples=400, deadline=None, suppress_health_check=[HealthCheck.function_scoped_fixture])


@SETTINGS
@given(p=problems(), fault=faults(FWD_IN, FWD_OUT))
def test_fwd_rejects_every_single_fault(lib, p, fault):
    ptr, q, expect = apply(p, fault, FWD_IN, FWD_OUT)
    args = [ptr[n] for n in FWD_IN] + [q["B"], q["H"], q["N_img"], q["N_txt"], q["d"], ptr["out"], ptr["lse"], None]
    rc = lib.jattn_fwd(*args)
    assert rc == STATUS_CODE[expect], (fault, q, rc)
    rc = lib.jattn_fwd_noalloc(*args)
    assert rc == STATUS_CODE[expect], ("noalloc", fault, q, rc)


@SETTINGS
@given(p=problems(), fault=faults(BWD_IN, BWD_OUT))
def test_bwd_rejects_every_single_fault(lib, p, fault):
    ptr, q, expect = apply(p, fault, BWD_IN, BWD_OUT)
    args = [ptr[n] for n in BWD_IN + BWD_OUT] + [q["B"], q["H"], q["N_img"], q["N_txt"], q["d"], None]
    rc = lib.jattn_bwd(*args)
    assert rc == STATUS_CODE[expect], (fault, q, rc)


@SETTINGS
@given(lens=st.lists(st.integers(1, 3000), min_size=1, max_size=256), H=st.integers(1, 16),
       d=st.sampled_from([64, 128]), fault=st.sampled_from(["start", "empty", "decrease", "count", "null"]))
def test_varlen_rejects_bad_sequence_tables(lib, lens, H, d, fault):
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    n = len(lens)
    ptr = {name: BASE + i * SPACING for i, name in enumerate(FWD_IN + FWD_OUT)}
    if fault == "start":
        cu[0] = 1
        expect = "JATTN_ERR_INVALID_ARG"
    elif fault == "empty":
        i = len(cu) // 2
        cu[i] = cu[i - 1]
        expect = "JATTN_ERR_INVALID_ARG"
    elif fault == "decrease":
        if n < 2:
            cu.append(cu[-1] - 1)
            n += 1
        else:
            cu[1], cu[2] = cu[2], cu[1]
        expect = "JATTN_ERR_INVALID_ARG"
    elif fault == "count":
        while len(cu) <= MAX_SEQS + 1:  # one sequence more than the header allows
            cu.append(cu[-1] + 1)
        n = len(cu) - 1
        expect = "JATTN_ERR_UNSUPPORTED"
    else:
        ptr["q"] = None
        expect = "JATTN_ERR_INVALID_ARG"
    arr = (ctypes.c_int * len(cu))(*cu)
    rc = lib.jattn_fwd_varlen(ptr["q"], ptr["k"], ptr["v"], ptr["gq"], ptr["gk"], arr, n, H, d, ptr["out"],
                              ptr["lse"], None)
    assert rc == STATUS_CODE[expect], (fault, cu[:4], n, rc)

