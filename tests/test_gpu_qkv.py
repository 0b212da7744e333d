"""GPU parity of the fused QKV projection + QK-RMSNorm call (jattn_qkv_norm)
against the CPU oracle, and of the chain it feeds (jattn_fwd_saved,
jattn_bwd_train) against the plain calls.

Tolerances, from the arithmetic:
* q, k, v: the kernel accumulates X W^T in fp32 on the tensor cores, adds the
  fp32 bias and rounds once to bf16; the oracle rounds the exact value once.
  Every element must equal the oracle's, or be a bf16 value whose rounding
  interval reaches the fp32 result's error interval: |got - exact| <=
  C 2^-23 (sum_c |x_c w_c| + |b|) + half a bf16 step at got (each of the C
  additions off by at most one fp32 ulp of the running magnitude, and the
  bias addition).  Such elements are rare (rounding ties, and values that
  cancel to far below their terms): at most 1e-3 of them.
* q_hat, k_hat: correctly rounded, so bit-exact on every row whose raw q / k
  equals the oracle's; 1/rms within 2^-21 relative there (rsqrtf and an
  fp32 sum of squares).
* The saved buffer it writes must drive the attention exactly as the one
  jattn_fwd_train writes from the same q, k, v: q_hat / k_hat bit for bit,
  so jattn_fwd_saved's out / lse equal jattn_fwd's bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from joint_attention_gb300.inputs import make_qkv_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ja():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from joint_attention_gb300.build import build

    build()
    import joint_attention_gb300 as pkg

    pkg.load_library()
    return pkg


def dev_bf16(a):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(torch.bfloat16).contiguous()


def dev_f32(a):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().contiguous()


def np64(t):
    return t.float().cpu().numpy().astype(np.float64)


def saved_parts(saved, B, H, N, d):
    """Views of the training pair's buffer (the library's private layout: q_hat,
    k_hat, then 1/rms of the q rows and of the k rows, each part at a 256-byte
    aligned offset)."""
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    elems, rows = B * H * N * d, B * H * N
    o_k = up(elems * 2)
    o_rq = o_k + up(elems * 2)
    o_rk = o_rq + up(rows * 4)
    qh = saved[0:elems * 2].view(torch.bfloat16).view(B, H, N, d)
    kh = saved[o_k:o_k + elems * 2].view(torch.bfloat16).view(B, H, N, d)
    rq = saved[o_rq:o_rq + rows * 4].view(torch.float32).view(B, H, N)
    rk = saved[o_rk:o_rk + rows * 4].view(torch.float32).view(B, H, N)
    return qh, kh, rq, rk


def bf16_bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.int64)


def check_projection(got, exact, absprod, C, where):
    """got: the kernel's bf16 values; exact: the oracle's unrounded float64;
    absprod: sum_c |x_c w_c| + |b| per element."""
    want = oracle.round_to_bf16(exact)
    bad = got != want
    if bad.any():
        g, e, a = got[bad], exact[bad], absprod[bad]
        # got's rounding interval must reach the fp32 result's error interval
        half_step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(g), 2.0 ** -126))) - 8)
        slack = np.abs(g - e) - (C * 2.0 ** -23 * a + half_step)
        assert np.all(slack <= 0), (where, "beyond the fp32 accumulation bound", g[slack > 0][:4], e[slack > 0][:4])
    assert bad.mean() <= 1e-3, (where, "mismatch fraction", bad.mean())
    return bad


def run_qkv(ja, inp, B, H, N_img, N_txt, d, C):
    x_img, w_img, b_img = dev_bf16(inp.x_img), dev_bf16(inp.w_img), dev_f32(inp.b_img)
    x_txt, w_txt, b_txt = dev_bf16(inp.x_txt), dev_bf16(inp.w_txt), dev_f32(inp.b_txt)
    gq, gk = dev_f32(inp.gq), dev_f32(inp.gk)
    N = N_img + N_txt
    q = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    k, v = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
    saved = torch.full((ja.jattn_saved_bytes(B, H, N_img, N_txt, d),), 0xFF, dtype=torch.uint8, device="cuda")
    ja.jattn_qkv_norm(x_img if N_img else None, w_img if N_img else None, b_img if N_img else None,
                      x_txt if N_txt else None, w_txt if N_txt else None, b_txt if N_txt else None, gq, gk, B, H,
                      N_img, N_txt, d, C, q, k, v, saved)
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0
    return q, k, v, saved, gq, gk


CASES = [
    # B, H, N_img, N_txt, d, C, bias
    (2, 4, 200, 77, 64, 256, True),     # ragged row tails in both streams; 3 column tiles
    (1, 3, 130, 5, 64, 200, False),     # partial column tile (9 heads of 64) and a partial K step
    (2, 2, 96, 0, 128, 128, True),      # no caption stream, d = 128
    (1, 4, 0, 40, 128, 64, True),       # caption stream only
    (1, 1, 1, 1, 64, 8, True),          # one token per stream, the narrowest width
    (3, 12, 256, 77, 64, 768, True),    # the 768-wide model (12 heads of 64)
]


@pytest.mark.parametrize("B,H,N_img,N_txt,d,C,bias", CASES)
def test_qkv_norm_matches_oracle(ja, B, H, N_img, N_txt, d, C, bias):
    inp = make_qkv_inputs(B, H, N_img, N_txt, d, C, seed=2000 + N_img + C + d, bias=bias)
    q, k, v, saved, _, _ = run_qkv(ja, inp, B, H, N_img, N_txt, d, C)
    ref = oracle.qkv_norm_streams(inp.x_img, inp.w_img, inp.b_img, inp.x_txt, inp.w_txt, inp.b_txt, inp.gq,
                                  inp.gk, H)
    ab = lambda a: None if a is None else np.abs(a)  # noqa: E731
    absprod = oracle.qkv_norm_streams(np.abs(inp.x_img), np.abs(inp.w_img), ab(inp.b_img), np.abs(inp.x_txt),
                                      np.abs(inp.w_txt), ab(inp.b_txt), inp.gq, inp.gk, H)["y_exact"]
    N = N_img + N_txt
    bad = [check_projection(np64(t), ref["y_exact"][i], absprod[i], C, f"{'qkv'[i]} {B, H, N_img, N_txt, d, C}")
           for i, t in enumerate((q, k, v))]
    qh, kh, rq, rk = saved_parts(saved, B, H, N, d)
    for name, got_h, got_r, want_h, want_r, b in (("q", qh, rq, ref["qhat"], ref["rq"], bad[0]),
                                                 ("k", kh, rk, ref["khat"], ref["rk"], bad[1])):
        same = ~b.any(axis=-1)  # rows whose raw values equal the oracle's
        gh, gr = np64(got_h), np64(got_r)
        np.testing.assert_array_equal(gh[same], want_h[same], err_msg=f"{name}_hat")
        rel = np.abs(gr[same] - want_r[same]) / want_r[same]
        assert rel.max(initial=0.0) <= 2.0 ** -21, (name, "1/rms", rel.max())
        # The other rows: the norm of a row that is off by one bf16 ulp somewhere.
        if (~same).any():
            assert np.max(np.abs(gh[~same] - want_h[~same])) <= 2.0 ** -6 * np.max(np.abs(want_h[~same])) + 1e-30


@pytest.mark.parametrize("d", [64, 128])
def test_qkv_norm_rounds_at_bf16_midpoints(ja, d):
    """Unit-vector tokens make each projected row one weight column (no
    accumulation error).  Columns of +-8 give rows of equal values, and gains
    on bf16 midpoints (1 + 3 2^-8) put g x r a relative 8e-9 below a midpoint,
    where fp32 arithmetic lands on the midpoint itself.  q_hat / k_hat must
    still be the bf16 value nearest the exact product, as in the oracle; the
    random columns beside them take the common path."""
    B, H, N_img, N_txt, C = 2, 2, 150, 21, 64
    inp = make_qkv_inputs(B, H, N_img, N_txt, d, C, seed=2400 + d, bias=False)
    rng = np.random.default_rng(d)
    for x, w in ((inp.x_img, inp.w_img), (inp.x_txt, inp.w_txt)):
        cols = rng.integers(0, C, x.shape[:2])
        x[...] = 0.0
        np.put_along_axis(x, cols[..., None], 1.0, axis=2)
        w[: 2 * H * d, ::3] = 8.0      # q and k rows of every third column: all 8
        w[: 2 * H * d, 1::6] = -8.0
    inp.gq[::2] = 1.0 + 3 * 2.0 ** -8
    inp.gk[1::2] = 1.0 + 3 * 2.0 ** -8
    q, k, v, saved, _, _ = run_qkv(ja, inp, B, H, N_img, N_txt, d, C)
    ref = oracle.qkv_norm_streams(inp.x_img, inp.w_img, None, inp.x_txt, inp.w_txt, None, inp.gq, inp.gk, H)
    N = N_img + N_txt
    for i, t in enumerate((q, k, v)):
        np.testing.assert_array_equal(np64(t), ref["qkv"[i]])
    qh, kh, rq, rk = saved_parts(saved, B, H, N, d)
    np.testing.assert_array_equal(np64(qh), ref["qhat"])
    np.testing.assert_array_equal(np64(kh), ref["khat"])
    # The constant rows are there, and on them the fp32 path alone would round the other way.
    const_rows = np.all(np.abs(ref["q"]) == 8.0, axis=-1)
    assert const_rows.sum() >= 20


@pytest.mark.parametrize("d", [64, 128])
def test_projected_chain_matches_the_plain_training_pair(ja, d):
    """q, k, v from the projection fed to jattn_fwd_train give the same q_hat /
    k_hat as the projection's own saved buffer (bit for bit) and 1/rms to fp32
    rounding; jattn_fwd_saved then equals jattn_fwd bit for bit, and the
    backward from either saved buffer agrees (deterministic mode)."""
    B, H, N_img, N_txt, C = 2, 4, 333, 77, 256
    inp = make_qkv_inputs(B, H, N_img, N_txt, d, C, seed=2100 + d)
    q, k, v, saved, gq, gk = run_qkv(ja, inp, B, H, N_img, N_txt, d, C)
    N = N_img + N_txt
    out0, lse0, saved0 = ja.forward_train(q, k, v, gq, gk, N_txt)
    out1, lse1 = torch.empty_like(out0), torch.empty_like(lse0)
    ja.jattn_fwd_saved(v, B, H, N_img, N_txt, d, out1, lse1, saved)
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0
    p0, p1 = saved_parts(saved0, B, H, N, d), saved_parts(saved, B, H, N, d)
    assert torch.equal(p0[0].view(torch.int16), p1[0].view(torch.int16))
    assert torch.equal(p0[1].view(torch.int16), p1[1].view(torch.int16))
    for a, b in ((p0[2], p1[2]), (p0[3], p1[3])):
        rel = ((a - b).abs() / a.abs()).max().item()
        assert rel <= 2.0 ** -21, rel
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(lse0.view(torch.int32), lse1.view(torch.int32))
    g = torch.Generator(device="cuda").manual_seed(7)
    dout = torch.randn(out0.shape, generator=g, device="cuda").to(torch.bfloat16)
    ja.jattn_set_deterministic(True)
    try:
        g0 = ja.backward_train(q, k, v, gq, gk, out0, lse0, dout, saved0, N_txt)
        g1 = ja.backward_train(q, k, v, gq, gk, out1, lse1, dout, saved, N_txt)
        torch.cuda.synchronize()
        assert ja.jattn_last_device_error() == 0
    finally:
        ja.jattn_set_deterministic(False)
    # dv reads no 1/rms.  The others see 1/rms values up to 2^-21 apart: a bf16
    # output then flips to its neighbour (one step, 2^-8 relative) with a chance
    # of about 2^-21 / 2^-8 = 2^-13, a relative Frobenius difference near
    # sqrt(2^-13) 2^-8 = 4e-5; the fp32 gain gradients move far less.
    assert torch.equal(g0[2].view(torch.int16), g1[2].view(torch.int16))
    for name, a, b in zip(("dq", "dk", "dv", "dgq", "dgk"), g0, g1):
        a64, b64 = np64(a), np64(b)
        rel = np.linalg.norm(a64 - b64) / max(np.linalg.norm(a64), 1e-30)
        assert rel <= 2e-4, (name, rel)


def test_full_size_512px_sampled_rows(ja):
    """The 512 px workload (B 16, 1024 image + 77 caption tokens, 12 heads of
    64, width 768) in the launch the benchmark times, compared on sampled
    token rows of both streams."""
    B, H, N_img, N_txt, d, C = 16, 12, 1024, 77, 64, 768
    inp = make_qkv_inputs(B, H, N_img, N_txt, d, C, seed=2200)
    q, k, v, saved, _, _ = run_qkv(ja, inp, B, H, N_img, N_txt, d, C)
    N = N_img + N_txt
    qh, kh, rq, rk = saved_parts(saved, B, H, N, d)
    rng = np.random.default_rng(5)
    for stream, x, w, bias, n_s, row0 in (("img", inp.x_img, inp.w_img, inp.b_img, N_img, N_txt),
                                          ("txt", inp.x_txt, inp.w_txt, inp.b_txt, N_txt, 0)):
        bi = rng.integers(0, B, 96)
        ni = rng.integers(0, n_s, 96)
        ni[:2] = (0, n_s - 1)
        xs = x[bi, ni][None]  # [1, S, C]
        exact, _ = oracle.qkv_projection(xs, w, bias, H)
        absprod, _ = oracle.qkv_projection(np.abs(xs), np.abs(w), np.abs(bias), H)
        rows = row0 + ni
        got = [np64(t[torch.from_numpy(bi).cuda(), :, torch.from_numpy(rows).cuda(), :]) for t in (q, k, v)]
        # got[i]: [S, H, d]; exact[i]: [1, H, S, d]
        for i in range(3):
            e = exact[i][0].transpose(1, 0, 2)
            a = absprod[i][0].transpose(1, 0, 2)
            bad = check_projection(got[i], e, a, C, f"{stream} {'qkv'[i]}")
            if i < 2:
                hat = np64((qh, kh)[i][torch.from_numpy(bi).cuda(), :, torch.from_numpy(rows).cuda(), :])
                r = np64((rq, rk)[i][torch.from_numpy(bi).cuda(), :, torch.from_numpy(rows).cuda()])
                g = (inp.gq, inp.gk)[i]
                want_hat, want_r = oracle.rmsnorm_fwd(oracle.round_to_bf16(e), g)
                same = ~bad.any(axis=-1)
                np.testing.assert_array_equal(hat[same], oracle.round_to_bf16(want_hat)[same])
                assert np.max(np.abs(r[same] - want_r[..., 0][same]) / want_r[..., 0][same]) <= 2.0 ** -21


def test_qkv_norm_argument_checks(ja):
    B, H, N_img, N_txt, d, C = 1, 2, 40, 8, 64, 64
    inp = make_qkv_inputs(B, H, N_img, N_txt, d, C, seed=2300)
    x_img, w_img, x_txt, w_txt = dev_bf16(inp.x_img), dev_bf16(inp.w_img), dev_bf16(inp.x_txt), dev_bf16(inp.w_txt)
    gq, gk = dev_f32(inp.gq), dev_f32(inp.gk)
    N = N_img + N_txt
    q = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k, v = torch.empty_like(q), torch.empty_like(q)
    saved = torch.empty(ja.jattn_saved_bytes(B, H, N_img, N_txt, d), dtype=torch.uint8, device="cuda")
    code = ja.STATUS_CODE
    lib = ja.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    call = lambda **kw: lib.jattn_qkv_norm(*[kw.get(n, val) for n, val in (  # noqa: E731
        ("x_img", P(x_img)), ("w_img", P(w_img)), ("b_img", None), ("x_txt", P(x_txt)), ("w_txt", P(w_txt)),
        ("b_txt", None), ("gq", P(gq)), ("gk", P(gk)), ("B", B), ("H", H), ("N_img", N_img), ("N_txt", N_txt),
        ("d", d), ("C", C), ("q", P(q)), ("k", P(k)), ("v", P(v)), ("saved", P(saved)))], stream)
    assert call(saved=0) == code["JATTN_ERR_INVALID_ARG"]
    assert call(w_txt=0) == code["JATTN_ERR_INVALID_ARG"]
    assert call(d=96) == code["JATTN_ERR_UNSUPPORTED"]
    assert call(C=60) == code["JATTN_ERR_UNSUPPORTED"]
    assert call(C=0) == code["JATTN_ERR_INVALID_ARG"]
    assert call(q=P(k)) == code["JATTN_ERR_ALIAS"]
    assert call(v=P(x_img)) == code["JATTN_ERR_ALIAS"]
    assert call(saved=P(saved) + 8) == code["JATTN_ERR_MISALIGNED"]
    assert call(b_img=P(gq) + 4) == code["JATTN_ERR_MISALIGNED"]
    assert call() == 0
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0
