"""GPU invariants of joint attention with QK-RMSNorm, checked on libjattn's
own outputs (through the C ABI), independent of the oracle's values.

Each test states what the mathematics fixes and the slack the bf16 inputs and
outputs leave:
  * head / batch independence: every (b, h) is computed from its own rows only;
  * exact scaling: doubling v doubles O, doubling dout doubles dq, dk, dv, dgq,
    dgk (multiplying by 2 is exact in bf16 and in the fp32 accumulations);
  * RMSNorm scale invariance: q -> 2q leaves q_hat unchanged up to eps;
  * the RMSNorm backward makes every dq row orthogonal to its q row;
  * softmax rows sum to one, so the key-sum of dv equals the query-sum of dout.
"""
import numpy as np
import pytest
import torch

from joint_attention_gb300.inputs import make_inputs

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
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(torch.bfloat16).contiguous()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().contiguous()


def run(ja, q, k, v, gq, gk, dout, n_txt):
    tq, tk, tv, tgq, tgk = dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_f32(gq), dev_f32(gk)
    out, lse = ja.forward(tq, tk, tv, tgq, tgk, n_txt)
    dq, dk, dv, dgq, dgk = ja.backward(tq, tk, tv, tgq, tgk, out, lse, dev_bf16(dout), n_txt)
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0
    return {name: t.float().cpu().numpy().astype(np.float64)
            for name, t in dict(O=out, LSE=lse, dq=dq, dk=dk, dv=dv, dgq=dgq, dgk=dgk).items()}


def relF(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


@pytest.mark.parametrize("d", [64, 128])
def test_heads_and_batch_items_are_independent(ja, d):
    """A (b, h) slice run alone gives the same O, LSE, dk and dv bit for bit
    (both kernels walk one head's tiles in a fixed order); dq, accumulated by
    fp32 reduce-adds in arrival order, agrees to rounding."""
    B, H, N, n_txt = 2, 3, 333, 77
    inp = make_inputs(B, H, N, d, seed=31)
    full = run(ja, inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    b, h = 1, 2
    sl = (slice(b, b + 1), slice(h, h + 1))
    one = run(ja, inp.q[sl], inp.k[sl], inp.v[sl], inp.gq, inp.gk, inp.dout[sl], n_txt)
    for name in ("O", "LSE", "dk", "dv"):
        assert np.array_equal(one[name][0, 0], full[name][b, h]), name
    assert relF(one["dq"][0, 0], full["dq"][b, h]) < 1e-2


def test_doubling_v_and_dout_is_exact(ja):
    """O(2v) = 2 O(v) and every gradient scales by 2 with dout -> 2 dout, bit
    for bit: the power-of-two factor passes exactly through bf16 rounding and
    the fp32 accumulations."""
    B, H, N, d, n_txt = 1, 2, 300, 64, 44
    inp = make_inputs(B, H, N, d, seed=32)
    base = run(ja, inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    v2 = run(ja, inp.q, inp.k, 2.0 * inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    assert np.array_equal(v2["O"], 2.0 * base["O"])
    assert np.array_equal(v2["LSE"], base["LSE"])
    g2 = run(ja, inp.q, inp.k, inp.v, inp.gq, inp.gk, 2.0 * inp.dout, n_txt)
    for name in ("dk", "dv", "dgk"):
        assert np.array_equal(g2[name], 2.0 * base[name]), name
    # dq and dgq pass through the fp32 accumulator, whose reduce-adds land in
    # arrival order: equal to rounding.
    for name in ("dq", "dgq"):
        assert relF(g2[name], 2.0 * base[name]) < 1e-3, name


def test_rmsnorm_scale_invariance(ja):
    """q -> 2q and k -> 2k leave q_hat, k_hat unchanged up to eps = 1e-6 (far
    below bf16 resolution), so O and LSE are unchanged; dq and dk halve."""
    B, H, N, d, n_txt = 1, 2, 257, 64, 1
    inp = make_inputs(B, H, N, d, seed=33)
    base = run(ja, inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    sc = run(ja, 2.0 * inp.q, 2.0 * inp.k, inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    assert float(np.max(np.abs(sc["O"] - base["O"]))) <= 1e-2
    assert float(np.max(np.abs(sc["LSE"] - base["LSE"]))) <= 1e-3
    for name in ("dq", "dk"):
        assert relF(2.0 * sc[name], base[name]) < 2e-2, name
    for name in ("dv", "dgq", "dgk"):
        assert relF(sc[name], base[name]) < 2e-2, name


def test_dq_rows_orthogonal_to_q_rows(ja):
    """dq = r u - (r^3/d) q (u . q) gives q . dq = r (u . q)(1 - r^2 |q|^2 / d),
    which vanishes up to eps; the bf16 output and the kernel's rounding bound
    the measured cosine."""
    B, H, N, d, n_txt = 1, 2, 200, 64, 23
    inp = make_inputs(B, H, N, d, seed=34)
    g = run(ja, inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    q = inp.q.astype(np.float64)
    dots = np.abs(np.sum(q * g["dq"], axis=-1))
    scale = np.linalg.norm(q, axis=-1) * np.linalg.norm(g["dq"], axis=-1) + 1e-30
    assert float(np.max(dots / scale)) < 2e-2
    k = inp.k.astype(np.float64)
    dots = np.abs(np.sum(k * g["dk"], axis=-1))
    scale = np.linalg.norm(k, axis=-1) * np.linalg.norm(g["dk"], axis=-1) + 1e-30
    assert float(np.max(dots / scale)) < 2e-2


def test_key_sum_of_dv_equals_query_sum_of_dout(ja):
    """dV = P^T dO and the rows of P sum to one, so sum_n dv[n] = sum_n dout[n]
    per (b, h); P in bf16 leaves a relative error of order 2^-9."""
    B, H, N, d, n_txt = 2, 2, 333, 64, 77
    inp = make_inputs(B, H, N, d, seed=35)
    g = run(ja, inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, n_txt)
    lhs = g["dv"].sum(axis=2)
    rhs = inp.dout.astype(np.float64).sum(axis=2)
    assert relF(lhs, rhs) < 2e-2
