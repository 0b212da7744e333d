"""Pins for the CPU oracle: it is checked against things other than itself.

* finite differences of every input element (tiny shapes, float64);
* a float64 torch cross-check (``F.rms_norm`` + SDPA math path + autograd);
* closed forms (all keys equal, N = 1, duplicated keys = one key with a
  ln(multiplicity) logit bias);
* invariants (softmax rows sum to one, token-permutation equivariance, head
  independence, linearity in V, RMSNorm scale invariance, sum_j x_j dx_j = 0
  at eps = 0, sum over keys of dk_hat = 0, sum over keys of dv = sum over
  queries of dout);
* bf16 rounding against torch's conversion, including exact ties;
* planted mistakes in a copy of the oracle are caught by the pins.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import jattn_oracle as jo
from joint_attention_gb300.inputs import CONFIGS, CfgStream, make_config_inputs, make_inputs, to_bf16_values

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def relF(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def rand_case(B, H, N, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, N, d)) * scale
    k = rng.standard_normal((B, H, N, d)) * scale
    v = rng.standard_normal((B, H, N, d))
    dout = rng.standard_normal((B, H, N, d))
    gq = rng.uniform(0.5, 1.5, d)
    gk = rng.uniform(0.5, 1.5, d)
    return q, k, v, dout, gq, gk


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def test_round_to_bf16_matches_torch_including_ties():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    # exact ties: a bf16 value plus half an ulp (low 16 bits = 0x8000)
    base = to_bf16_values(rng.standard_normal(5000).astype(np.float32)).view(np.uint32)
    ties = (base | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1.0, -1.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(to_bf16_values(x).astype(np.float64), want)


def test_round_to_bf16_single_rounding_from_float64():
    # 1 + 2^-8 + 2^-40 is above the tie between 1 and 1 + 2^-7: must round up
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8])
    got = oracle.round_to_bf16(x)
    np.testing.assert_array_equal(got, [1.0 + 2.0 ** -7, 1.0, 1.0 + 2.0 ** -6])


def test_q_hat_rounds_the_exact_product_at_a_bf16_midpoint():
    """A row of equal values 8 gives r = (64 + eps)^(-1/2), just below 1/8, so
    g x r = g (1 - eps/128 + ...).  With g the midpoint 1 + 3 * 2^-8 between
    the bf16 values 1 + 2^-7 and 1 + 2^-6 the exact product lies below the
    midpoint and must round down; with g one float32 step above it, up.  An
    fp32 r rounds to exactly 1/8 here and would put the product on the
    midpoint itself, where ties-to-even rounds up (1 + 2^-6 is the even one)."""
    d = 64
    x = np.full((1, 1, 1, d), 8.0)
    mid = 1.0 + 3 * 2.0 ** -8
    above = float(np.nextafter(np.float32(mid), np.float32(2.0)))
    for g, want in ((mid, 1.0 + 2.0 ** -7), (above, 1.0 + 2.0 ** -6), (-mid, None)):
        gv = np.full(d, g)
        xh, r = jo.rmsnorm_fwd(x, gv)
        assert r[0, 0, 0, 0] < 0.125
        got = jo.round_to_bf16(xh)
        if want is None:  # negative gain: the mirror image
            np.testing.assert_array_equal(got, -(1.0 + 2.0 ** -7))
        else:
            np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------------------
# Finite differences (no bf16 step, float64)
# ---------------------------------------------------------------------------
def _loss(q, k, v, gq, gk, dout, eps):
    O, _ = oracle.joint_attention_fwd(q, k, v, gq, gk, eps=eps, round_qk=False)
    return float(np.sum(O * dout))


def _fd_grad(arr, f, h=1e-6):
    g = np.zeros_like(arr)
    flat = arr.reshape(-1)
    gf = g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + h
        lp = f()
        flat[i] = old - h
        lm = f()
        flat[i] = old
        gf[i] = (lp - lm) / (2 * h)
    return g


def _check_fd(bwd_fn, B, H, N, d, seed, eps=jo.EPS, tol=1e-6):
    q, k, v, dout, gq, gk = rand_case(B, H, N, d, seed)
    an = bwd_fn(q, k, v, gq, gk, dout, eps=eps, round_qk=False)
    f = lambda: _loss(q, k, v, gq, gk, dout, eps)  # noqa: E731
    errs = {}
    for name, arr, key in (("q", q, "dq"), ("k", k, "dk"), ("v", v, "dv"), ("gq", gq, "dgq"), ("gk", gk, "dgk")):
        fd = _fd_grad(arr, f)
        errs[name] = relF(an[key], fd)
    return errs


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 4), (1, 2, 3, 4), (1, 1, 24, 4), (1, 1, 3, 64), (1, 1, 24, 64)])
def test_oracle_matches_finite_differences(B, H, N, d):
    errs = _check_fd(oracle.joint_attention_bwd, B, H, N, d, seed=N * 100 + d)
    for name, e in errs.items():
        if N == 1 and name in ("q", "k", "gq", "gk"):
            # N = 1: these gradients are exactly zero; compare absolutely
            continue
        assert e <= 1e-6, (name, e)


def test_n1_gradients_zero_by_finite_differences():
    q, k, v, dout, gq, gk = rand_case(1, 1, 1, 8, 5)
    an = oracle.joint_attention_bwd(q, k, v, gq, gk, dout, round_qk=False)
    for name, arr, key in (("q", q, "dq"), ("k", k, "dk"), ("gq", gq, "dgq"), ("gk", gk, "dgk")):
        fd = _fd_grad(arr, lambda: _loss(q, k, v, gq, gk, dout, jo.EPS))
        assert np.max(np.abs(fd)) < 1e-8
        assert np.max(np.abs(an[key])) < 1e-12


# ---------------------------------------------------------------------------
# Planted mistakes must be caught by the finite-difference pin
# ---------------------------------------------------------------------------
def _mutant_bwd(kind):
    def rmsnorm_bwd_mut(x, g, r, dxhat):
        d = x.shape[-1]
        u = g * dxhat
        if kind == "drop_r3_term":
            dx = r * u
        elif kind == "sign_r3_term":
            dx = r * u + (r ** 3 / d) * x * np.sum(u * x, axis=-1, keepdims=True)
        else:
            dx = r * u - (r ** 3 / d) * x * np.sum(u * x, axis=-1, keepdims=True)
        dg = np.sum((dxhat * x * (r if kind != "dg_no_r" else 1.0)).reshape(-1, d), axis=0)
        return dx, dg

    def attn_bwd_mut(qh, kh, v, P, O, dout, scale):
        if kind == "transpose_dv":
            dv = P @ dout
        else:
            dv = P.T @ dout
        dP = dout @ v.T
        D = np.sum(dout * O, axis=1, keepdims=True)
        dS = P * (dP - (0.0 if kind == "drop_D" else D))
        dqh = (dS @ kh) * (1.0 if kind == "no_scale_dq" else scale)
        dkh = (dS @ qh if kind == "dk_no_transpose" else dS.T @ qh) * scale
        return dqh, dkh, dv

    def bwd(q, k, v, gq, gk, dout, eps=jo.EPS, round_qk=True):
        saved = (jo.rmsnorm_bwd, jo.attention_bwd_head)
        jo.rmsnorm_bwd, jo.attention_bwd_head = rmsnorm_bwd_mut, attn_bwd_mut
        try:
            return jo.joint_attention_bwd(q, k, v, gq, gk, dout, eps=eps, round_qk=round_qk)
        finally:
            jo.rmsnorm_bwd, jo.attention_bwd_head = saved

    return bwd


@pytest.mark.parametrize("kind", ["drop_r3_term", "sign_r3_term", "dg_no_r", "transpose_dv", "drop_D",
                                  "no_scale_dq", "dk_no_transpose"])
def test_planted_mistakes_are_caught(kind):
    errs = _check_fd(_mutant_bwd(kind), 1, 1, 5, 4, seed=11)
    assert max(errs.values()) > 1e-3, (kind, errs)


# ---------------------------------------------------------------------------
# Library cross-check: torch float64 (F.rms_norm, SDPA, autograd)
# ---------------------------------------------------------------------------
def torch_reference(q, k, v, gq, gk, dout, eps=jo.EPS, round_qk=True):
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)  # noqa: E731
    tq, tk, tv, tgq, tgk = t(q), t(k), t(v), t(gq), t(gk)
    d = q.shape[-1]
    qh = F.rms_norm(tq, (d,), weight=tgq, eps=eps)
    kh = F.rms_norm(tk, (d,), weight=tgk, eps=eps)
    if round_qk:
        # straight-through bf16 rounding (via float32; a double-rounding
        # difference would need an exact bf16 tie after the float32 step)
        qh = qh + (qh.detach().float().to(torch.bfloat16).double() - qh.detach())
        kh = kh + (kh.detach().float().to(torch.bfloat16).double() - kh.detach())
    from torch.nn.attention import SDPBackend, sdpa_kernel
    with sdpa_kernel(SDPBackend.MATH):
        O = F.scaled_dot_product_attention(qh, kh, tv, scale=1.0 / math.sqrt(d))
    lse = torch.logsumexp((qh @ kh.transpose(-1, -2)) / math.sqrt(d), dim=-1)
    (O * torch.tensor(np.asarray(dout, np.float64))).sum().backward()
    return {"O": O.detach().numpy(), "LSE": lse.detach().numpy(), "dq": tq.grad.numpy(), "dk": tk.grad.numpy(),
            "dv": tv.grad.numpy(), "dgq": tgq.grad.numpy(), "dgk": tgk.grad.numpy()}


@pytest.mark.parametrize("round_qk", [False, True])
@pytest.mark.parametrize("B,H,N,d,seed", [(1, 2, 24, 64, 0), (2, 3, 37, 128, 1), (1, 1, 129, 64, 2)])
def test_oracle_matches_torch_float64(B, H, N, d, seed, round_qk):
    q, k, v, dout, gq, gk = rand_case(B, H, N, d, seed)
    ours = oracle.joint_attention_bwd(q, k, v, gq, gk, dout, round_qk=round_qk)
    ref = torch_reference(q, k, v, gq, gk, dout, round_qk=round_qk)
    for key in ("O", "LSE", "dq", "dk", "dv", "dgq", "dgk"):
        assert relF(ours[key], ref[key]) < 1e-12, key


def torch_reference_block_diagonal(q, k, v, gq, gk, dout, cu, eps=jo.EPS):
    """Packed sequences as one attention over all T rows with a block-diagonal
    boolean mask (torch float64, SDPA math path, autograd): an independent
    formulation of the per-sequence split."""
    t = lambda a: torch.tensor(np.asarray(a, np.float64)[None], requires_grad=True)  # noqa: E731
    tq, tk, tv = t(q), t(k), t(v)
    tgq = torch.tensor(np.asarray(gq, np.float64), requires_grad=True)
    tgk = torch.tensor(np.asarray(gk, np.float64), requires_grad=True)
    d, T = q.shape[-1], q.shape[1]
    seg = np.zeros(T, dtype=np.int64)
    for s_, (a, b) in enumerate(zip(cu, cu[1:])):
        seg[a:b] = s_
    mask = torch.tensor(seg[:, None] == seg[None, :])
    # No bf16 step: the rounding is pinned on its own; this pins the split.
    qh = F.rms_norm(tq, (d,), weight=tgq, eps=eps)
    kh = F.rms_norm(tk, (d,), weight=tgk, eps=eps)
    from torch.nn.attention import SDPBackend, sdpa_kernel
    with sdpa_kernel(SDPBackend.MATH):
        O = F.scaled_dot_product_attention(qh, kh, tv, attn_mask=mask, scale=1.0 / math.sqrt(d))
    S = (qh @ kh.transpose(-1, -2)) / math.sqrt(d)
    lse = torch.logsumexp(S.masked_fill(~mask, float("-inf")), dim=-1)
    (O * torch.tensor(np.asarray(dout, np.float64)[None])).sum().backward()
    return {"O": O.detach().numpy()[0], "LSE": lse.detach().numpy()[0], "dq": tq.grad.numpy()[0],
            "dk": tk.grad.numpy()[0], "dv": tv.grad.numpy()[0], "dgq": tgq.grad.numpy(), "dgk": tgk.grad.numpy()}


@pytest.mark.parametrize("cu,d", [([0, 24, 25, 70, 203], 64), ([0, 7, 140], 128), ([0, 1], 64)])
def test_varlen_oracle_matches_block_diagonal_masked_attention(cu, d):
    rng = np.random.default_rng(len(cu) * 100 + d)
    H, T = 2, cu[-1]
    q, k, v, dout = (rng.standard_normal((H, T, d)) for _ in range(4))
    gq, gk = rng.uniform(0.5, 1.5, d), rng.uniform(0.5, 1.5, d)
    ours = oracle.joint_attention_varlen_bwd(q, k, v, gq, gk, dout, cu, round_qk=False)
    ref = torch_reference_block_diagonal(q, k, v, gq, gk, dout, cu)
    for key in ("O", "LSE", "dq", "dk", "dv", "dgq", "dgk"):
        assert relF(ours[key], ref[key]) < 1e-12, key


def test_varlen_oracle_rejects_bad_offsets():
    q = np.zeros((1, 5, 4))
    for cu in ([1, 5], [0, 3, 3, 5], [0, 4]):
        with pytest.raises(ValueError):
            oracle.joint_attention_varlen_bwd(q, q, q, np.ones(4), np.ones(4), q, cu)


@pytest.mark.parametrize("name", ["tiny", "256px"])
def test_oracle_matches_torch_on_workloads(name):
    inp = make_config_inputs(CONFIGS[name])
    sl = slice(0, 2)  # first two batch items, all heads
    args = [a[sl] for a in (inp.q, inp.k, inp.v)]
    # round_qk=False: torch converts float64 -> bf16 through float32, and on
    # half a million elements a few of those double roundings land on a tie.
    # The rounding itself is pinned by the two tests above.
    ours = oracle.joint_attention_bwd(*args, inp.gq, inp.gk, inp.dout[sl], round_qk=False)
    ref = torch_reference(*args, inp.gq, inp.gk, inp.dout[sl], round_qk=False)
    for key in ("O", "LSE", "dq", "dk", "dv", "dgq", "dgk"):
        assert relF(ours[key], ref[key]) < 1e-11, key


def test_oracle_matches_torch_on_sampled_heads_of_large_workloads():
    for name in ("512px", "768px_d128"):
        c = CONFIGS[name]
        inp = make_inputs(1, 1, c.N, c.d, seed=c.seed + 100, value_scale=c.value_scale)
        ours = oracle.joint_attention_bwd(inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, round_qk=False)
        ref = torch_reference(inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout, round_qk=False)
        for key in ("O", "LSE", "dq", "dk", "dv", "dgq", "dgk"):
            assert relF(ours[key], ref[key]) < 1e-11, (name, key)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
def test_all_keys_equal_gives_mean_of_values():
    B, H, N, d = 1, 2, 17, 64
    q, k, v, dout, gq, gk = rand_case(B, H, N, d, 3)
    k[:] = k[:, :, :1, :]
    res = oracle.joint_attention_bwd(q, k, v, gq, gk, dout, return_state=True)
    np.testing.assert_allclose(res["O"], np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape), atol=1e-13)
    s_const = np.einsum("bhnd,bhd->bhn", res["qhat"], res["khat"][:, :, 0, :]) / math.sqrt(d)
    np.testing.assert_allclose(res["LSE"], s_const + math.log(N), atol=1e-12)
    assert np.max(np.abs(res["dq"])) < 1e-12
    assert np.max(np.abs(res["dgq"])) < 1e-12


def test_single_token_closed_form():
    q, k, v, dout, gq, gk = rand_case(2, 3, 1, 64, 4)
    res = oracle.joint_attention_bwd(q, k, v, gq, gk, dout, return_state=True)
    np.testing.assert_allclose(res["O"], v, atol=1e-14)
    s = np.sum(res["qhat"] * res["khat"], axis=-1) / 8.0
    np.testing.assert_allclose(res["LSE"], s, atol=1e-13)
    np.testing.assert_allclose(res["dv"], dout, atol=1e-14)
    for key in ("dq", "dk", "dgq", "dgk"):
        assert np.max(np.abs(res[key])) < 1e-12


def test_duplicated_keys_act_as_one_key_with_log_multiplicity():
    # CFG unconditional branch: the m text rows share one key/value vector.
    rng = np.random.default_rng(7)
    d, n_img, m = 64, 30, 77
    gq, gk = rng.uniform(0.5, 1.5, d), rng.uniform(0.5, 1.5, d)
    q = rng.standard_normal((1, 1, m + n_img, d))
    k_img = rng.standard_normal((n_img, d))
    v_img = rng.standard_normal((n_img, d))
    kt, vt = rng.standard_normal(d), rng.standard_normal(d)
    k = np.concatenate([np.tile(kt, (m, 1)), k_img])[None, None]
    v = np.concatenate([np.tile(vt, (m, 1)), v_img])[None, None]
    O, lse, st = oracle.joint_attention_fwd(q, k, v, gq, gk, return_state=True)
    # collapsed sequence: one text key with logit + ln m, computed directly
    qh, khat = st["qhat"][0, 0], st["khat"][0, 0]
    S = qh @ khat[m - 1:].T / 8.0  # row 0 = the (one) text key, then image keys
    S[:, 0] += math.log(m)
    w = np.exp(S - S.max(axis=1, keepdims=True))
    want_lse = S.max(axis=1) + np.log(w.sum(axis=1))
    want_O = (w / w.sum(axis=1, keepdims=True)) @ np.concatenate([vt[None], v_img])
    np.testing.assert_allclose(O[0, 0], want_O, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], want_lse, atol=1e-12)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------
def test_softmax_rows_sum_to_one():
    q, k, v, dout, gq, gk = rand_case(1, 1, 50, 64, 8)
    qh, _ = oracle.rmsnorm_fwd(q[0, 0], gq)
    kh, _ = oracle.rmsnorm_fwd(k[0, 0], gk)
    _, lse, P = oracle.attention_fwd_head(qh, kh, v[0, 0], 1 / 8.0)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(P >= 0)


def test_token_permutation_equivariance():
    q, k, v, dout, gq, gk = rand_case(1, 2, 29, 64, 9)
    perm = np.random.default_rng(1).permutation(29)
    a = oracle.joint_attention_bwd(q, k, v, gq, gk, dout)
    b = oracle.joint_attention_bwd(q[:, :, perm], k[:, :, perm], v[:, :, perm], gq, gk, dout[:, :, perm])
    for key in ("O", "LSE", "dq", "dk", "dv"):
        np.testing.assert_allclose(b[key], a[key][:, :, perm], atol=1e-12, rtol=1e-12)
    for key in ("dgq", "dgk"):
        np.testing.assert_allclose(b[key], a[key], atol=1e-12, rtol=1e-12)


def test_head_and_batch_independence():
    q, k, v, dout, gq, gk = rand_case(2, 3, 11, 64, 10)
    full = oracle.joint_attention_bwd(q, k, v, gq, gk, dout)
    dgq = np.zeros(64)
    for b in range(2):
        for h in range(3):
            one = oracle.joint_attention_bwd(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], gq, gk,
                                             dout[b:b + 1, h:h + 1])
            for key in ("O", "LSE", "dq", "dk", "dv"):
                np.testing.assert_allclose(one[key][0, 0], full[key][b, h], atol=1e-14)
            dgq += one["dgq"]
    np.testing.assert_allclose(dgq, full["dgq"], atol=1e-12)


def test_output_linear_in_v():
    q, k, v, dout, gq, gk = rand_case(1, 1, 20, 64, 12)
    v2 = np.random.default_rng(2).standard_normal(v.shape)
    O1, _ = oracle.joint_attention_fwd(q, k, v, gq, gk)
    O2, _ = oracle.joint_attention_fwd(q, k, v2, gq, gk)
    O3, _ = oracle.joint_attention_fwd(q, k, 2.0 * v - 3.0 * v2, gq, gk)
    np.testing.assert_allclose(O3, 2.0 * O1 - 3.0 * O2, atol=1e-12)


def test_rmsnorm_scale_invariance():
    q, k, v, dout, gq, gk = rand_case(1, 2, 15, 64, 13)
    a = oracle.joint_attention_fwd(q, k, v, gq, gk, eps=0.0, round_qk=False)
    b = oracle.joint_attention_fwd(3.7 * q, 0.25 * k, v, gq, gk, eps=0.0, round_qk=False)
    np.testing.assert_allclose(b[0], a[0], atol=1e-12)
    np.testing.assert_allclose(b[1], a[1], atol=1e-12)


def test_norm_gradient_orthogonal_to_input_at_eps0():
    q, k, v, dout, gq, gk = rand_case(1, 2, 15, 64, 14)
    res = oracle.joint_attention_bwd(q, k, v, gq, gk, dout, eps=0.0, round_qk=False)
    for x, key in ((q, "dq"), (k, "dk")):
        dots = np.sum(x * res[key], axis=-1)
        assert np.max(np.abs(dots)) < 1e-12 * np.max(np.abs(res[key])) * 64 + 1e-13


def test_key_gradient_sums_and_value_gradient_sums():
    q, k, v, dout, gq, gk = rand_case(2, 2, 23, 64, 15)
    res = oracle.joint_attention_bwd(q, k, v, gq, gk, dout, return_state=True)
    np.testing.assert_allclose(res["dkhat"].sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(res["dv"].sum(axis=2), dout.sum(axis=2), atol=1e-12)


def test_stream_concat_and_split_matches_joint_sequence():
    rng = np.random.default_rng(16)
    n_txt, n_img, d = 7, 12, 64
    parts = [rng.standard_normal((1, 2, n, d)) for n in (n_txt, n_txt, n_txt, n_img, n_img, n_img)]
    gq, gk = rng.uniform(0.5, 1.5, d), rng.uniform(0.5, 1.5, d)
    o_txt, o_img, lse = oracle.joint_attention_streams(*parts, gq, gk)
    q = np.concatenate([parts[0], parts[3]], axis=2)
    k = np.concatenate([parts[1], parts[4]], axis=2)
    v = np.concatenate([parts[2], parts[5]], axis=2)
    O, L = oracle.joint_attention_fwd(q, k, v, gq, gk)
    np.testing.assert_array_equal(o_txt, O[:, :, :n_txt])
    np.testing.assert_array_equal(o_img, O[:, :, n_txt:])
    # joint attention differs from attending within each stream alone
    o_sep, _ = oracle.joint_attention_fwd(parts[3], parts[4], parts[5], gq, gk)
    assert np.max(np.abs(o_sep - o_img)) > 1e-3


def test_one_row_helper_matches_full():
    q, k, v, dout, gq, gk = rand_case(1, 1, 40, 64, 17)
    O, lse = oracle.joint_attention_fwd(q, k, v, gq, gk)
    for i in (0, 17, 39):
        o, l = oracle.attention_one_row(q[0, 0, i], k[0, 0], v[0, 0], gq, gk)
        np.testing.assert_allclose(o, O[0, 0, i], atol=1e-14)
        assert abs(l - lse[0, 0, i]) < 1e-13


# ---------------------------------------------------------------------------
# Input generator
# ---------------------------------------------------------------------------
def test_generator_is_seeded_bf16_and_in_draw_order():
    a = make_inputs(1, 2, 24, 64, seed=0)
    b = make_config_inputs(CONFIGS["tiny"])
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.dout, b.dout), (a.gq, b.gq), (a.gk, b.gk)):
        np.testing.assert_array_equal(x, y)
    rng = np.random.default_rng(0)
    np.testing.assert_array_equal(a.q, to_bf16_values(rng.standard_normal((1, 2, 24, 64), dtype=np.float32)))
    for x in (a.q, a.k, a.v, a.dout, a.gq, a.gk):
        np.testing.assert_array_equal(x, to_bf16_values(x))
    assert a.gq.min() >= 0.5 and a.gq.max() <= 1.5


def test_cfg_stream_uncond_text_rows_are_shared():
    st = CfgStream(CONFIGS["cfg_512px"])
    s0 = st.next_step()
    s1 = st.next_step()
    for arr in (s0.q, s0.k, s0.v):
        t = arr[8:, :, :77, :]
        assert np.all(t == t[:1, :, :1, :])
        assert not np.all(arr[:8, :, :77, :] == arr[:1, :, :1, :])
    assert not np.array_equal(s0.q, s1.q)
    np.testing.assert_array_equal(s0.gq, s1.gq)


def test_oracle_reproduces_its_stored_tiny_values():
    """tests/golden/tiny_oracle.json was written by tests/golden/make_oracle_golden.py, which calls
    only the oracle (the pages print no worked example).  A change to the oracle's arithmetic shows
    here first."""
    import json
    import os
    import sys

    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    try:
        from make_oracle_golden import golden
    finally:
        sys.path.remove(here)
    stored = json.load(open(os.path.join(here, "tiny_oracle.json")))
    now = golden()
    assert stored["workload"] == now["workload"] and stored["rows"] == now["rows"]
    for key in ("LSE", "dgq", "dgk", "O_rows", "dq_rows", "dk_rows", "dv_rows"):
        a, b = np.asarray(now[key]), np.asarray(stored[key])
        assert a.shape == b.shape, key
        assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b))), key
    for key, v in stored["norms"].items():
        assert abs(now["norms"][key] - v) <= 1e-12 * v, key


# ---------------------------------------------------------------------------
# QKV projection per stream, then QK-RMSNorm ("architecture flowchart")
# ---------------------------------------------------------------------------
def _one_hot_layout_errors(fn, B=2, H=3, d=4, N_img=5, N_txt=3, C=16, seed=3):
    """Tokens that are unit vectors turn the projection into a lookup: the
    token (b, n) of a stream with x = e_c gives, for head h and element e,
    q = w[h d + e, c] + b[h d + e], k = w[H d + h d + e, c] + ..., v = w[2 H d
    + h d + e, c] + ..., at joint row n (caption stream) or N_txt + n (image
    stream).  Returns the number of elements of q, k, v that differ from that
    lookup (with the bf16 rounding of each looked-up value)."""
    rng = np.random.default_rng(seed)
    ws = {s: to_bf16_values(rng.standard_normal((3 * H * d, C)).astype(np.float32)) for s in ("img", "txt")}
    bs = {s: rng.standard_normal(3 * H * d) for s in ("img", "txt")}
    cs = {"img": rng.integers(0, C, (B, N_img)), "txt": rng.integers(0, C, (B, N_txt))}
    xs = {}
    for s, n_s in (("img", N_img), ("txt", N_txt)):
        x = np.zeros((B, n_s, C))
        for b in range(B):
            for n in range(n_s):
                x[b, n, cs[s][b, n]] = 1.0
        xs[s] = x
    gq = rng.uniform(0.5, 1.5, d)
    gk = rng.uniform(0.5, 1.5, d)
    out = fn(xs["img"], ws["img"], bs["img"], xs["txt"], ws["txt"], bs["txt"], gq, gk, H)
    wrong = 0
    for s, n_s, row0 in (("img", N_img, N_txt), ("txt", N_txt, 0)):
        for b in range(B):
            for n in range(n_s):
                c = cs[s][b, n]
                for which, key in enumerate(("q", "k", "v")):
                    for h in range(H):
                        for e in range(d):
                            j = which * H * d + h * d + e
                            want = oracle.round_to_bf16(np.array([ws[s][j, c] + bs[s][j]]))[0]
                            wrong += int(out[key][b, h, row0 + n, e] != want)
    return wrong


def test_qkv_projection_one_hot_tokens_look_up_weight_columns():
    assert _one_hot_layout_errors(oracle.qkv_norm_streams) == 0


def test_qkv_projection_of_all_ones_tokens_is_the_weight_row_sum():
    rng = np.random.default_rng(4)
    B, N_s, C, H, d = 2, 3, 24, 2, 8
    w = rng.standard_normal((3 * H * d, C))
    b = rng.standard_normal(3 * H * d)
    Y, _ = oracle.qkv_projection(np.ones((B, N_s, C)), w, b, H)
    rowsum = w.sum(axis=1) + b
    for which in range(3):
        for h in range(H):
            want = rowsum[which * H * d + h * d:which * H * d + (h + 1) * d]
            np.testing.assert_allclose(Y[which, :, h], np.broadcast_to(want, (B, N_s, d)), rtol=1e-13, atol=1e-13)


def test_qkv_projection_rounds_the_exact_sum_once():
    """bf16 keeps 8 significant bits: at 1 its spacing is 2^-7.  An exact sum
    of 1 + 2^-8 is a tie and goes to the even neighbour 1; 1 + 3 2^-8 goes to
    1 + 2^-6; a bias of 2^-30 on the first tie moves the exact value above the
    midpoint, so one rounding gives 1 + 2^-7 (rounding through fp32 first
    would lose the 2^-30 and give 1)."""
    H, d = 1, 1
    w = np.zeros((3, 2))
    w[:, 0] = 1.0
    w[:, 1] = 2.0 ** -8
    x = np.array([[[1.0, 1.0], [1.0, 3.0]]])
    _, Yr = oracle.qkv_projection(x, w, None, H)
    assert Yr[0, 0, 0, 0, 0] == 1.0 and Yr[0, 0, 0, 1, 0] == 1.0 + 2.0 ** -6
    _, Yr = oracle.qkv_projection(x[:, :1], w, np.full(3, 2.0 ** -30), H)
    assert Yr[0, 0, 0, 0, 0] == 1.0 + 2.0 ** -7


def test_qkv_norm_streams_matches_torch_float64():
    """The float64 torch route (F.linear, view / permute into heads, cat along
    the tokens caption first, F.rms_norm) gives the same values."""
    B, H, N_img, N_txt, d, C = 2, 3, 7, 4, 8, 16
    from joint_attention_gb300.inputs import make_qkv_inputs

    inp = make_qkv_inputs(B, H, N_img, N_txt, d, C, seed=9)
    ref = oracle.qkv_norm_streams(inp.x_img, inp.w_img, inp.b_img, inp.x_txt, inp.w_txt, inp.b_txt, inp.gq,
                                  inp.gk, H)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))  # noqa: E731

    def proj(x, w, b):
        y = F.linear(t(x), t(w), t(b))                      # [B, N_s, 3 H d]
        return y.view(B, -1, 3, H, d).permute(2, 0, 3, 1, 4)  # [3, B, H, N_s, d]

    y = torch.cat([proj(inp.x_txt, inp.w_txt, inp.b_txt), proj(inp.x_img, inp.w_img, inp.b_img)], dim=3)
    np.testing.assert_allclose(ref["y_exact"], y.numpy(), rtol=1e-12, atol=1e-12)
    for key, i, g in (("qhat", 0, inp.gq), ("khat", 1, inp.gk)):
        xr = t(ref["qkv"[i]])
        want = F.rms_norm(xr, (d,), weight=t(g), eps=jo.EPS)
        np.testing.assert_allclose(ref[key], oracle.round_to_bf16(want.numpy()), rtol=0, atol=0)
        rr = torch.rsqrt(xr.pow(2).mean(-1) + jo.EPS)
        np.testing.assert_allclose(ref["r" + "qk"[i]], rr.numpy(), rtol=1e-14)


def _mutant_streams(kind):
    def proj(x, w, b, H):
        x, w = np.asarray(x, np.float64), np.asarray(w, np.float64)
        B, N_s, _ = x.shape
        d = w.shape[0] // (3 * H)
        Y = x @ w.T + (0.0 if kind == "no_bias" or b is None else b)
        if kind == "heads_outer":       # q / k / v interleaved per head
            Y = Y.reshape(B, N_s, H, 3, d).transpose(3, 0, 2, 1, 4)
        elif kind == "dim_outer":       # head index and element index swapped
            Y = Y.reshape(B, N_s, 3, d, H).transpose(2, 0, 4, 1, 3)
        else:
            Y = Y.reshape(B, N_s, 3, H, d).transpose(2, 0, 3, 1, 4)
        return Y, oracle.round_to_bf16(Y)

    def streams(x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk, H):
        parts = [proj(x_txt, w_txt, b_txt, H), proj(x_img, w_img, b_img, H)]
        if kind == "image_first":
            parts = parts[::-1]
        q, k, v = np.concatenate([p[1] for p in parts], axis=3)
        return {"q": q, "k": k, "v": v}

    return streams


@pytest.mark.parametrize("kind", ["no_bias", "heads_outer", "dim_outer", "image_first"])
def test_planted_projection_mistakes_are_caught(kind):
    assert _one_hot_layout_errors(_mutant_streams(kind)) > 0
