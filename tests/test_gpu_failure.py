"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The self-test kernel waits on an mbarrier that nothing arrives at, through the
same bounded wait the attention kernels use.  The wait must give up after its
limit (about 1 s), the host must read JATTN_ERR_TIMEOUT, and the context must
stay usable: a forward + backward right after it matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from joint_attention_gb300.inputs import CONFIGS, make_config_inputs

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


def test_bounded_wait_gives_up_and_the_context_stays_usable(ja):
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0  # also clears any earlier record
    t0 = time.perf_counter()
    ja.jattn_selftest_wait_timeout()
    rc = ja.jattn_last_device_error()  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert rc == ja.STATUS_CODE["JATTN_ERR_TIMEOUT"], ja.STATUS.get(rc, rc)
    assert 0.9 <= elapsed <= 30.0, elapsed
    # the record is cleared by the read
    assert ja.jattn_last_device_error() == 0

    cfg = CONFIGS["tiny"]
    inp = make_config_inputs(cfg)
    bf = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16).contiguous()  # noqa: E731
    f32 = lambda a: torch.from_numpy(a).cuda().float().contiguous()  # noqa: E731
    q, k, v, dout = bf(inp.q), bf(inp.k), bf(inp.v), bf(inp.dout)
    gq, gk = f32(inp.gq), f32(inp.gk)
    out, lse = ja.forward(q, k, v, gq, gk, cfg.N_txt)
    dq, dk, dv, dgq, dgk = ja.backward(q, k, v, gq, gk, out, lse, dout, cfg.N_txt)
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0
    ref = oracle.joint_attention_bwd(inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout)
    got_o = out.float().cpu().numpy().astype(np.float64)
    assert float(np.max(np.abs(got_o - ref["O"]))) <= 1e-2
    assert float(np.max(np.abs(lse.cpu().numpy() - ref["LSE"]))) <= 1e-3
    for key, t in (("dq", dq), ("dk", dk), ("dv", dv), ("dgq", dgq), ("dgk", dgk)):
        a = t.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(a - ref[key]) <= 2e-2 * np.linalg.norm(ref[key]), key
