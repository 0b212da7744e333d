"""jattn_fwd_noalloc: the forward whose scratch lives in a fixed device array.

Some callers cannot let a library allocate device memory (a serving process
that has reserved nearly all of HBM for its own pool, or a launch sequence that
must never block on or recover from an allocator call).  For them the library
exports jattn_fwd_noalloc, which keeps its q_hat / k_hat scratch in one
64 MiB file-scope device array instead of a per-call allocation.  These tests
call it through the C ABI and check it against jattn_fwd; the file is named so
that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import joint_attention_gb300 as ja
from joint_attention_gb300 import STATUS_CODE
from joint_attention_gb300.build import build
from joint_attention_gb300.inputs import CONFIGS, make_config_inputs, make_inputs

O_MAXABS, O_RELF, LSE_MAXABS = 1e-2, 5e-3, 1e-3


def test_noalloc_rejects_problems_beyond_its_array():
    build()
    lib = ja.load_library()
    A = 0x7F0000000000  # never dereferenced: the size check comes before any CUDA call
    # 768 px, d = 128: B*H*N*d = 4*24*2381*128 > 2^24 elements
    rc = lib.jattn_fwd_noalloc(A, A + 0x10000000, A + 0x20000000, A + 0x30000000, A + 0x30001000, 4, 24, 2304, 77,
                               128, A + 0x40000000, A + 0x50000000, None)
    assert rc == STATUS_CODE["JATTN_ERR_SCRATCH_LIMIT"]
    assert ja.jattn_status_string(rc) != "unknown status"
    # the ordinary argument checks still apply
    rc = lib.jattn_fwd_noalloc(None, A, A, A, A, 1, 1, 1, 0, 64, A, A, None)
    assert rc == STATUS_CODE["JATTN_ERR_INVALID_ARG"]


@pytest.mark.gpu
def test_noalloc_matches_jattn_fwd_on_two_calls_in_a_row():
    """Two no-allocation calls back to back on one stream, on different inputs, with no
    synchronisation between them: the second call's normalisation pass reuses the shared array
    while the first call's attention may still read it, so the outputs show whether the launch
    order keeps them apart.  Each is compared with jattn_fwd on the same inputs."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build()
    ja.load_library()
    dev = torch.device("cuda:0")
    bf = lambda a: torch.from_numpy(a).to(dev).to(torch.bfloat16).contiguous()  # noqa: E731
    f32 = lambda a: torch.from_numpy(a).to(dev).float().contiguous()  # noqa: E731
    cases = [(make_config_inputs(CONFIGS["512px"]), CONFIGS["512px"].N_txt),
             (make_inputs(2, 3, 333, 128, seed=21), 77),
             (make_inputs(16, 12, 1101, 64, seed=22), 77)]
    runs = []
    for inp, n_txt in cases:
        B, H, N, d = inp.q.shape
        t = dict(q=bf(inp.q), k=bf(inp.k), v=bf(inp.v), gq=f32(inp.gq), gk=f32(inp.gk))
        t["out_a"], t["lse_a"] = torch.empty_like(t["q"]), torch.empty((B, H, N), device=dev, dtype=torch.float32)
        t["out_b"] = torch.full_like(t["q"], float("nan"))
        t["lse_b"] = torch.full((B, H, N), float("nan"), device=dev, dtype=torch.float32)
        ja.jattn_fwd(t["q"], t["k"], t["v"], t["gq"], t["gk"], B, H, N - n_txt, n_txt, d, t["out_a"], t["lse_a"])
        runs.append((t, (B, H, N, d, n_txt)))
    torch.cuda.synchronize()
    for t, (B, H, N, d, n_txt) in runs:  # back to back, same stream, no synchronisation
        rc = ja.jattn_fwd_noalloc(t["q"], t["k"], t["v"], t["gq"], t["gk"], B, H, N - n_txt, n_txt, d, t["out_b"],
                                  t["lse_b"])
        assert rc == 0
    torch.cuda.synchronize()
    assert ja.jattn_last_device_error() == 0
    for t, _ in runs:
        a = t["out_a"].float().cpu().numpy().astype(np.float64)
        b = t["out_b"].float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(b))
        assert float(np.max(np.abs(a - b))) <= O_MAXABS
        assert float(np.linalg.norm(a - b) / np.linalg.norm(a)) <= O_RELF
        assert float((t["lse_a"] - t["lse_b"]).abs().max()) <= LSE_MAXABS
