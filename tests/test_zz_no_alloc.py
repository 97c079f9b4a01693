"""The GEMM form's allocation-free entry point against the workspace one.

Callers that cannot allocate device memory (plug-ins whose host program owns
all of it, runtimes that forbid allocation once serving, latency-critical
code that cannot take cudaMalloc's implicit synchronisation) use
rarn_gemm_add_rms_norm_noalloc, which keeps its partial sums in an array the
library reserves on the GPU.  The same inputs go through both entry points;
the allocation-free one is called twice in a row, so the second call runs on
the scratch the first one left behind; every output must be bit-identical to
the workspace form's.  The file is collected last so that a run stopping at
the first failure has already run every other test."""
import pytest

import residual_add_rmsnorm_gb300 as rarn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,K", [
    (8, 4096, 4096),     # split K: its partial products fit the scratch too
    (300, 1024, 512),
    (4096, 4096, 1024),
    (40000, 8192, 64),   # 32 column tiles: more rows than the scratch holds (three launch
                         # sequences of 16128, 16128 and 7744 rows)
])
def test_noalloc_matches_workspace_entry_two_calls(T, H, K):
    import torch
    gen = torch.Generator(device="cuda").manual_seed(T + H + K)
    a = torch.randn(T, K, device="cuda", generator=gen).to(torch.bfloat16)
    w = (torch.randn(H, K, device="cuda", generator=gen) / K ** 0.5).to(torch.bfloat16)
    r0 = torch.randn(T, H, device="cuda", generator=gen).to(torch.bfloat16)
    g = (torch.rand(H, device="cuda", generator=gen) + 0.5).to(torch.bfloat16)
    r_ws = r0.clone()
    y_ws = rarn.gemm_add_rms_norm(a, w, r_ws, g, 1e-6)
    outs = []
    for _ in range(2):
        r_na = r0.clone()
        y_na = rarn.gemm_add_rms_norm_noalloc(a, w, r_na, g, 1e-6)
        outs.append((y_na, r_na))
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    for y_na, r_na in outs:
        assert torch.equal(y_na, y_ws)
        assert torch.equal(r_na, r_ws)
