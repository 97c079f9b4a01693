"""Failure detection on the GPU without a GPU fault: a bounded wait that runs
out.  The stream kernel's test hook leaves one pipeline fill without its
copies; the consumers' wait on it gives up after a short limit, the kernel
sets the watchdog word and returns, and the context stays usable."""
import pytest

import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import workloads as W

from gpu_util import check_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset():
    rarn.watchdog(clear=True)
    yield
    rarn.set_path("auto")


@pytest.mark.parametrize("fill", [0, 5])
def test_wait_runs_out_and_is_reported(fill):
    import torch
    lib = rarn.library()
    w = W.workload("reduce_add_rms_norm", "bf16", 1000, 4096, R=3, eps=1e-6, seed=fill)
    d = W.generate(w)
    rarn.set_path("stream")
    assert lib.rarn_test_stall(fill, 20_000_000) == 0  # 20 ms bound
    run_gpu(w, d)  # outputs are not valid; the call must return
    torch.cuda.synchronize()
    flags = rarn.watchdog(clear=True)
    assert flags & 1, f"consumer timeout not reported (flags={flags})"
    # the context is still usable and the next launch is correct
    check_parity(w, d, what="after a watchdog timeout")
    assert rarn.watchdog(clear=True) == 0


# (the pair kernel's stages hold two K slabs: 8 fills per item at K = 1024;
# the one-SM kernel's one: 16)
@pytest.mark.parametrize("K,fill,pair,T", [(1024, 0, 1, 1000), (1024, 5, 1, 1000),
                                           (1024, 0, 0, 1000), (1024, 9, 0, 1000),
                                           (256, 0, None, 1000), (256, 2, None, 1000),
                                           (2048, 0, None, 64), (2048, 5, None, 64)])
def test_gemm_wait_runs_out_and_is_reported(K, fill, pair, T, tune):
    """The GEMM form (persistent kernel for K = 1024, on SM pairs or on one SM
    per tile; two CTAs per SM for K = 256; split K for 64 rows): one ring
    fill of CTA 0 never completes; every role's wait gives up within the
    limit, the CTA (or the pair) drains what it issued and frees its tensor
    memory, the watchdog bit is set, and the next call is correct."""
    import torch
    if pair is not None:
        # the persistent kernels, not split K, with y in their epilogue
        tune(gemm_pair=pair, gemm_split_k=0, gemm_norm_in_epilogue=1)
    H = 2048
    gen = torch.Generator(device="cuda").manual_seed(K + fill)
    a = torch.randn(T, K, device="cuda", generator=gen).to(torch.bfloat16)
    w = (torch.randn(H, K, device="cuda", generator=gen) / K ** 0.5).to(torch.bfloat16)
    r0 = torch.randn(T, H, device="cuda", generator=gen).to(torch.bfloat16)
    g = (torch.rand(H, device="cuda", generator=gen) + 0.5).to(torch.bfloat16)
    r_ref = r0.clone()
    y_ref = rarn.gemm_add_rms_norm(a, w, r_ref, g, 1e-6)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    lib = rarn.library()
    assert lib.rarn_test_stall(fill, 20_000_000) == 0  # 20 ms bound
    r_bad = r0.clone()
    rarn.gemm_add_rms_norm(a, w, r_bad, g, 1e-6)  # outputs not valid; the call must return
    torch.cuda.synchronize()
    flags = rarn.watchdog(clear=True)
    assert flags & 4, f"GEMM timeout not reported (flags={flags})"
    # the context is still usable and the next call is correct (bit-identical
    # to the clean run: deterministic kernels)
    r_again = r0.clone()
    y_again = rarn.gemm_add_rms_norm(a, w, r_again, g, 1e-6)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    assert torch.equal(y_again, y_ref) and torch.equal(r_again, r_ref)
