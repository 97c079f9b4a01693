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
