"""The allocation-free prefill entry point, w4a8_prefill_linear_noalloc.

Some callers cannot give the library a workspace: they run where device allocation is
not allowed or not wanted (allocator-free runtimes, code that must not synchronize the
device the way cudaMalloc/cudaFree can, or a fixed device-memory budget).  For them the
library keeps one statically reserved scratch array per GPU and this entry point uses it
instead of a caller-provided workspace.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_y, inputs_to_dev
from w4a8_block_quantized_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a8_block_quantized_gb300 import binding, build
    build.build()
    binding.load()
    oracle.build()
    torch.cuda.set_device(0)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    """Two consecutive calls of different shapes (the second reuses the scratch the first
    left behind) agree with w4a8_prefill_linear bit for bit and with the oracle within the
    fp32 tolerance."""
    from w4a8_block_quantized_gb300 import binding as b
    for M, K, N, seed in ((300, 1024, 700, 31), (512, 2048, 1024, 32)):
        d = synth.random_small(M, K, N, seed=seed, bias=True)
        g = inputs_to_dev(d)
        y_ws = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
        y = torch.full((M, N), float("nan"), device=g["x"].device)
        b.prefill_linear_noalloc(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y)
        assert b.sync_status() == 0
        assert torch.equal(y, y_ws)
        y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
        check_y(y, y_ref, bound, f"noalloc {M}x{K}->{N}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    from w4a8_block_quantized_gb300 import binding as b
    M, K, N = 4096, 4096, 256  # needs about 39 MB of scratch, more than the 16 MiB array
    assert b.prefill_workspace_bytes(M, N, K) > b.NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    x = torch.zeros((M, K), device=dev)
    wq = torch.zeros((N, K // 2), dtype=torch.uint8, device=dev)
    s = torch.zeros((N, K // 64), dtype=torch.float16, device=dev)
    y = torch.full((M, N), 7.0, device=dev)
    with pytest.raises(b.W4A8Error) as e:
        b.prefill_linear_noalloc(x, wq, s, s, None, y=y)
    assert e.value.status == b.W4A8_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())  # nothing was launched
