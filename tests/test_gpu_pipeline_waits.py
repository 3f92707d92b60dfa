"""The bounded waits of the streaming pipeline (every decode kernel runs on it): a
stage whose barrier can never complete makes the waiting warp give up after a short
limit, the kernel returns with RSSM_DEVERR_TIMEOUT set, and the next call on the
same stream runs normally.

The stalled stage is armed for 16 bytes more than its bulk copy delivers: the copy
itself lands, so nothing is left in flight when the CTA winds down (the producers
also wait, bounded, for the copies they issued). No wait in the library is
unbounded, so the GPU is never left waiting."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu

TILE = 4096  # floats per 16 KB tile


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def test_pipeline_copy_without_stall_is_exact():
    import ssm_linear_attention_gb300 as ssm
    n = 1000
    src = torch.randn(n * TILE, device="cuda")
    dst = torch.zeros_like(src)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm.rssm_debug_pipeline_copy(src, dst, n, -1, 1000, err)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)
    assert int(err.item()) == 0


@pytest.mark.parametrize("stall", [0, 517, 1999])
def test_stalled_stage_times_out_and_the_next_call_succeeds(stall):
    import ssm_linear_attention_gb300 as ssm
    n = 2000
    src = torch.randn(n * TILE, device="cuda")
    dst = torch.zeros_like(src)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ssm.rssm_debug_pipeline_copy(src, dst, n, stall, 2000, err)   # 2 ms wait limit
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert int(err.item()) & ssm.RSSM_DEVERR_TIMEOUT
    assert took < 1.0, took   # a few wait limits, not the 2 s of the decode kernels
    # the tiles of the CTAs that did not stall were copied
    done = (dst.view(n, TILE) == src.view(n, TILE)).all(dim=1)
    assert int(done.sum()) >= n // 2
    # the context is usable: the same stream runs the next call normally
    err.zero_()
    dst.zero_()
    ssm.rssm_debug_pipeline_copy(src, dst, n, -1, 2000, err)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)
    assert int(err.item()) == 0
