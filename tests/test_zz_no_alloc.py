"""rssm_mamba2_decode_noalloc against rssm_mamba2_decode.

The no-allocation entry point serves callers that cannot allocate device memory
(its workspace is a fixed array inside the library's device image). It must give
the same decode results as the regular entry point, which takes a caller-allocated
workspace. Two decoders start from identical state and see identical inputs; for
two calls in a row, one decodes through rssm_mamba2_decode and the other through
rssm_mamba2_decode_noalloc, both through the C ABI. Outputs, flushed states and
cursors must agree within the bf16-state tolerance (the kernels are the same, so
they agree exactly). This file is collected last so that a run stopping at the
first failure has run every other test; it passes alone or after the rest.
"""
import numpy as np
import pytest
import torch

import rssm_workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    import ssm_linear_attention_gb300 as ssm
    # batch 64 x 128 heads x L 16: 1.2 MB of tables; desynchronised write_pos and a
    # forced flush rate so both calls contain flush rows
    wl = W.mamba2_large(batch=64, num_slots=128, steps=2, force_rate=0.3)
    ref = Hn.make_mamba2_decoder(wl, out_dtype=torch.float32)
    new = Hn.make_mamba2_decoder(wl, out_dtype=torch.float32)
    assert torch.equal(ref.state, new.state)
    dims = new.dims(wl.batch)
    assert ssm.rssm_mamba2_workspace_size(dims) <= ssm.RSSM_NOALLOC_WORKSPACE_BYTES
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    tol = Hn.tol_for(wl.state_dtype)
    for t in range(2):
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(t))
        force = Hn.to_dev(wl.force_mask(t), torch.uint8)
        ref.advance(ci, force)
        ref.append(x, dt, Bm, ci)
        y_ref = torch.full((wl.batch, wl.nheads, wl.headdim), float("nan"), device="cuda")
        ssm.rssm_mamba2_decode(dims, ref.state, ref.A, C, ref.D, z, ref.ring_x, ref.ring_dt,
                               ref.ring_B, ci, ref.row_wp, ref.row_flush, ref.workspace,
                               ref.ws_bytes, y_ref, ref.dev_err)
        new.advance(ci, force)
        new.append(x, dt, Bm, ci)
        y_new = torch.full_like(y_ref, float("nan"))
        ssm.rssm_mamba2_decode_noalloc(dims, new.state, new.A, C, new.D, z, new.ring_x,
                                       new.ring_dt, new.ring_B, ci, new.row_wp, new.row_flush,
                                       y_new, new.dev_err)
        torch.cuda.synchronize()
        assert torch.equal(ref.row_wp, new.row_wp) and torch.equal(ref.row_flush, new.row_flush)
        assert int(new.row_flush[: wl.batch].sum()) > 0
        assert Hn.err(y_new.cpu().numpy(), y_ref.cpu().numpy()) <= tol, "call %d" % t
        ok, e, _ = Hn.state_ok(new.state.float().cpu().numpy(), ref.state.float().cpu().numpy(),
                               wl.state_dtype)
        assert ok, "call %d: flushed state differs (%.3g)" % (t, e)
    assert int(new.dev_err.abs().sum()) == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    import ssm_linear_attention_gb300 as ssm
    # 4096 rows x 128 heads x L 16 needs 72 MiB of tables, beyond the 16 MiB array
    dims = ssm.Mamba2Dims(4096, 128, 64, 128, 8, 16, 8192, ssm.RSSM_BF16, ssm.RSSM_BF16,
                          ssm.RSSM_BF16)
    assert ssm.rssm_mamba2_workspace_size(dims) > ssm.RSSM_NOALLOC_WORKSPACE_BYTES
    fake = 0x10000
    rc = ssm.lib().rssm_mamba2_decode_noalloc(
        __import__("ctypes").byref(dims), fake, fake, fake, fake, None, fake, fake, fake, fake,
        fake, fake, fake, None, None)
    assert rc == ssm.RSSM_ERR_UNSUPPORTED
