"""GPU: the fused per-row prologue (cursor advance + ring append + tables in one
launch) gives bit-identical results to the separate calls.

The fused entry points run the same arithmetic in the same order as
rssm_advance_cursors -> ring append -> precompute, so every output element, ring
entry, checkpoint and cursor must be equal, not merely within tolerance. Parity of
the separate calls with the oracle is covered by the other GPU tests; the fused
step is also what the decoders' step() runs in those tests."""
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


def _mamba2_equal(a, b):
    for name in ("state", "ring_x", "ring_dt", "ring_B", "slot_wp"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("sdt,L", [("bf16", 16), ("fp32", 4), ("bf16", 1)])
def test_mamba2_fused_step_equals_staged_calls(sdt, L):
    wl = W.mamba2_large(batch=64, num_slots=128, steps=2 * L + 3, L=L, state_dtype=sdt,
                        force_rate=0.1)
    fused = Hn.make_mamba2_decoder(wl)
    staged = Hn.make_mamba2_decoder(wl)
    shared = Hn.make_mamba2_decoder(wl)   # advance by a separate call, then prepare(advance=False)
    for j in range(wl.max_history()):
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.history_inputs(j))
        hci = Hn.to_dev(wl.history_ci(j), torch.int32)
        fused.step(x, dt, Bm, C, z, hci)
        staged.step_staged(x, dt, Bm, C, z, hci)
        shared.advance(hci)
        shared.prepare(x, dt, Bm, C, hci, advance=False)
        shared.output(C, z, hci)
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    for t in range(wl.steps):
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(t))
        f = Hn.to_dev(wl.force_mask(t), torch.uint8)
        ya = fused.step(x, dt, Bm, C, z, ci, f).clone()
        yb = staged.step_staged(x, dt, Bm, C, z, ci, f).clone()
        shared.advance(ci, f)
        shared.prepare(x, dt, Bm, C, ci, advance=False)
        yc = shared.output(C, z, ci).clone()
        assert torch.equal(ya, yb) and torch.equal(ya, yc), t
        assert torch.equal(fused.row_wp, staged.row_wp)
        assert torch.equal(fused.row_flush, staged.row_flush)
    torch.cuda.synchronize()
    _mamba2_equal(fused, staged)
    _mamba2_equal(fused, shared)
    for d in (fused, staged, shared):
        assert int(d.dev_err.abs().sum()) == 0


def test_mamba2_fused_prologue_padding_and_bad_slots():
    import ssm_linear_attention_gb300 as ssm
    wl = W.mamba2_large(batch=8, nheads=8, ngroups=2, num_slots=16, L=4, steps=1, wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl)
    ci = wl.cache_indices().copy()
    ci[2] = -1
    ci[5] = wl.num_slots + 3
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(0))
    slot_before = dec.slot_wp.clone()
    ring_before = dec.ring_x.clone()
    dec.row_wp.fill_(7)
    dec.prepare(x, dt, Bm, C, Hn.to_dev(ci, torch.int32))
    torch.cuda.synchronize()
    assert int(dec.dev_err[0].item()) & ssm.RSSM_DEVERR_SLOT
    rw = dec.row_wp.cpu().numpy()
    assert rw[2] == 0 and rw[5] == 0          # padding / invalid rows get w = 0, no flush
    valid = [b for b in range(8) if b not in (2, 5)]
    moved = dec.slot_wp.cpu().numpy() - slot_before.cpu().numpy()
    assert sorted(np.nonzero(moved)[0].tolist()) == sorted(int(ci[b]) for b in valid)
    # only the valid rows' slots received a ring entry
    changed = torch.nonzero((dec.ring_x != ring_before).flatten(1).any(1)).flatten().tolist()
    assert sorted(changed) == sorted(int(ci[b]) for b in valid)


def _gdn_equal(a, b):
    for name in ("state", "ring_d", "ring_k", "ring_g", "slot_wp"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("L", [16, 3, 1])
def test_gdn_fused_step_equals_staged_calls(L):
    wl = W.gdn_decode(batch=32, num_slots=64, L=L, steps=2 * L + 3, wp_mode="uniform",
                      force_rate=0.1)
    fused = Hn.make_gdn_decoder(wl)
    staged = Hn.make_gdn_decoder(wl)
    shared = Hn.make_gdn_decoder(wl)
    for j in range(wl.max_history()):
        q, k, v, be, g = Hn.gdn_inputs_dev(wl, wl.history_inputs(j))
        hci = Hn.to_dev(wl.history_ci(j), torch.int32)
        fused.step(q, k, v, be, g, hci)
        staged.step_staged(q, k, v, be, g, hci)
        shared.advance(hci)
        shared.prepare(q, k, be, g, hci, advance=False)
        shared.output(q, v, hci)
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    for t in range(wl.steps):
        q, k, v, be, g = Hn.gdn_inputs_dev(wl, wl.step_inputs(t))
        f = Hn.to_dev(wl.force_mask(t), torch.uint8)
        oa = fused.step(q, k, v, be, g, ci, f).clone()
        ob = staged.step_staged(q, k, v, be, g, ci, f).clone()
        shared.advance(ci, f)
        shared.prepare(q, k, be, g, ci, advance=False)
        oc = shared.output(q, v, ci).clone()
        assert torch.equal(oa, ob) and torch.equal(oa, oc), t
        assert torch.equal(fused.row_flush, staged.row_flush)
    torch.cuda.synchronize()
    _gdn_equal(fused, staged)
    _gdn_equal(fused, shared)
    for d in (fused, staged, shared):
        assert int(d.dev_err.abs().sum()) == 0
