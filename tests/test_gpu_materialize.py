"""GPU: the materialize entry points return the recurrent state the oracle holds
after the same steps (checkpoint folded with the live ring entries), and leave the
pool, the rings and the cursors untouched.

Tolerances as the other parity tests: e <= 1e-4 for an fp32 checkpoint, 2e-3 for
a bf16 checkpoint (metric in harness.py)."""
import numpy as np
import pytest
import torch

import oracle
import rssm_workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def _snapshot(dec, names):
    return {n: getattr(dec, n).clone() for n in names}


@pytest.mark.parametrize("sdt", ["fp32", "bf16"])
def test_mamba2_materialize_matches_recurrence(sdt):
    wl = W.mamba2_large(batch=24, num_slots=48, nheads=16, ngroups=2, L=8, steps=11,
                        state_dtype=sdt, force_rate=0.1)
    g = Hn.run_gpu_mamba2(wl, steps=wl.steps)
    dec = g["dec"]
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    names = ("state", "ring_x", "ring_dt", "ring_B", "slot_wp")
    before = _snapshot(dec, names)
    out = dec.materialize(ci)
    torch.cuda.synchronize()
    for n in names:
        assert torch.equal(before[n], getattr(dec, n)), n
    ref = oracle.mamba2_run(wl, steps=wl.steps, keep_y=False)
    e = Hn.err(out.cpu().numpy(), ref["state"])
    assert e <= Hn.tol_for(sdt), e
    assert int(dec.dev_err.abs().sum()) == 0


def test_mamba2_materialize_skips_padding_and_flags_bad_slots():
    import ssm_linear_attention_gb300 as ssm
    wl = W.mamba2_tiny(steps=2)
    g = Hn.run_gpu_mamba2(wl, steps=2)
    dec = g["dec"]
    slots = torch.tensor([0, -1, wl.num_slots + 2, 3], dtype=torch.int32, device="cuda")
    out = torch.full((4, wl.nheads, wl.headdim, wl.dstate), 7.0, device="cuda")
    dec.materialize(slots, out=out)
    torch.cuda.synchronize()
    assert torch.all(out[1] == 7.0) and torch.all(out[2] == 7.0)
    assert int(dec.dev_err[0].item()) & ssm.RSSM_DEVERR_SLOT
    ref = oracle.mamba2_run(wl, steps=2, keep_y=False)
    assert Hn.err(out[[0, 3]].cpu().numpy(), ref["state"][[0, 3]]) <= 1e-4


def test_gdn_materialize_matches_recurrence():
    wl = W.gdn_decode(batch=12, num_slots=24, num_v_heads=4, num_k_heads=2, L=6, steps=9,
                      wp_mode="uniform", force_rate=0.1)
    g = Hn.run_gpu_gdn(wl, steps=wl.steps)
    dec = g["dec"]
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    names = ("state", "ring_d", "ring_k", "ring_g", "slot_wp")
    before = _snapshot(dec, names)
    out = dec.materialize(ci)
    torch.cuda.synchronize()
    for n in names:
        assert torch.equal(before[n], getattr(dec, n)), n
    ref = oracle.gdn_run(wl, steps=wl.steps, keep_o=False)
    e = Hn.err(out.cpu().numpy(), ref["state"])
    assert e <= 1e-4, e
    assert int(dec.dev_err.abs().sum()) == 0


@pytest.mark.parametrize("T,L,rounds", [(4, 8, 7), (2, 5, 9), (3, 16, 12)])
def test_spec_materialize_matches_recurrence(T, L, rounds):
    wl = W.gdn_spec(batch=6, num_v_heads=4, num_k_heads=2, num_slots=12, L=L, T=T, rounds=rounds)
    g = Hn.run_gpu_spec(wl, rounds=rounds)
    ver = g["ver"]
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    names = ("state", "ring_d", "ring_k", "ring_g", "slot_cnt", "slot_base", "slot_flush")
    before = _snapshot(ver, names)
    out = ver.materialize(ci)
    torch.cuda.synchronize()
    for n in names:
        assert torch.equal(before[n], getattr(ver, n)), n
    ref = oracle.gdn_spec_run(wl, rounds=rounds)
    e = Hn.err(out.cpu().numpy(), ref["state"])
    assert e <= 1e-4, e
    assert int(ver.dev_err.abs().sum()) == 0
