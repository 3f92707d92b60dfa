"""GPU tests of the slot fork (rssm_copy_slots; "GDN ReplaySSM decode (Part A of RFC
28511)", 实现拆解 item 3 and 评论区精华: copy_from carries the rings and cursors).

A fork taken in the middle of a ring (live entries, no flush) must continue exactly
as its source: the copied records are byte-identical, and a step that feeds the
same inputs to the source rows and to their forks in one batch gives bit-identical
outputs for each pair, which also agree with the oracle continuing the source."""
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


def _dup(inp):
    return {k: (None if v is None else np.concatenate([v, v])) for k, v in inp.items()}


def _i32(a):
    return Hn.to_dev(np.asarray(a, dtype=np.int32), torch.int32)


def _free_slots(wl, n):
    return np.setdiff1d(np.arange(wl.num_slots), wl.cache_indices())[:n].astype(np.int32)


def test_mamba2_fork_continues_like_source():
    wl = W.mamba2_large(batch=12, nheads=8, ngroups=2, num_slots=40, L=8, steps=3)
    dec = Hn.make_mamba2_decoder(wl, max_batch=2 * wl.batch)
    ci = wl.cache_indices()
    for j in range(wl.max_history()):
        dec.step(*Hn.mamba2_inputs_dev(wl, wl.history_inputs(j)), _i32(wl.history_ci(j)))
    for t in range(2):
        dec.step(*Hn.mamba2_inputs_dev(wl, wl.step_inputs(t)), _i32(ci))
    torch.cuda.synchronize()
    assert int(dec.slot_wp[torch.as_tensor(ci.astype(np.int64), device="cuda")].max()) > 0
    free = _free_slots(wl, wl.batch)
    dec.copy_slots(_i32(ci), _i32(free))
    torch.cuda.synchronize()
    src = torch.as_tensor(ci.astype(np.int64), device="cuda")
    dst = torch.as_tensor(free.astype(np.int64), device="cuda")
    for buf in (dec.state, dec.ring_x, dec.ring_dt, dec.ring_B, dec.slot_wp):
        assert torch.equal(buf[dst], buf[src])
    y = dec.step(*Hn.mamba2_inputs_dev(wl, _dup(wl.step_inputs(2))),
                 _i32(np.concatenate([ci, free])))
    torch.cuda.synchronize()
    b = wl.batch
    assert torch.equal(y[:b], y[b:2 * b])
    ref = oracle.mamba2_run(wl, steps=3)
    assert Hn.err(y[:b].float().cpu().numpy(), ref["y"][2]) <= Hn.tol_for(wl.state_dtype)
    assert int(dec.dev_err.abs().sum()) == 0


def test_fork_padding_bad_slots_and_self_copy():
    import ssm_linear_attention_gb300 as ssm
    wl = W.mamba2_large(batch=4, nheads=8, ngroups=2, num_slots=16, L=4, steps=1,
                        wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl)
    ci = wl.cache_indices()
    free = _free_slots(wl, 3)
    before = dec.state.clone()
    src = _i32([ci[0], -1, ci[2], ci[3], ci[1]])
    dst = _i32([free[0], free[1], -1, wl.num_slots + 2, ci[1]])
    dec.copy_slots(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(dec.state[int(free[0])], dec.state[int(ci[0])])
    for s in range(wl.num_slots):     # padding, bad and self pairs wrote nothing
        if s != int(free[0]):
            assert torch.equal(dec.state[s], before[s]), s
    assert int(dec.dev_err[0].item()) & ssm.RSSM_DEVERR_SLOT
    # n = 0 is a no-op
    dec.copy_slots(_i32([]), _i32([]))


def test_gdn_fork_continues_like_source():
    wl = W.gdn_decode(batch=8, num_v_heads=8, num_k_heads=4, num_slots=24, L=8, steps=3,
                      wp_mode="uniform")
    dec = Hn.make_gdn_decoder(wl, max_batch=2 * wl.batch)
    ci = wl.cache_indices()
    for j in range(wl.max_history()):
        dec.step(*Hn.gdn_inputs_dev(wl, wl.history_inputs(j)), _i32(wl.history_ci(j)))
    for t in range(2):
        dec.step(*Hn.gdn_inputs_dev(wl, wl.step_inputs(t)), _i32(ci))
    free = _free_slots(wl, wl.batch)
    dec.copy_slots(_i32(ci), _i32(free))
    torch.cuda.synchronize()
    src = torch.as_tensor(ci.astype(np.int64), device="cuda")
    dst = torch.as_tensor(free.astype(np.int64), device="cuda")
    for buf in (dec.state, dec.ring_d, dec.ring_k, dec.ring_g, dec.slot_wp):
        assert torch.equal(buf[dst], buf[src])
    o = dec.step(*Hn.gdn_inputs_dev(wl, _dup(wl.step_inputs(2))),
                 _i32(np.concatenate([ci, free])))
    torch.cuda.synchronize()
    b = wl.batch
    assert torch.equal(o[:b], o[b:2 * b])
    ref = oracle.gdn_run(wl, steps=3)
    assert Hn.err(o[:b].float().cpu().numpy(), ref["o"][2]) <= 1e-4


def test_spec_fork_continues_like_source():
    from ssm_linear_attention_gb300 import GDNSpecVerifier
    wl = W.gdn_spec(batch=8, num_v_heads=8, num_k_heads=4, num_slots=24, L=8, T=3, rounds=4)
    ver = GDNSpecVerifier(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.L,
                          wl.T, wl.num_slots, 2 * wl.batch, act_dtype=torch.bfloat16,
                          out_dtype=torch.float32)
    ci = wl.cache_indices()
    for s in ci:
        ver.state[int(s)] = Hn.to_dev(wl.slot_state(int(s)), torch.float32)
    ci_d = _i32(ci)
    for r in range(3):
        ver.verify(*Hn.gdn_inputs_dev(wl, wl.round_inputs(r)), ci_d)
        ver.commit(ci_d, _i32(wl.accepted(r)))
    free = _free_slots(wl, wl.batch)
    ver.copy_slots(ci_d, _i32(free))
    torch.cuda.synchronize()
    src = torch.as_tensor(ci.astype(np.int64), device="cuda")
    dst = torch.as_tensor(free.astype(np.int64), device="cuda")
    for buf in (ver.state, ver.ring_d, ver.ring_k, ver.ring_g, ver.ring_v, ver.ring_beta,
                ver.slot_cnt, ver.slot_base, ver.slot_flush):
        assert torch.equal(buf[dst], buf[src])
    both = _i32(np.concatenate([ci, free]))
    o = ver.verify(*Hn.gdn_inputs_dev(wl, _dup(wl.round_inputs(3))), both)
    ver.commit(both, _i32(np.concatenate([wl.accepted(3), wl.accepted(3)])))
    torch.cuda.synchronize()
    b = wl.batch
    assert torch.equal(o[:b], o[b:2 * b])
    for buf in (ver.slot_cnt, ver.slot_base, ver.slot_flush):
        assert torch.equal(buf[dst], buf[src])
    ref = oracle.gdn_spec_run(wl, rounds=4)
    assert Hn.err(o[:b].float().cpu().numpy(), ref["o"][3]) <= 1e-4
