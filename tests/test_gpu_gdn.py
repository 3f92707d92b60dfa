"""GPU parity: gated-delta-net ReplaySSM decode, full-state decode and speculative
verify vs the oracle (fp32 state: e <= 1e-4; cursors bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import rssm_workloads as W
from oracle import cursors
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def _gdn_cursor_ref(wl, steps):
    slot_wp = [0] * wl.num_slots
    for j in range(wl.max_history()):
        cursors.advance_standard(slot_wp, wl.history_ci(j), None, wl.L)
    wps, fls = [], []
    for t in range(steps):
        rw, rf = cursors.advance_standard(slot_wp, wl.cache_indices(), wl.force_mask(t), wl.L)
        wps.append(rw)
        fls.append(rf)
    return np.array(wps), np.array(fls)


def _check_gdn(wl, rows, steps, out_dtype=torch.float32, chunk=128):
    """Run the GPU path once for `rows`, then the oracle chunk by chunk of rows, and
    compare every output of every step and every stored checkpoint."""
    rows = np.asarray(rows)
    g = Hn.run_gpu_gdn(wl, steps=steps, out_dtype=out_dtype, rows=rows)
    cw, cf = _gdn_cursor_ref(wl, steps)
    assert np.array_equal(g["row_wp"], cw) and np.array_equal(g["row_flush"], cf)
    ci = wl.cache_indices()
    for c0, sub in Hn.row_chunks(rows, chunk):
        ref = oracle.gdn_run(wl, rows=sub, steps=steps, mode="replay")
        sl = slice(c0, c0 + len(sub))
        for t in range(steps):
            ro, go = ref["o"][t], g["o"][t][sl]
            if out_dtype == torch.bfloat16:
                d = np.abs(go - ro)
                assert np.all(d <= TOL * np.maximum(1, np.abs(ro)) + Hn.bf16_spacing(ro)), \
                    "step %d rows %d..: bf16 output off by more than tol + 1 spacing" % (t, c0)
            else:
                e = Hn.err(go, ro)
                assert e <= TOL, "step %d rows %d..: o error %.3g" % (t, c0, e)
        st = g["dec"].state[torch.as_tensor(ci[sub].astype(np.int64), device="cuda")].cpu().numpy()
        ok, e, _ = Hn.state_ok(st, ref["ckpt"], "fp32")
        assert ok, "rows %d..: checkpoint error %.3g" % (c0, e)
        del ref, st
    assert int(g["dec"].dev_err.abs().sum()) == 0


def test_gdn_small_desync_with_forced_flushes():
    wl = W.gdn_decode(batch=6, num_v_heads=4, num_k_heads=2, num_slots=12, L=4, steps=14,
                      wp_mode="uniform", force_rate=0.15)
    _check_gdn(wl, rows=np.arange(6), steps=14)


def test_gdn_decode_config_all_rows():
    # batch 256, HV 32, HK 16, K = V = 128, L 16, 64 steps, fp32 state N(0, 0.05): every
    # row's output at every step (four flushes per row) and every stored checkpoint
    wl = W.gdn_decode()
    _check_gdn(wl, rows=np.arange(wl.batch), steps=wl.steps)


def test_gdn_decode_bf16_output_desync():
    wl = W.gdn_decode(batch=64, num_slots=128, steps=20, wp_mode="uniform")
    _check_gdn(wl, rows=np.arange(wl.batch), steps=20, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("L", [1, 2, 8])
def test_gdn_ring_lengths_and_v256(L):
    wl = W.gdn_decode(batch=5, num_v_heads=4, num_k_heads=4, head_v_dim=256, num_slots=9, L=L,
                      steps=10, wp_mode="uniform", act_dtype="fp32")
    _check_gdn(wl, rows=np.arange(5), steps=10)


def test_gdn_full_state_kernel():
    wl = W.gdn_decode(batch=12, num_slots=20, steps=6)
    g = Hn.run_gpu_gdn(wl, steps=6, full_state=True)
    ref = oracle.gdn_run(wl, steps=6, mode="full")
    for t in range(6):
        assert Hn.err(g["o"][t], ref["o"][t]) <= TOL
    ci = wl.cache_indices()
    st = g["dec"].state[torch.as_tensor(ci.astype(np.int64), device="cuda")].cpu().numpy()
    assert Hn.state_ok(st, ref["ckpt"], "fp32")[0]


def _check_spec(wl, rows, rounds, chunk=128):
    rows = np.asarray(rows)
    g = Hn.run_gpu_spec(wl, rounds=rounds, rows=rows)
    # cursors: bit-exact against the integer model for every row
    cnt, base, fl = [0] * wl.num_slots, [0] * wl.num_slots, [0] * wl.num_slots
    ci = wl.cache_indices()
    folds = 0
    for r in range(rounds + 1):
        assert np.array_equal(g["cnt"][r], [cnt[s] for s in ci]), r
        assert np.array_equal(g["base"][r], [base[s] for s in ci]), r
        assert np.array_equal(g["flush"][r], [fl[s] for s in ci]), r
        if r < rounds:
            folds += int(np.count_nonzero(g["flush"][r][rows]))
            cursors.spec_commit(cnt, base, fl, ci, wl.accepted(r), wl.L, wl.T)
    # an exact fold ran for the compared rows, so the stored checkpoints were rewritten
    assert folds > 0, "no fold among the compared rows"
    worst = 0.0
    for c0, sub in Hn.row_chunks(rows, chunk):
        ref = oracle.gdn_spec_run(wl, rows=sub, rounds=rounds)
        sl = slice(c0, c0 + len(sub))
        for r in range(rounds):
            e = Hn.err(g["o"][r][sl], ref["o"][r])
            worst = max(worst, e)
            assert e <= TOL, "round %d rows %d..: draft output error %.3g" % (r, c0, e)
        st = g["ver"].state[torch.as_tensor(ci[sub].astype(np.int64), device="cuda")].cpu().numpy()
        ok, e, _ = Hn.state_ok(st, ref["ckpt"], "fp32")
        assert ok, "rows %d..: folded checkpoint error %.3g" % (c0, e)
        del ref, st
    assert int(g["ver"].dev_err.abs().sum()) == 0
    return worst


def test_spec_small_all_rows():
    wl = W.gdn_spec(batch=5, num_v_heads=4, num_k_heads=2, num_slots=10, L=8, T=4, rounds=16)
    _check_spec(wl, rows=np.arange(5), rounds=16)


@pytest.mark.parametrize("T,L", [(1, 2), (2, 5), (3, 8), (5, 10), (6, 13), (7, 15), (8, 16)])
def test_spec_draft_lengths(T, L):
    wl = W.gdn_spec(batch=4, num_v_heads=2, num_k_heads=1, num_slots=8, L=L, T=T, rounds=12,
                    act_dtype="fp32")
    _check_spec(wl, rows=np.arange(4), rounds=12)


@pytest.mark.parametrize("T,L,adt,rounds", [(4, 24, "bf16", 22), (8, 32, "fp32", 16)])
def test_spec_long_rings(T, L, adt, rounds):
    # more than 16 committed entries: the fold stages them in two chunks and the table
    # CTAs read the history keys past the ones they hold in registers
    wl = W.gdn_spec(batch=4, num_v_heads=4, num_k_heads=2, num_slots=8, L=L, T=T, rounds=rounds,
                    act_dtype=adt)
    _check_spec(wl, rows=np.arange(4), rounds=rounds)


def test_spec_config_all_rows():
    # batch 128, T 4, HV 32, HK 16, K = V = 128, L 16, 32 rounds, accepted ~ U{0..4}:
    # every row's draft outputs in every round and every folded checkpoint
    wl = W.gdn_spec()
    _check_spec(wl, rows=np.arange(wl.batch), rounds=wl.rounds)


def test_spec_rejects_short_ring():
    import ssm_linear_attention_gb300 as ssm
    wl = W.gdn_spec(batch=2, num_v_heads=2, num_k_heads=1, num_slots=4, L=7, T=4, rounds=1)
    with pytest.raises(ssm.RSSMError) as ei:
        Hn.run_gpu_spec(wl, rounds=1)
    assert ei.value.status == ssm.RSSM_ERR_CONFIG


@pytest.mark.parametrize("T,L", [(4, 16), (2, 5), (8, 16)])
def test_spec_full_state_baseline_matches_oracle(T, L):
    # the conventional verify: per-draft outputs equal the recurrence, and after each
    # commit the slot holds the state after the accepted prefix
    from ssm_linear_attention_gb300 import GDNSpecFullStateVerifier
    wl = W.gdn_spec(batch=5, num_v_heads=4, num_k_heads=2, num_slots=10, L=L, T=T, rounds=9)
    ad = Hn.torch_dt(wl.act_dtype)
    ver = GDNSpecFullStateVerifier(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim,
                                   T, wl.num_slots, wl.batch, act_dtype=ad,
                                   out_dtype=torch.float32)
    ci = wl.cache_indices()
    for s in ci:
        ver.state[int(s)] = Hn.to_dev(wl.slot_state(int(s)), torch.float32)
    ci_d = Hn.to_dev(ci, torch.int32)
    ref = oracle.gdn_spec_run(wl, rounds=wl.rounds)
    for r in range(wl.rounds):
        inp = wl.round_inputs(r)
        o = ver.verify(Hn.to_dev(inp["q"], ad), Hn.to_dev(inp["k"], ad), Hn.to_dev(inp["v"], ad),
                       Hn.to_dev(inp["beta"], torch.float32), Hn.to_dev(inp["g"], torch.float32),
                       ci_d)
        e = Hn.err(o.cpu().numpy(), ref["o"][r])
        assert e <= TOL, "round %d: %.3g" % (r, e)
        ver.commit(ci_d, Hn.to_dev(wl.accepted(r), torch.int32))
    torch.cuda.synchronize()
    st = ver.state[torch.as_tensor(ci.astype(np.int64), device="cuda")].cpu().numpy()
    assert Hn.err(st, ref["state"]) <= TOL
    assert int(ver.dev_err.abs().sum()) == 0
