"""GPU parity: cursor kernel and Mamba2 ReplaySSM / full-state kernels vs the oracle.

All calls go through the C ABI (ctypes binding). Tolerances: cursors bit-exact;
outputs and flushed states e <= 1e-4 (fp32 state) / 2e-3 (bf16 state), see
harness.py for the metric."""
import numpy as np
import pytest
import torch

import oracle
import rssm_workloads as W
from oracle import cursors
from tests import harness as Hn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def _dev(a, dt):
    return Hn.to_dev(a, dt)


# --------------------------------------------------------------------------- #
# cursors                                                                     #
# --------------------------------------------------------------------------- #

def test_cursor_standard_matches_model():
    import ssm_linear_attention_gb300 as ssm
    r = np.random.default_rng(0)
    for L in (1, 2, 5, 16):
        num_slots, batch = 300, 257
        slot_wp = r.integers(0, L, num_slots).astype(np.int32)
        ci = r.permutation(num_slots)[:batch].astype(np.int32)
        ci[r.random(batch) < 0.1] = -1
        d_slot = _dev(slot_wp, torch.int32)
        d_ci = _dev(ci, torch.int32)
        row_wp = torch.full((batch,), 77, dtype=torch.int32, device="cuda")
        row_fl = torch.full((batch,), 9, dtype=torch.uint8, device="cuda")
        model = list(slot_wp)
        for step in range(3 * L + 1):
            force = (r.random(batch) < 0.2).astype(np.uint8) if step % 2 else None
            ssm.rssm_advance_cursors(ssm.RSSM_CURSOR_STANDARD, d_slot, None, None, d_ci,
                                     None if force is None else _dev(force, torch.uint8), None,
                                     batch, num_slots, L, 0, row_wp, row_fl)
            rw, rf = cursors.advance_standard(model, ci, force, L)
            assert np.array_equal(row_wp.cpu().numpy(), rw)
            assert np.array_equal(row_fl.cpu().numpy(), rf)
            assert np.array_equal(d_slot.cpu().numpy(), model)


def test_cursor_spec_commit_and_reset_match_model():
    import ssm_linear_attention_gb300 as ssm
    r = np.random.default_rng(1)
    L, T, num_slots, batch = 16, 4, 64, 40
    ci = r.permutation(num_slots)[:batch].astype(np.int32)
    cnt, base, fl = [0] * num_slots, [0] * num_slots, [0] * num_slots
    d_cnt = torch.zeros(num_slots, dtype=torch.int32, device="cuda")
    d_base = torch.zeros(num_slots, dtype=torch.int32, device="cuda")
    d_fl = torch.zeros(num_slots, dtype=torch.uint8, device="cuda")
    row_c = torch.zeros(batch, dtype=torch.int32, device="cuda")
    row_f = torch.zeros(batch, dtype=torch.uint8, device="cuda")
    d_ci = _dev(ci, torch.int32)
    for rnd in range(60):
        acc = r.integers(0, T + 1, batch).astype(np.int32)
        ssm.rssm_advance_cursors(ssm.RSSM_CURSOR_SPEC_COMMIT, d_cnt, d_base, d_fl, d_ci, None,
                                 _dev(acc, torch.int32), batch, num_slots, L, T, row_c, row_f)
        cursors.spec_commit(cnt, base, fl, ci, acc, L, T)
        assert np.array_equal(d_cnt.cpu().numpy(), cnt)
        assert np.array_equal(d_base.cpu().numpy(), base)
        assert np.array_equal(d_fl.cpu().numpy(), fl)
        assert np.array_equal(row_c.cpu().numpy(), [cnt[s] for s in ci])
        if rnd % 7 == 3:
            sl = ci[:5].copy()
            ssm.rssm_advance_cursors(ssm.RSSM_CURSOR_RESET, d_cnt, d_base, d_fl,
                                     _dev(sl, torch.int32), None, None, 5, num_slots, L, T, None,
                                     None)
            cursors.spec_reset(cnt, base, fl, sl)


# --------------------------------------------------------------------------- #
# Mamba2 ReplaySSM                                                            #
# --------------------------------------------------------------------------- #

def _check_mamba2(wl, rows, steps, out_dtype=torch.float32, y_tol=None, chunk=128):
    """Run the GPU path once for `rows`, then the oracle chunk by chunk of rows, and
    compare every output of every step and every stored checkpoint."""
    rows = np.asarray(rows)
    g = Hn.run_gpu_mamba2(wl, steps=steps, out_dtype=out_dtype, rows=rows)
    # cursors: bit-exact for every row
    cw, cf, _ = Hn.cursor_reference(wl, steps)
    assert np.array_equal(g["row_wp"], cw)
    assert np.array_equal(g["row_flush"], cf)
    tol = Hn.tol_for(wl.state_dtype) if y_tol is None else y_tol
    ci = wl.cache_indices()
    worst, flips, n_el = 0.0, 0, 0
    for c0, sub in Hn.row_chunks(rows, chunk):
        ref = oracle.mamba2_run(wl, rows=sub, steps=steps, mode="replay")
        sl = slice(c0, c0 + len(sub))
        for t in range(steps):
            ry, gy = ref["y"][t], g["y"][t][sl]
            if out_dtype == torch.bfloat16:
                # the output store itself rounds to bf16: allow one bf16 spacing on top
                d = np.abs(gy - ry)
                lim = tol * np.maximum(1, np.abs(ry)) + Hn.bf16_spacing(ry)
                assert np.all(d <= lim), \
                    "step %d rows %d..: bf16 output off by more than tol + 1 spacing" % (t, c0)
            else:
                e = Hn.err(gy, ry)
                worst = max(worst, e)
                assert e <= tol, "step %d rows %d..: y error %.3g > %.3g" % (t, c0, e, tol)
        # checkpoints (the pool content)
        st = g["dec"].state[torch.as_tensor(ci[sub].astype(np.int64), device="cuda")] \
            .float().cpu().numpy()
        ok, e, fl = Hn.state_ok(st, ref["ckpt"], wl.state_dtype)
        assert ok, "rows %d..: checkpoint error %.3g (flips %d)" % (c0, e, fl)
        flips += fl
        n_el += st.size
        del ref, st
    frac = flips / max(1, n_el)
    assert frac < 1e-3, "too many one-spacing disagreements: %g" % frac
    assert int(g["dec"].dev_err.abs().sum()) == 0
    return worst


def test_mamba2_tiny_config_all_rows():
    wl = W.mamba2_tiny()
    _check_mamba2(wl, rows=np.arange(wl.batch), steps=wl.steps)


def test_mamba2_large_config_all_rows():
    # batch 512, H 128, P 64, N 128, G 8, L 16, bf16 state, 1024 slots, desync write_pos:
    # every row's output at every step and every row's stored checkpoint
    wl = W.mamba2_large()
    _check_mamba2(wl, rows=np.arange(wl.batch), steps=wl.steps)


def test_mamba2_large_config_bf16_output_all_rows():
    wl = W.mamba2_large()
    _check_mamba2(wl, rows=np.arange(wl.batch), steps=20, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("batch,L,sdt", [(16, 1, "bf16"), (64, 4, "fp32"), (37, 8, "bf16"),
                                         (128, 16, "fp32"), (1, 16, "bf16")])
def test_mamba2_sweep_points(batch, L, sdt):
    wl = W.mamba2_sweep(batch, L, sdt, steps=12)
    _check_mamba2(wl, rows=np.arange(batch), steps=12)


@pytest.mark.parametrize("P,N", [(128, 128), (64, 64), (128, 64)])
@pytest.mark.parametrize("sdt", ["fp32", "bf16"])
def test_mamba2_other_tile_shapes(P, N, sdt):
    wl = W.mamba2_large(batch=9, nheads=8, ngroups=2, headdim=P, dstate=N, num_slots=20, L=4,
                        steps=10, state_dtype=sdt, force_rate=0.1)
    _check_mamba2(wl, rows=np.arange(9), steps=10)


def test_mamba2_no_gate_and_fp32_activations():
    wl = W.mamba2_large(batch=6, nheads=16, ngroups=4, num_slots=12, L=5, steps=9,
                        state_dtype="fp32", act_dtype="fp32", with_z=False)
    _check_mamba2(wl, rows=np.arange(6), steps=9)


# --------------------------------------------------------------------------- #
# Mamba2 full-state kernel                                                    #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("wl", [W.mamba2_tiny(),
                                W.mamba2_large(batch=24, num_slots=64, steps=6),
                                W.mamba2_large(batch=5, nheads=8, ngroups=2, headdim=128,
                                               dstate=64, num_slots=8, steps=5,
                                               state_dtype="fp32")],
                         ids=["tiny", "large_geom", "p128n64"])
def test_mamba2_full_state_kernel(wl):
    steps = wl.steps
    rows = np.arange(wl.batch)
    g = Hn.run_gpu_mamba2(wl, steps=steps, full_state=True)
    ref = oracle.mamba2_run(wl, rows=rows, steps=steps, mode="full")
    tol = Hn.tol_for(wl.state_dtype)
    for t in range(steps):
        assert Hn.err(g["y"][t], ref["y"][t]) <= tol
    ci = wl.cache_indices()
    st = g["dec"].state[torch.as_tensor(ci.astype(np.int64), device="cuda")].float().cpu().numpy()
    ok, e, flips = Hn.state_ok(st, ref["ckpt"], wl.state_dtype)
    assert ok, (e, flips)


# --------------------------------------------------------------------------- #
# edge cases                                                                  #
# --------------------------------------------------------------------------- #

def test_padding_rows_are_untouched_and_bad_slots_flagged():
    import ssm_linear_attention_gb300 as ssm
    wl = W.mamba2_large(batch=8, nheads=8, ngroups=2, num_slots=16, L=4, steps=3, wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl)
    ci = wl.cache_indices().copy()
    ci[2] = -1
    ci[5] = wl.num_slots + 3          # out of range: skipped, flagged
    before = dec.state.clone()
    inp = wl.step_inputs(0)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, inp)
    y = torch.full((8, wl.nheads, wl.headdim), 123.0, device="cuda")
    dec.step(x, dt, Bm, C, z, Hn.to_dev(ci, torch.int32), y=y)
    torch.cuda.synchronize()
    assert torch.all(y[2] == 123.0) and torch.all(y[5] == 123.0)
    assert int(dec.dev_err[0].item()) & ssm.RSSM_DEVERR_SLOT
    # the valid rows agree with the oracle
    ref = oracle.mamba2_run(wl, rows=[0, 1, 3], steps=1)
    assert Hn.err(y[[0, 1, 3]].cpu().numpy(), ref["y"][0]) <= 2e-3
    # no slot other than the valid rows' was written (no flush at w = 0 with L = 4)
    assert torch.equal(dec.state, before)


def test_small_batch_bad_cursor_is_flagged_and_skipped():
    # the one-launch step (batch <= 16) reads the cursor itself: a slot whose write_pos is
    # outside the ring is skipped (its output, state and cursor untouched) and flagged,
    # while the other rows advance as usual
    import ssm_linear_attention_gb300 as ssm
    wl = W.mamba2_large(batch=6, nheads=8, ngroups=2, num_slots=12, L=4, steps=1, wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl)
    ci = wl.cache_indices()
    bad = int(ci[3])
    dec.slot_wp[bad] = wl.L + 2
    before = dec.state.clone()
    inp = wl.step_inputs(0)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, inp)
    y = torch.full((6, wl.nheads, wl.headdim), 7.0, device="cuda")
    dec.step(x, dt, Bm, C, z, Hn.to_dev(ci, torch.int32), y=y)
    torch.cuda.synchronize()
    assert int(dec.dev_err[0].item()) & ssm.RSSM_DEVERR_CURSOR
    assert torch.all(y[3] == 7.0)
    assert int(dec.slot_wp[bad].item()) == wl.L + 2
    assert torch.equal(dec.state, before)  # write_pos 0, L 4: no row flushes
    for r in (0, 1, 2, 4, 5):
        assert int(dec.slot_wp[int(ci[r])].item()) == 1
    ref = oracle.mamba2_run(wl, rows=[0, 1, 2, 4, 5], steps=1)
    assert Hn.err(y[[0, 1, 2, 4, 5]].cpu().numpy(), ref["y"][0]) <= 2e-3


def test_desync_rows_are_independent():
    # Permuting the rows of a batch changes no row's output bit (no cross-row coupling).
    wl = W.mamba2_large(batch=48, num_slots=96, steps=6, force_rate=0.1)
    a = Hn.run_gpu_mamba2(wl, steps=6, rows=np.arange(48))
    perm = np.random.default_rng(5).permutation(48)

    class Permuted(W.Mamba2Workload):
        pass

    wp = W.mamba2_large(batch=48, num_slots=96, steps=6, force_rate=0.1)
    base_ci, base_h = wl.cache_indices(), wl.history_len()
    wp._cache["ci"] = base_ci[perm].copy()
    wp._cache["wp"] = base_h[perm].copy()
    wp._cache["params"] = wl.params()
    orig_step, orig_hist, orig_force = wl.step_inputs, wl.history_inputs, wl.force_mask

    def permute(d):
        return {k: (None if v is None else v[perm]) for k, v in d.items()}

    wp.step_inputs = lambda t: permute(orig_step(t))
    wp.history_inputs = lambda j: permute(orig_hist(j))
    wp.force_mask = lambda t: orig_force(t)[perm]
    b = Hn.run_gpu_mamba2(wp, steps=6, rows=np.arange(48))
    for t in range(6):
        assert np.array_equal(a["y"][t][perm], b["y"][t])


def test_batch_zero_is_a_no_op():
    import ssm_linear_attention_gb300 as ssm
    wl = W.mamba2_tiny()
    dec = Hn.make_mamba2_decoder(wl)
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    ssm.rssm_advance_cursors(ssm.RSSM_CURSOR_STANDARD, dec.slot_wp, None, None, e, None, None, 0,
                             wl.num_slots, wl.L, 0, dec.row_wp, dec.row_flush)
    ssm.rssm_mamba2_decode(dec.dims(0), dec.state, dec.A, dec.y, dec.D, None, dec.ring_x,
                           dec.ring_dt, dec.ring_B, e, dec.row_wp, dec.row_flush, dec.workspace,
                           dec.ws_bytes, dec.y)
    torch.cuda.synchronize()


@pytest.mark.parametrize("batch,L,sdt", [(16, 16, "bf16"), (1, 16, "fp32"), (7, 5, "bf16")])
def test_small_batch_step_matches_staged_calls(batch, L, sdt):
    # Batches of up to 16 rows run the whole step in one launch; the staged calls
    # (cursor, append, precompute, output) are the two-launch path. Cursors and ring
    # entries are copies and must be equal; outputs and flushed states agree within the
    # state dtype's bar (the tables' float32 sums run in a different order).
    wl = W.mamba2_large(batch=batch, num_slots=2 * batch + 3, L=L, steps=2 * L + 3,
                        state_dtype=sdt, force_rate=0.2)
    one = Hn.make_mamba2_decoder(wl)
    two = Hn.make_mamba2_decoder(wl)
    for j in range(wl.max_history()):
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.history_inputs(j))
        hci = Hn.to_dev(wl.history_ci(j), torch.int32)
        one.step(x, dt, Bm, C, z, hci)
        two.step_staged(x, dt, Bm, C, z, hci)
    ci = Hn.to_dev(wl.cache_indices(), torch.int32)
    tol = Hn.tol_for(sdt)
    for t in range(wl.steps):
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(t))
        f = Hn.to_dev(wl.force_mask(t), torch.uint8)
        ya = one.step(x, dt, Bm, C, z, ci, f).float().cpu().numpy()
        yb = two.step_staged(x, dt, Bm, C, z, ci, f).float().cpu().numpy()
        assert Hn.err(ya, yb) <= tol, t
        assert torch.equal(one.row_wp[:batch], two.row_wp[:batch])
        assert torch.equal(one.row_flush[:batch], two.row_flush[:batch])
    torch.cuda.synchronize()
    for name in ("ring_x", "ring_dt", "ring_B", "slot_wp"):
        assert torch.equal(getattr(one, name), getattr(two, name)), name
    ok, e, flips = Hn.state_ok(one.state.float().cpu().numpy(), two.state.float().cpu().numpy(), sdt)
    assert ok, (e, flips)
    assert int(one.dev_err.abs().sum()) == 0 and int(two.dev_err.abs().sum()) == 0
