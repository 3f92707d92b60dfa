"""GPU parity of the stochastic rounding of the bf16 Mamba2 state ([M2] 评论区精华:
stochastic rounding for quantised models): the generator bit-exact against the
oracle's Philox4x32-10, the rounded states against the oracle's rounding of the
exact float64 state with the same bits, unbiasedness over many draws, and the
offset that moves on after every call (eagerly and in graph replays).

Tolerance: every stored value meets the bf16-state bar of the other parity tests
(within 2e-3 of the oracle relative to max(1, |ref|), or one bf16 spacing), and at
most 0.1 % of elements differ from the oracle's rounding at all. The kernel decides
from its float32 accumulation and the oracle from the float32 rounding of the exact
value; these differ by a few float32 spacings of the step's terms, so a decision
differs only where the random bits fall in that gap (measured: ~15 of 1M elements
per step; where the two terms of the update nearly cancel, the float32 error spans
several bf16 spacings of the tiny result, as it does with round-to-nearest). Bits
taken from the wrong counter or word would change about a third of the decisions."""
import numpy as np
import pytest
import torch

import oracle
import rssm_workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu

SEED = 0x5EED_0123_4567_89AB


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def _oracle_pool(wl):
    pool = np.zeros((wl.num_slots, wl.nheads, wl.headdim, wl.dstate))
    for s in wl.cache_indices():
        if s >= 0:
            pool[int(s)] = wl.slot_state(int(s))
    return pool


def _oracle_step(wl, pool, t):
    prm = wl.params()
    inp = wl.step_inputs(t)
    oracle.mamba2_step(pool, inp["x"], inp["dt_raw"], prm["A"], inp["B"], inp["C"], prm["D"],
                       inp["z"], prm["dt_bias"], wl.dt_softplus, ci=wl.cache_indices())


def _compare_sr(gpu, ref, max_flip=1e-3):
    gpu = np.asarray(gpu, dtype=np.float64)
    ok, e, flips = Hn.state_ok(gpu, ref, "bf16")
    assert ok, e
    frac = flips / max(gpu.size, 1)
    assert frac <= max_flip, frac
    return frac


def _slots_state(dec, wl):
    idx = torch.as_tensor(wl.cache_indices().astype(np.int64), device="cuda")
    return dec.state[idx].float().cpu().numpy()


def test_philox_fill_matches_oracle():
    import ssm_linear_attention_gb300 as ssm
    for seed, offset, n in ((0, 0, 1), (SEED, 7, 1000), (2 ** 64 - 1, 2 ** 40 + 3, 333)):
        out = torch.zeros(4 * n, device="cuda", dtype=torch.int32)
        ssm.rssm_philox4x32_fill(seed, offset, out, n)
        got = out.cpu().numpy().view(np.uint32).reshape(n, 4)
        for g in range(n):
            want = oracle.philox4x32_10(
                [g & 0xFFFFFFFF, g >> 32, offset & 0xFFFFFFFF, offset >> 32],
                [seed & 0xFFFFFFFF, seed >> 32])
            assert list(got[g]) == want, (seed, offset, g)


# Each step below starts from the workload's initial states (the decoder's pool is
# reset to them): a decision that differs at one step would otherwise move the next
# step's input by a bf16 spacing, which cancellation can turn into several spacings
# of the next result.

def test_full_state_sr_matches_oracle_and_advances():
    wl = W.mamba2_large(batch=16, nheads=8, ngroups=2, num_slots=40, L=4, steps=2,
                        wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl, full_state=True, sr_seed=SEED)
    ci_d = Hn.to_dev(wl.cache_indices(), torch.int32)
    init = dec.state.clone()
    for t in range(3):
        dec.state.copy_(init)
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(t))
        dec.step(x, dt, Bm, C, z, ci_d)
        torch.cuda.synchronize()
        pool = _oracle_pool(wl)
        _oracle_step(wl, pool, t)
        oracle.round_slots_sr(pool, wl.cache_indices(), SEED, t)
        _compare_sr(_slots_state(dec, wl), pool[wl.cache_indices()])
        assert int(dec.sr[1].item()) == t + 1


def test_replay_flush_sr_matches_oracle():
    # wp starts at 0 and every row is forced to flush: the fold of a one-entry ring is
    # one full-state step, so the stored state is SR(one step) at offsets 0, 1, 2
    wl = W.mamba2_large(batch=24, nheads=8, ngroups=2, num_slots=64, L=4, steps=3,
                        wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl, sr_seed=SEED)
    ci_d = Hn.to_dev(wl.cache_indices(), torch.int32)
    force = torch.ones(wl.batch, device="cuda", dtype=torch.uint8)
    init = dec.state.clone()
    for t in range(3):
        dec.state.copy_(init)
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(t))
        dec.step(x, dt, Bm, C, z, ci_d, force)
        torch.cuda.synchronize()
        assert int(dec.slot_wp.abs().sum().item()) == 0   # every row flushed at w = 0
        pool = _oracle_pool(wl)
        _oracle_step(wl, pool, t)
        oracle.round_slots_sr(pool, wl.cache_indices(), SEED, t)
        _compare_sr(_slots_state(dec, wl), pool[wl.cache_indices()])
    assert int(dec.sr[1].item()) == 3


def _boundary_window(exact, bound, seed, offset, elems):
    """For the listed pool elements: (distance of the float32 value of `exact` to the
    stochastic-rounding decision boundary its random bits set, allowed distance).
    Rounding goes away from zero iff (low 16 bits of the float32) + r >= 2^16, so the
    boundary sits (low + r - 2^16) float32 spacings from the value; the allowed
    distance is the float32 error of a fold of at most L + 2 fused terms of total
    magnitude `bound`, plus the float32 rounding of the exact value itself."""
    f = exact.astype(np.float32)
    u = f.view(np.uint32).astype(np.int64)
    lo = u & 0xFFFF
    r = np.array([oracle.sr_bits(seed, offset, int(e)) for e in elems], dtype=np.int64)
    ulp = np.spacing(np.abs(f)).astype(np.float64)
    dist = np.abs(lo + r - 65536).astype(np.float64) * ulp
    return dist, bound * 2.0 ** -24 + ulp


def test_replay_flush_sr_multi_entry_fold_matches_oracle():
    # Rows start with desynchronised write_pos w ~ U{0..7} (w history entries in the
    # ring, none of them flushing) and every row is forced to flush at the next step, so
    # each stored state is the stochastic rounding of a fold of w + 1 ring entries into
    # the checkpoint. Each element must equal the oracle's rounding of the exact state
    # with the same bits, or (where the float32 fold sits within its accumulation error
    # of the decision boundary) the neighbouring bf16 value.
    wl = W.mamba2_large(batch=32, nheads=8, ngroups=2, num_slots=64, L=8, steps=1)
    hist = wl.history_len()
    assert hist.max() >= 5 and np.count_nonzero(hist >= 1) >= 24
    dec = Hn.make_mamba2_decoder(wl, sr_seed=SEED)
    for j in range(wl.max_history()):
        x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.history_inputs(j))
        dec.step(x, dt, Bm, C, z, Hn.to_dev(wl.history_ci(j), torch.int32))
    torch.cuda.synchronize()
    off = int(dec.sr[1].item())
    ci = wl.cache_indices()
    ci_d = Hn.to_dev(ci, torch.int32)
    force = torch.ones(wl.batch, device="cuda", dtype=torch.uint8)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(0))
    dec.step(x, dt, Bm, C, z, ci_d, force)
    torch.cuda.synchronize()
    assert np.array_equal(dec.row_wp[: wl.batch].cpu().numpy(), hist)
    assert int(dec.row_flush[: wl.batch].sum()) == wl.batch
    gpu = _slots_state(dec, wl).astype(np.float64)

    # oracle: the exact state after the history and the step (no rounding before the
    # flush), rounded stochastically with the generator the flush launch used
    prm = wl.params()
    pool = _oracle_pool(wl)
    mag = np.abs(pool)

    def run(pool_, absolute):
        for j in range(wl.max_history() + 1):
            inp = wl.history_inputs(j) if j < wl.max_history() else wl.step_inputs(0)
            c = wl.history_ci(j) if j < wl.max_history() else ci
            xx = np.abs(inp["x"]) if absolute else inp["x"]
            bb = np.abs(inp["B"]) if absolute else inp["B"]
            oracle.mamba2_step(pool_, xx, inp["dt_raw"], prm["A"], bb, inp["C"], prm["D"],
                               inp["z"], prm["dt_bias"], wl.dt_softplus, ci=c)

    run(pool, False)
    run(mag, True)   # sum of the magnitudes of every term of each element's fold
    exact = pool[ci].copy()
    ref = pool.copy()
    oracle.round_slots_sr(ref, ci, SEED, off)
    ref = ref[ci]
    d = np.abs(gpu - ref)
    # the window is a small fraction of a bf16 spacing for almost every element, so
    # the boundary condition below constrains nearly all decisions
    win = (wl.L + 2) * mag[ci] * 2.0 ** -24 + np.spacing(np.abs(exact).astype(np.float32))
    assert np.mean(win < 0.5 * Hn.bf16_spacing(exact)) > 0.99
    diff = np.nonzero(d.ravel() > 0)[0]
    frac = diff.size / gpu.size
    assert frac <= 1e-3, frac
    if diff.size:
        per_slot = wl.nheads * wl.headdim * wl.dstate
        row = diff // per_slot
        elems = ci[row].astype(np.int64) * per_slot + diff % per_slot
        ex = exact.ravel()[diff]
        dist, allow = _boundary_window(ex, (wl.L + 2) * mag[ci].ravel()[diff], SEED, off, elems)
        g = gpu.ravel()[diff]
        # every stored value is a rounding of a value inside the fold's float32 window
        assert np.all(np.abs(g - ex) <= allow + Hn.bf16_spacing(np.abs(ex) + allow) * 1.0000001), \
            "a stored value is not a rounding of the exact state"
        # where the window is narrower than half a bf16 spacing (no cancellation), the two
        # roundings are neighbours and the decision differs only near its boundary
        narrow = allow < 0.5 * Hn.bf16_spacing(ex)
        assert np.all(d.ravel()[diff][narrow] <= Hn.bf16_spacing(ref.ravel()[diff][narrow]) *
                      1.0000001), "a stored value is not a bf16 neighbour"
        assert np.all(dist[narrow] <= allow[narrow]), \
            "a rounding decision differs away from its boundary"

    assert int(dec.dev_err.abs().sum()) == 0


def test_staged_output_sr_equals_fused_step_sr():
    wl = W.mamba2_large(batch=12, nheads=8, ngroups=2, num_slots=32, L=4, steps=1,
                        wp_mode="zero")
    a = Hn.make_mamba2_decoder(wl, sr_seed=SEED)
    b = Hn.make_mamba2_decoder(wl, sr_seed=SEED)
    ci_d = Hn.to_dev(wl.cache_indices(), torch.int32)
    force = torch.ones(wl.batch, device="cuda", dtype=torch.uint8)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(0))
    a.step(x, dt, Bm, C, z, ci_d, force)
    b.step_staged(x, dt, Bm, C, z, ci_d, force)
    torch.cuda.synchronize()
    assert torch.equal(a.state, b.state)
    assert torch.equal(a.sr, b.sr)


def test_sr_mean_converges_to_exact_state():
    wl = W.mamba2_large(batch=8, nheads=8, ngroups=2, num_slots=16, L=4, steps=1,
                        wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl, full_state=True, sr_seed=SEED)
    rne = Hn.make_mamba2_decoder(wl, full_state=True)
    ci_d = Hn.to_dev(wl.cache_indices(), torch.int32)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(0))
    init = dec.state.clone()
    T = 64
    acc = torch.zeros_like(dec.state, dtype=torch.float64)
    for _ in range(T):
        dec.state.copy_(init)
        dec.step(x, dt, Bm, C, z, ci_d)
        acc += dec.state.double()
    rne.step(x, dt, Bm, C, z, ci_d)
    torch.cuda.synchronize()
    pool = _oracle_pool(wl)
    _oracle_step(wl, pool, 0)
    ci = wl.cache_indices()
    exact = pool[ci]
    idx = torch.as_tensor(ci.astype(np.int64), device="cuda")
    mean = (acc[idx] / T).cpu().numpy()
    sp = Hn.bf16_spacing(exact)
    err_sr = float(np.mean(np.abs(mean - exact) / sp))
    err_rne = float(np.mean(np.abs(_slots_state(rne, wl) - exact) / sp))
    assert err_rne > 0.15, err_rne
    assert err_sr < 0.07, err_sr
    assert int(dec.sr[1].item()) == T


def test_sr_leaves_fp32_state_unchanged():
    wl = W.mamba2_large(batch=8, nheads=8, ngroups=2, num_slots=16, L=4, steps=1,
                        wp_mode="zero", state_dtype="fp32")
    a = Hn.make_mamba2_decoder(wl, full_state=True, sr_seed=SEED)
    b = Hn.make_mamba2_decoder(wl, full_state=True)
    ci_d = Hn.to_dev(wl.cache_indices(), torch.int32)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(0))
    ya = a.step(x, dt, Bm, C, z, ci_d).clone()
    yb = b.step(x, dt, Bm, C, z, ci_d).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.state, b.state) and torch.equal(ya, yb)
    assert int(a.sr[1].item()) == 1


def test_graph_replays_draw_fresh_bits():
    wl = W.mamba2_large(batch=16, nheads=8, ngroups=2, num_slots=32, L=4, steps=2,
                        wp_mode="zero")
    dec = Hn.make_mamba2_decoder(wl, sr_seed=SEED)
    ci_d = Hn.to_dev(wl.cache_indices(), torch.int32)
    force = torch.ones(wl.batch, device="cuda", dtype=torch.uint8)
    x, dt, Bm, C, z = Hn.mamba2_inputs_dev(wl, wl.step_inputs(0))
    init = dec.state.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dec.step(x, dt, Bm, C, z, ci_d, force, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    dec.sr[1] = 0
    pool0 = _oracle_pool(wl)
    _oracle_step(wl, pool0, 0)
    outs = []
    for r in range(2):
        dec.state.copy_(init)
        dec.slot_wp.zero_()
        g.replay()
        torch.cuda.synchronize()
        st = _slots_state(dec, wl)
        ref = pool0.copy()
        oracle.round_slots_sr(ref, wl.cache_indices(), SEED, r)
        _compare_sr(st, ref[wl.cache_indices()])
        outs.append(st)
    assert not np.array_equal(outs[0], outs[1])
    assert int(dec.sr[1].item()) == 2
