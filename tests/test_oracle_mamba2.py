"""Pins for the Mamba2 side of the float64 oracle.

Each test checks the oracle against something other than itself: a library
routine (scipy.signal.lfilter, torch's bfloat16 conversion), a closed form, a
hand-worked example, or an algebraic invariant between two different routes.
"""
import math

import numpy as np
import pytest
import scipy.signal
import torch

import oracle
import rssm_workloads as W


def _silu(z):
    return z / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------- #
# scalar helpers                                                              #
# --------------------------------------------------------------------------- #

def test_softplus_identities():
    # softplus(0) = ln 2; softplus(x) - softplus(-x) = x; softplus(x) -> x for large x
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    for x in (-30.0, -3.0, -0.5, 0.25, 2.0, 40.0, 700.0):
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, abs=1e-12 * max(1, abs(x)))
    assert oracle.softplus(800.0) == 800.0
    assert oracle.softplus(-800.0) == 0.0


def test_round_bf16_matches_torch_on_float32_inputs():
    r = np.random.default_rng(1)
    vals = np.concatenate([r.standard_normal(20000), r.standard_normal(2000) * 1e-30,
                           r.standard_normal(2000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals])
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even():
    # bfloat16 spacing in [1, 2) is 2^-7; exact midpoints round to the even neighbour
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7
    assert oracle.round_f32(1.0 + 2.0 ** -24) == 1.0
    assert oracle.round_f32(1.0 + 3 * 2.0 ** -24) == 1.0 + 2.0 ** -22


# --------------------------------------------------------------------------- #
# the recurrence                                                              #
# --------------------------------------------------------------------------- #

def test_mamba2_hand_example():
    # headdim 1, dstate 2, one head, no softplus. dt = 0.5, A = -2 ln 2 so dA = 1/2.
    # h0 = [1, 3], x = 2, B = [1, -1], C = [1, 2], D = 0.25.
    #   h1 = 0.5*h0 + 0.5*2*B = [0.5+1, 1.5-1] = [1.5, 0.5]
    #   y  = 1.5*1 + 0.5*2 + 0.25*2 = 3.0
    # with z = 1: y *= 1/(1+e^-1)
    state = np.array([[[[1.0, 3.0]]]])
    y = oracle.mamba2_step(state, x=[[[2.0]]], dt_raw=[[0.5]], A=[-2 * math.log(2.0)],
                           B=[[[1.0, -1.0]]], C=[[[1.0, 2.0]]], D=[0.25], dt_softplus=False)
    assert state[0, 0, 0].tolist() == pytest.approx([1.5, 0.5], abs=1e-15)
    assert y[0, 0, 0] == pytest.approx(3.0, abs=1e-15)
    state = np.array([[[[1.0, 3.0]]]])
    y = oracle.mamba2_step(state, x=[[[2.0]]], dt_raw=[[0.5]], A=[-2 * math.log(2.0)],
                           B=[[[1.0, -1.0]]], C=[[[1.0, 2.0]]], D=[0.25], z=[[[1.0]]],
                           dt_softplus=False)
    assert y[0, 0, 0] == pytest.approx(3.0 / (1.0 + math.exp(-1.0)), abs=1e-15)


def test_mamba2_matches_lfilter_for_constant_decay():
    # With dt fixed per head over time, every state element h[p, n] is the
    # first-order IIR filter h_t = dA h_{t-1} + u_t, u_t = dt x_t[p] B_t[n]:
    # scipy.signal.lfilter([1], [1, -dA], u, zi=[dA h_{-1}]).
    r = np.random.default_rng(7)
    H, P, N, G, Tn = 4, 3, 5, 2, 9
    A = -np.exp(r.uniform(0, np.log(16), H))
    D = r.standard_normal(H)
    dt_bias = r.uniform(-4, -2, H)
    dt_raw = r.standard_normal(H)
    h0 = r.standard_normal((1, H, P, N)) * 0.1
    xs = r.standard_normal((Tn, 1, H, P))
    Bs = r.standard_normal((Tn, 1, G, N))
    Cs = r.standard_normal((Tn, 1, G, N))
    zs = r.standard_normal((Tn, 1, H, P))
    state = h0.copy()
    ys = np.stack([oracle.mamba2_step(state, xs[t], dt_raw[None], A, Bs[t], Cs[t], D, zs[t],
                                      dt_bias) for t in range(Tn)])
    hpg = H // G
    for h in range(H):
        g = h // hpg
        dt = math.log1p(math.exp(dt_raw[h] + dt_bias[h]))
        a = math.exp(A[h] * dt)
        for p in range(P):
            hist = np.zeros((Tn, N))
            for n in range(N):
                u = dt * xs[:, 0, h, p] * Bs[:, 0, g, n]
                hist[:, n], _ = scipy.signal.lfilter([1.0], [1.0, -a], u, zi=[a * h0[0, h, p, n]])
            assert np.allclose(state[0, h, p], hist[-1], rtol=1e-12, atol=1e-14)
            ref_y = (hist * Cs[:, 0, g, :]).sum(1) + D[h] * xs[:, 0, h, p]
            ref_y = ref_y * _silu(zs[:, 0, h, p])
            assert np.allclose(ys[:, 0, h, p], ref_y, rtol=1e-11, atol=1e-13)


def test_mamba2_first_step_from_zero_state():
    # From h = 0: y = (dt * x[p] * (B . C) + D x[p]) * silu(z[p])
    r = np.random.default_rng(3)
    H, P, N, G = 4, 8, 16, 2
    x, z = r.standard_normal((1, H, P)), r.standard_normal((1, H, P))
    B, C = r.standard_normal((1, G, N)), r.standard_normal((1, G, N))
    A, D, dt_raw, dt_bias = -np.ones(H), r.standard_normal(H), r.standard_normal((1, H)), np.zeros(H)
    state = np.zeros((1, H, P, N))
    y = oracle.mamba2_step(state, x, dt_raw, A, B, C, D, z, dt_bias)
    for h in range(H):
        g = h // (H // G)
        dt = math.log1p(math.exp(dt_raw[0, h]))
        ref = (dt * x[0, h] * (B[0, g] @ C[0, g]) + D[h] * x[0, h]) * _silu(z[0, h])
        assert np.allclose(y[0, h], ref, rtol=1e-13, atol=1e-15)


def test_mamba2_no_decay_is_a_plain_sum():
    # A = 0 gives dA = 1: h = h0 + sum_t dt_t x_t B_t^T
    r = np.random.default_rng(4)
    H, P, N = 2, 3, 4
    h0 = r.standard_normal((1, H, P, N))
    state = h0.copy()
    acc = h0.copy()
    for t in range(6):
        x, B, C = r.standard_normal((1, H, P)), r.standard_normal((1, 1, N)), r.standard_normal((1, 1, N))
        dt_raw = r.standard_normal((1, H))
        oracle.mamba2_step(state, x, dt_raw, np.zeros(H), B, C, np.zeros(H))
        dt = np.log1p(np.exp(dt_raw[0]))
        acc[0] += dt[:, None, None] * x[0][:, :, None] * B[0, 0][None, None, :]
    assert np.allclose(state, acc, rtol=1e-13, atol=1e-14)


def test_mamba2_group_mapping_is_contiguous_blocks():
    # 8 heads, 4 groups: heads 2g and 2g+1 read group g. Only group 2 has a
    # non-zero B, so only heads 4 and 5 gain state.
    H, P, N, G = 8, 2, 3, 4
    B = np.zeros((1, G, N))
    B[0, 2] = [1.0, 2.0, 3.0]
    state = np.zeros((1, H, P, N))
    oracle.mamba2_step(state, np.ones((1, H, P)), np.zeros((1, H)), -np.ones(H), B,
                       np.ones((1, G, N)), np.zeros(H))
    nz = [h for h in range(H) if np.abs(state[0, h]).sum() > 0]
    assert nz == [4, 5]


def test_mamba2_slot_indexing_and_padding():
    # rows write only their own slot; a row with index -1 touches nothing
    r = np.random.default_rng(5)
    H, P, N = 2, 2, 4
    pool = r.standard_normal((5, H, P, N))
    before = pool.copy()
    ci = np.array([3, -1, 0])
    oracle.mamba2_step(pool, r.standard_normal((3, H, P)), r.standard_normal((3, H)), -np.ones(H),
                       r.standard_normal((3, 1, N)), r.standard_normal((3, 1, N)), np.zeros(H), ci=ci)
    for s in (1, 2, 4):
        assert np.array_equal(pool[s], before[s])
    assert not np.array_equal(pool[3], before[3]) and not np.array_equal(pool[0], before[0])


# --------------------------------------------------------------------------- #
# ReplaySSM closed form vs the recurrence                                     #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("L", [1, 2, 5, 16])
def test_mamba2_replay_form_equals_recurrence(L):
    r = np.random.default_rng(10 + L)
    b, H, P, N, G = 3, 4, 5, 6, 2
    A = -np.exp(r.uniform(0, np.log(16), H))
    D, dt_bias = r.standard_normal(H), r.uniform(-4, -2, H)
    S0 = r.standard_normal((b, H, P, N)) * 0.1
    ex = r.standard_normal((b, L, H, P))
    edt = r.standard_normal((b, L, H))
    eB = r.standard_normal((b, L, G, N)) / 4
    eC = r.standard_normal((b, L, G, N)) / 4
    z = r.standard_normal((b, H, P))
    wp = r.integers(0, L, b)
    # recurrence: each row steps through its entries 0..wp[b]
    state = S0.copy()
    y_rec = np.zeros((b, H, P))
    for i in range(L):
        ci = np.where(wp >= i, np.arange(b), -1)
        y = oracle.mamba2_step(state, ex[:, i], edt[:, i], A, eB[:, i], eC[:, i], D, z, dt_bias, ci=ci)
        y_rec[wp == i] = y[wp == i]
    Cw = eC[np.arange(b), wp]
    y_rep, S_fold = oracle.mamba2_replay(L, S0, np.arange(b), wp, ex, edt, A, eB, Cw, D, z, dt_bias,
                                         want_fold=True)
    assert np.allclose(y_rep, y_rec, rtol=1e-12, atol=1e-13)
    assert np.allclose(S_fold, state, rtol=1e-12, atol=1e-13)


def test_mamba2_prefill_then_decode():
    # A prompt of n steps run through the recurrence and stored as the checkpoint,
    # then m decode steps through the closed form, equals n+m recurrence steps.
    r = np.random.default_rng(21)
    H, P, N, n, m, L = 2, 4, 8, 5, 4, 8
    A = -np.exp(r.uniform(0, np.log(16), H))
    D, dt_bias = r.standard_normal(H), r.uniform(-4, -2, H)
    xs, dts = r.standard_normal((n + m, 1, H, P)), r.standard_normal((n + m, 1, H))
    Bs, Cs = r.standard_normal((n + m, 1, 1, N)) / 3, r.standard_normal((n + m, 1, 1, N)) / 3
    h0 = r.standard_normal((1, H, P, N)) * 0.1
    full = h0.copy()
    y_full = [oracle.mamba2_step(full, xs[t], dts[t], A, Bs[t], Cs[t], D, None, dt_bias)
              for t in range(n + m)]
    S0 = h0.copy()
    for t in range(n):
        oracle.mamba2_step(S0, xs[t], dts[t], A, Bs[t], Cs[t], D, None, dt_bias)
    ex = np.zeros((1, L, H, P)); edt = np.zeros((1, L, H)); eB = np.zeros((1, L, 1, N))
    for j in range(m):
        ex[0, j], edt[0, j], eB[0, j] = xs[n + j, 0], dts[n + j, 0], Bs[n + j, 0]
        y = oracle.mamba2_replay(L, S0, [0], [j], ex, edt, A, eB, Cs[n + j], D, None, dt_bias)
        assert np.allclose(y, y_full[n + j], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- #
# the workload driver                                                         #
# --------------------------------------------------------------------------- #

def test_driver_L1_replay_equals_full_state_rounding():
    # L = 1 flushes every step, so ReplaySSM storage equals per-step storage.
    wl = W.mamba2_large(batch=3, nheads=4, ngroups=2, headdim=8, dstate=16, num_slots=8, L=1,
                        steps=5)
    a = oracle.mamba2_run(wl, mode="replay")
    b = oracle.mamba2_run(wl, mode="full")
    assert np.all(a["row_flush"] == 1) and np.all(a["row_wp"] == 0)
    for ya, yb in zip(a["y"], b["y"]):
        assert np.array_equal(ya, yb)
    assert np.array_equal(a["ckpt"], b["ckpt"])


def test_driver_history_and_checkpoints():
    # fp32 state: the driver's state after history + steps equals a plain loop of
    # recurrence steps (up to the fp32 rounding at flushes), and the checkpoint is
    # the state of each row's last flush.
    wl = W.mamba2_large(batch=4, nheads=4, ngroups=2, headdim=8, dstate=16, num_slots=8, L=4,
                        steps=7, state_dtype="fp32")
    res = oracle.mamba2_run(wl, mode="replay")
    prm, ci = wl.params(), wl.cache_indices()
    hist = wl.history_len()
    for b in range(wl.batch):
        st = wl.slot_state(int(ci[b]))[None].astype(np.float64)
        ck = st.copy()
        wp = 0
        seq = [wl.history_inputs(j) for j in range(int(hist[b]))] + \
              [wl.step_inputs(t) for t in range(wl.steps)]
        for k, inp in enumerate(seq):
            oracle.mamba2_step(st, inp["x"][b:b + 1], inp["dt_raw"][b:b + 1], prm["A"],
                               inp["B"][b:b + 1], inp["C"][b:b + 1], prm["D"],
                               inp["z"][b:b + 1], prm["dt_bias"])
            if wp == wl.L - 1:
                ck = st.copy()
                wp = 0
            else:
                wp += 1
        assert np.allclose(res["state"][b], st[0], rtol=1e-6, atol=1e-7)
        assert np.allclose(res["ckpt"][b], ck[0], rtol=1e-6, atol=1e-7)
        assert res["slot_wp"][b] == wp


# --------------------------------------------------------------------------- #
# speculative verify round                                                    #
# --------------------------------------------------------------------------- #

def _spec_inputs(r, b, T, H, P, N, G):
    return dict(x=r.standard_normal((b, T, H, P)), dt_raw=r.standard_normal((b, T, H)),
                B=r.standard_normal((b, T, G, N)) / np.sqrt(N),
                C=r.standard_normal((b, T, G, N)) / np.sqrt(N), z=r.standard_normal((b, T, H, P)))


def test_mamba2_spec_round_equals_sequential_steps():
    # draft j's output = the recurrence after drafts 0..j; the slot keeps the state
    # after the accepted prefix only
    r = np.random.default_rng(31)
    b, T, H, P, N, G, slots = 3, 4, 4, 3, 5, 2, 6
    A = -np.exp(r.uniform(0, 2, H))
    D = r.standard_normal(H)
    dtb = r.uniform(-3, -2, H)
    S = r.standard_normal((slots, H, P, N))
    ci = np.array([5, 1, 3], dtype=np.int32)
    acc = np.array([2, 0, 4], dtype=np.int32)
    inp = _spec_inputs(r, b, T, H, P, N, G)
    S_spec = S.copy()
    y = oracle.mamba2_spec_round(S_spec, T, inp["x"], inp["dt_raw"], A, inp["B"], inp["C"], D, acc,
                                 inp["z"], dtb, True, ci)
    for row in range(b):
        St = S.copy()
        for j in range(T):
            sl = slice(row, row + 1)
            yj = oracle.mamba2_step(St, inp["x"][sl, j], inp["dt_raw"][sl, j], A, inp["B"][sl, j],
                                    inp["C"][sl, j], D, inp["z"][sl, j], dtb, True, ci=ci[sl])
            assert np.allclose(y[row, j], yj[0], rtol=0, atol=1e-12)
            if j + 1 == acc[row]:
                keep = St[ci[row]].copy()
        want = S[ci[row]] if acc[row] == 0 else keep
        assert np.array_equal(S_spec[ci[row]], want)


def test_mamba2_spec_run_t1_always_accept_equals_decode():
    # T = 1 with every draft accepted is plain decode (flush every L - 1 rounds)
    wl = W.mamba2_spec(batch=3, nheads=4, ngroups=2, num_slots=6, L=4, T=1, rounds=6,
                       state_dtype="fp32", act_dtype="fp32")
    wl.accepted = lambda r: np.ones(wl.batch, dtype=np.int32)
    ref = oracle.mamba2_spec_run(wl)
    prm = wl.params()
    S = np.stack([wl.slot_state(int(s)) for s in wl.cache_indices()]).astype(np.float64)
    for r in range(6):
        inp = wl.round_inputs(r)
        y = oracle.mamba2_step(S, inp["x"][:, 0], inp["dt_raw"][:, 0], prm["A"], inp["B"][:, 0],
                               inp["C"][:, 0], prm["D"], inp["z"][:, 0], prm["dt_bias"], True)
        assert np.allclose(ref["y"][r][:, 0], y, rtol=0, atol=1e-5)
