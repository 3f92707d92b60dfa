"""Pins for the gated-delta-net side of the float64 oracle (decode and spec verify)."""
import numpy as np
import pytest

import oracle
import rssm_workloads as W


def _unit(a):
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


def test_gdn_hand_example():
    # K = V = 2, S0 = I, k = e1, v = e2, beta = 1/2, g = 1/2, q = e2.
    #   u = S0 k = [1, 0];  d = 0.5 * ([0, 1] - 0.5 * [1, 0]) = [-0.25, 0.5]
    #   S = 0.5 I + d k^T = [[0.5 - 0.25, 0], [0.5, 0.5]] = [[0.25, 0], [0.5, 0.5]]
    #   o = S q = [0, 0.5]
    S = np.eye(2)[None, None].copy()
    o = oracle.gdn_step(S, q=[[[0.0, 1.0]]], k=[[[1.0, 0.0]]], v=[[[0.0, 1.0]]], beta=[[0.5]],
                        g=[[0.5]])
    assert S[0, 0].tolist() == [[0.25, 0.0], [0.5, 0.5]]
    assert o[0, 0].tolist() == [0.0, 0.5]


def test_gdn_matches_matrix_form():
    # S <- g S + beta (v - g S k) k^T  ==  S (g (I - beta k k^T)) + beta v k^T, o = S q
    r = np.random.default_rng(2)
    HV, HK, K, V = 4, 2, 6, 5
    S = r.standard_normal((1, HV, V, K))
    ref = S.copy()
    for t in range(5):
        q, k = _unit(r.standard_normal((1, HK, K))), _unit(r.standard_normal((1, HK, K)))
        v = r.standard_normal((1, HV, V))
        beta, g = r.uniform(0, 1, (1, HV)), r.uniform(0, 1, (1, HV))
        o = oracle.gdn_step(S, q, k, v, beta, g)
        for hv in range(HV):
            kh = hv // (HV // HK)
            kk = k[0, kh]
            M = g[0, hv] * (np.eye(K) - beta[0, hv] * np.outer(kk, kk))
            ref[0, hv] = ref[0, hv] @ M + beta[0, hv] * np.outer(v[0, hv], kk)
            assert np.allclose(o[0, hv], ref[0, hv] @ q[0, kh], rtol=1e-12, atol=1e-13)
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-13)


def test_gdn_delta_rule_memorises_orthonormal_keys():
    # beta = 1, g = 1, orthonormal keys: after writing (k_i, v_i) for i = 1..m,
    # S k_i = v_i for every i, so querying with q = k_i returns v_i.
    r = np.random.default_rng(3)
    K, V, m = 8, 5, 6
    Q, _ = np.linalg.qr(r.standard_normal((K, K)))
    keys = Q[:, :m].T
    vals = r.standard_normal((m, V))
    S = r.standard_normal((1, 1, V, K))
    for i in range(m):
        oracle.gdn_step(S, keys[i][None, None], keys[i][None, None], vals[i][None, None], [[1.0]],
                        [[1.0]])
    for i in range(m):
        assert np.allclose(S[0, 0] @ keys[i], vals[i], atol=1e-12)
    o = oracle.gdn_step(S.copy(), keys[2][None, None], keys[m - 1][None, None], vals[m - 1][None, None],
                        [[1.0]], [[1.0]])
    assert np.allclose(o[0, 0], vals[2], atol=1e-12)


def test_gdn_degenerate_gates():
    r = np.random.default_rng(4)
    K, V = 4, 3
    S0 = r.standard_normal((1, 1, V, K))
    q, k, v = r.standard_normal((1, 1, K)), r.standard_normal((1, 1, K)), r.standard_normal((1, 1, V))
    S = S0.copy()
    oracle.gdn_step(S, q, k, v, [[0.7]], [[0.0]])     # g = 0: S = beta v k^T
    assert np.allclose(S[0, 0], 0.7 * np.outer(v[0, 0], k[0, 0]), atol=1e-15)
    S = S0.copy()
    oracle.gdn_step(S, q, k, v, [[0.0]], [[0.3]])     # beta = 0: S = g S0
    assert np.allclose(S[0, 0], 0.3 * S0[0, 0], atol=1e-15)


def test_gdn_gqa_mapping():
    # HV = 4 value heads over HK = 2 key heads: value heads 0,1 read key head 0,
    # heads 2,3 read key head 1. Perturbing key head 1 changes only heads 2, 3.
    r = np.random.default_rng(5)
    HV, HK, K, V = 4, 2, 4, 3
    S = r.standard_normal((1, HV, V, K))
    q, k = r.standard_normal((1, HK, K)), r.standard_normal((1, HK, K))
    v, beta, g = r.standard_normal((1, HV, V)), np.full((1, HV), 0.5), np.full((1, HV), 0.9)
    o1 = oracle.gdn_step(S.copy(), q, k, v, beta, g)
    k2 = k.copy()
    k2[0, 1] += 1.0
    o2 = oracle.gdn_step(S.copy(), q, k2, v, beta, g)
    changed = [h for h in range(HV) if not np.allclose(o1[0, h], o2[0, h])]
    assert changed == [2, 3]


@pytest.mark.parametrize("L", [1, 3, 8, 16])
def test_gdn_replay_form_equals_recurrence(L):
    r = np.random.default_rng(30 + L)
    b, HV, HK, K, V = 3, 4, 2, 8, 6
    S0 = r.standard_normal((b, HV, V, K)) * 0.05
    ek, eq = _unit(r.standard_normal((b, L, HK, K))), _unit(r.standard_normal((b, L, HK, K)))
    ev = r.standard_normal((b, L, HV, V))
    ebeta = 1 / (1 + np.exp(-r.standard_normal((b, L, HV))))
    eg = np.exp(-np.log1p(np.exp(r.standard_normal((b, L, HV)) + 1)))
    wp = r.integers(0, L, b)
    state = S0.copy()
    o_rec = np.zeros((b, HV, V))
    for i in range(L):
        ci = np.where(wp >= i, np.arange(b), -1)
        o = oracle.gdn_step(state, eq[:, i], ek[:, i], ev[:, i], ebeta[:, i], eg[:, i], ci=ci)
        o_rec[wp == i] = o[wp == i]
    qw = eq[np.arange(b), wp]
    o_rep, S_fold = oracle.gdn_replay(L, S0, np.arange(b), wp, ek, ev, ebeta, eg, qw, want_fold=True)
    assert np.allclose(o_rep, o_rec, rtol=1e-12, atol=1e-13)
    assert np.allclose(S_fold, state, rtol=1e-12, atol=1e-13)


def test_gdn_replay_d_entries_are_the_recurrence_deltas():
    # The ring entry d_i = beta_i (v_i - g_i S_{i-1} k_i) equals the recurrence's delta.
    r = np.random.default_rng(40)
    L, HV, HK, K, V = 5, 2, 1, 4, 3
    S0 = r.standard_normal((1, HV, V, K))
    ek = _unit(r.standard_normal((1, L, HK, K)))
    ev = r.standard_normal((1, L, HV, V))
    eb, eg = r.uniform(0, 1, (1, L, HV)), r.uniform(0, 1, (1, L, HV))
    _, dd = oracle.gdn_replay(L, S0, [0], [L - 1], ek, ev, eb, eg, ek[:, -1], want_d=True)
    S = S0[0].copy()
    for i in range(L):
        for hv in range(HV):
            d_ref = eb[0, i, hv] * (ev[0, i, hv] - eg[0, i, hv] * S[hv] @ ek[0, i, 0])
            assert np.allclose(dd[0, i, hv], d_ref, rtol=1e-12, atol=1e-13)
            S[hv] = eg[0, i, hv] * S[hv] + np.outer(d_ref, ek[0, i, 0])


# --------------------------------------------------------------------------- #
# speculative verify round                                                    #
# --------------------------------------------------------------------------- #

def test_spec_round_outputs_are_sequential_steps():
    r = np.random.default_rng(50)
    b, T, HV, HK, K, V = 3, 4, 2, 1, 6, 5
    S0 = r.standard_normal((b, HV, V, K)) * 0.1
    q, k = _unit(r.standard_normal((b, T, HK, K))), _unit(r.standard_normal((b, T, HK, K)))
    v = r.standard_normal((b, T, HV, V))
    beta, g = r.uniform(0, 1, (b, T, HV)), r.uniform(0, 1, (b, T, HV))
    acc = np.array([0, 2, 4])
    S = S0.copy()
    o = oracle.gdn_spec_round(S, T, q, k, v, beta, g, acc)
    ref = S0.copy()
    for j in range(T):
        oj = oracle.gdn_step(ref, q[:, j], k[:, j], v[:, j], beta[:, j], g[:, j])
        assert np.allclose(o[:, j], oj, rtol=1e-13, atol=1e-14)
        for row in range(b):
            if acc[row] == j + 1:
                assert np.array_equal(S[row], ref[row])
    assert np.array_equal(S[0], S0[0])   # nothing accepted: state unchanged


def test_spec_T1_always_accept_equals_decode():
    wl = W.gdn_spec(batch=2, num_v_heads=2, num_k_heads=1, head_k_dim=8, head_v_dim=4, T=1, L=4,
                    num_slots=4, rounds=5)
    wl.accepted = lambda r: np.ones(wl.batch, dtype=np.int32)
    res = oracle.gdn_spec_run(wl)
    st = np.stack([wl.slot_state(int(s)) for s in wl.cache_indices()]).astype(np.float64)
    for rr in range(5):
        inp = wl.round_inputs(rr)
        o = oracle.gdn_step(st, inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], inp["beta"][:, 0],
                            inp["g"][:, 0])
        # the spec path rounds the state to fp32 at folds; compare loosely
        assert np.allclose(res["o"][rr][:, 0], o, rtol=1e-6, atol=1e-7)
