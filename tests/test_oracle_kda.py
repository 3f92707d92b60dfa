"""Pins for the KDA (per-key-channel gate) part of the float64 oracle: the step
against the scalar-gate GDN step (already pinned) and the numpy matrix form, the
closed form against the recurrence, and the decay-only and memorisation cases."""
import numpy as np
import pytest

import oracle
import rssm_workloads as W


def _unit(a):
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


def test_kda_with_uniform_gate_is_gdn():
    r = np.random.default_rng(11)
    HV, HK, K, V = 4, 2, 8, 6
    S1 = r.standard_normal((2, HV, V, K))
    S2 = S1.copy()
    for t in range(4):
        q, k = _unit(r.standard_normal((2, HK, K))), _unit(r.standard_normal((2, HK, K)))
        v = r.standard_normal((2, HV, V))
        beta, g = r.uniform(0, 1, (2, HV)), r.uniform(0.2, 1, (2, HV))
        a = np.repeat(g[:, :, None], K, axis=2)
        o1 = oracle.kda_step(S1, q, k, v, beta, a)
        o2 = oracle.gdn_step(S2, q, k, v, beta, g)
        assert np.allclose(o1, o2, rtol=0, atol=1e-13)
        assert np.allclose(S1, S2, rtol=0, atol=1e-13)


def test_kda_matches_matrix_form():
    # S <- S Diag(a) + beta (v - S Diag(a) k) k^T  ==  S Diag(a) (I - beta k k^T) + beta v k^T
    r = np.random.default_rng(12)
    HV, HK, K, V = 4, 2, 6, 5
    S = r.standard_normal((1, HV, V, K))
    ref = S.copy()
    for t in range(5):
        q, k = _unit(r.standard_normal((1, HK, K))), _unit(r.standard_normal((1, HK, K)))
        v = r.standard_normal((1, HV, V))
        beta, a = r.uniform(0, 1, (1, HV)), r.uniform(0, 1, (1, HV, K))
        o = oracle.kda_step(S, q, k, v, beta, a)
        for hv in range(HV):
            kk = k[0, hv // (HV // HK)]
            M = np.diag(a[0, hv]) @ (np.eye(K) - beta[0, hv] * np.outer(kk, kk))
            ref[0, hv] = ref[0, hv] @ M + beta[0, hv] * np.outer(v[0, hv], kk)
            assert np.allclose(o[0, hv], ref[0, hv] @ q[0, hv // (HV // HK)], atol=1e-12)
    assert np.allclose(S, ref, atol=1e-12)


def test_kda_decay_only_scales_columns():
    # beta = 0: S <- S Diag(a), so after n steps column k is scaled by prod a[k]
    r = np.random.default_rng(13)
    HV, HK, K, V = 2, 1, 5, 3
    S = r.standard_normal((1, HV, V, K))
    S0 = S.copy()
    prod = np.ones((HV, K))
    for t in range(6):
        a = r.uniform(0.1, 1, (1, HV, K))
        oracle.kda_step(S, r.standard_normal((1, HK, K)), r.standard_normal((1, HK, K)),
                        r.standard_normal((1, HV, V)), np.zeros((1, HV)), a)
        prod *= a[0]
    assert np.allclose(S[0], S0[0] * prod[:, None, :], rtol=1e-13, atol=0)


def test_kda_memorises_orthonormal_keys_without_decay():
    # a = 1, beta = 1, orthonormal keys: after writing (k_i, v_i) pairs, S k_i = v_i
    K, V = 8, 4
    Q, _ = np.linalg.qr(np.random.default_rng(14).standard_normal((K, K)))
    S = np.zeros((1, 1, V, K))
    vs = np.random.default_rng(15).standard_normal((5, V))
    for i in range(5):
        oracle.kda_step(S, Q[None, None, :, i], Q[None, None, :, i], vs[i][None, None],
                        np.ones((1, 1)), np.ones((1, 1, K)))
    for i in range(5):
        assert np.allclose(S[0, 0] @ Q[:, i], vs[i], atol=1e-12)


@pytest.mark.parametrize("L", [1, 3, 8, 16])
def test_kda_closed_form_equals_recurrence(L):
    r = np.random.default_rng(20 + L)
    b, HV, HK, K, V, slots = 3, 4, 2, 8, 6, 5
    S0 = r.standard_normal((slots, HV, V, K))
    ci = np.array([4, 0, 2], dtype=np.int32)
    wp = np.array([L - 1, 0, min(2, L - 1)], dtype=np.int32)
    ek = _unit(r.standard_normal((b, L, HK, K)))
    ev = r.standard_normal((b, L, HV, V))
    ebeta = r.uniform(0, 1, (b, L, HV))
    ea = r.uniform(0.3, 1, (b, L, HV, K))
    q = _unit(r.standard_normal((b, HK, K)))
    o, Sf, dd = oracle.kda_replay(L, S0, ci, wp, ek, ev, ebeta, ea, q, want_fold=True, want_d=True)
    for row in range(b):
        S = S0.copy()
        w = wp[row]
        for i in range(w + 1):
            qq = q[row:row + 1] if i == w else ek[row:row + 1, i]
            oi = oracle.kda_step(S, qq, ek[row:row + 1, i], ev[row:row + 1, i],
                                 ebeta[row:row + 1, i], ea[row:row + 1, i], ci=ci[row:row + 1])
        assert np.allclose(o[row], oi[0], atol=1e-11)
        assert np.allclose(Sf[row], S[ci[row]], atol=1e-11)


def test_kda_workload_gates_in_range_and_run_is_consistent():
    wl = W.kda_decode(batch=3, num_v_heads=4, num_k_heads=2, num_slots=6, L=4, steps=5,
                      wp_mode="uniform")
    inp = wl.step_inputs(0)
    assert inp["a"].shape == (3, 4, 128) and np.all((inp["a"] > 0) & (inp["a"] < 1))
    a = oracle.kda_run(wl, steps=5, mode="replay")
    b = oracle.kda_run(wl, steps=5, mode="full")
    for t in range(5):
        assert np.allclose(a["o"][t], b["o"][t], rtol=0, atol=1e-5)
