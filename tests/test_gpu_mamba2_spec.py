"""GPU parity of the Mamba2 speculative verify (rssm_mamba2_spec_verify + the
SPEC_COMMIT cursor step) against the oracle's round-by-round recurrence: per-draft
outputs within the state dtype's bar (1e-4 fp32, 2e-3 bf16; harness metric),
cursors bit-exact, the checkpoints written by the folds within the same bar."""
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


def _check(wl, rows=None, chunk=64):
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    g = Hn.run_gpu_m2spec(wl, rows=rows)
    tol = Hn.tol_for(wl.state_dtype)
    ci_all = wl.cache_indices()
    flips, n_el, folds = 0, 0, 0
    for c0, sub in Hn.row_chunks(rows, chunk):
        ref = oracle.mamba2_spec_run(wl, rows=sub)
        sl = slice(c0, c0 + len(sub))
        for r in range(wl.rounds):
            e = Hn.err(g["y"][r][sl], ref["y"][r])
            assert e <= tol, (r, c0, e)
        assert np.array_equal(g["cnt"][:, sub], ref["cnt"])
        assert np.array_equal(g["base"][:, sub], ref["base"])
        assert np.array_equal(g["flush"][:, sub], ref["flush"])
        folds += int(np.count_nonzero(ref["flush"][:-1]))
        ci = ci_all[sub]
        st = g["ver"].state[torch.as_tensor(ci.astype(np.int64), device="cuda")].float().cpu().numpy()
        ok, e, fl = Hn.state_ok(st, ref["ckpt"], wl.state_dtype)
        assert ok, (c0, e, fl)
        flips += fl
        n_el += st.size
        del ref, st
    # at least one fold happened, so the stored checkpoints were rewritten
    assert folds > 0
    if wl.state_dtype == "bf16":
        assert flips / max(1, n_el) < 1e-3, flips / max(1, n_el)
    assert int(g["ver"].dev_err.abs().sum()) == 0


@pytest.mark.parametrize("T,L", [(1, 2), (2, 5), (3, 8), (4, 8), (4, 16)])
@pytest.mark.parametrize("sdt", ["bf16", "fp32"])
def test_mamba2_spec_matches_oracle(T, L, sdt):
    wl = W.mamba2_spec(batch=6, nheads=8, ngroups=2, num_slots=12, L=L, T=T, rounds=12,
                       state_dtype=sdt)
    _check(wl)


def test_mamba2_spec_fp32_activations_and_other_tile():
    wl = W.mamba2_spec(batch=4, nheads=4, ngroups=2, headdim=128, dstate=64, num_slots=8, L=8,
                       T=3, rounds=10, state_dtype="fp32", act_dtype="fp32")
    _check(wl)


@pytest.mark.parametrize("headdim,dstate,L,T,sdt,adt,rounds", [
    (128, 128, 32, 4, "bf16", "fp32", 26),  # bf16 state with float32 activations; 32 rows a thread
    (64, 64, 20, 3, "bf16", "bf16", 18),    # 8 rows a thread; a ring longer than 16 entries
    (128, 128, 12, 2, "fp32", "bf16", 20),  # float32 state with 32 rows a thread
])
def test_mamba2_spec_fold_shapes(headdim, dstate, L, T, sdt, adt, rounds):
    # the prologue's fold paths: staging batches, rows held per thread, dtype pairs
    wl = W.mamba2_spec(batch=5, nheads=8, ngroups=2, headdim=headdim, dstate=dstate,
                       num_slots=10, L=L, T=T, rounds=rounds, state_dtype=sdt, act_dtype=adt)
    _check(wl)


def test_mamba2_spec_bench_geometry_all_rows():
    # batch 128, T 4, H 128, P 64, N 128, G 8, L 16, bf16 state: every row's draft
    # outputs in every round and every folded checkpoint
    wl = W.mamba2_spec(batch=128, num_slots=256, rounds=12)
    _check(wl)


def test_mamba2_spec_padding_and_bad_slot():
    import ssm_linear_attention_gb300 as ssm
    from ssm_linear_attention_gb300 import Mamba2SpecVerifier
    wl = W.mamba2_spec(batch=4, nheads=8, ngroups=2, num_slots=8, L=8, T=2, rounds=1)
    prm = wl.params()
    ver = Mamba2SpecVerifier(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.L, wl.T,
                             wl.num_slots, wl.batch, prm["A"], prm["D"], prm["dt_bias"],
                             out_dtype=torch.float32)
    ci = wl.cache_indices().copy()
    ci[1] = -1
    ci[2] = wl.num_slots + 1
    inp = wl.round_inputs(0)
    bf = torch.bfloat16
    y = torch.full((wl.batch, wl.T, wl.nheads, wl.headdim), 3.0, device="cuda")
    ver.verify(Hn.to_dev(inp["x"], bf), Hn.to_dev(inp["dt_raw"], torch.float32),
               Hn.to_dev(inp["B"], bf), Hn.to_dev(inp["C"], bf), Hn.to_dev(inp["z"], bf),
               Hn.to_dev(ci, torch.int32), y=y)
    torch.cuda.synchronize()
    assert torch.all(y[1] == 3.0) and torch.all(y[2] == 3.0)
    assert int(ver.dev_err[0].item()) & ssm.RSSM_DEVERR_SLOT
