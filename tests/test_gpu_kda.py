"""GPU parity of the KDA (per-key-channel gate) decode path against the oracle
("GDN ReplaySSM decode (Part A of RFC 28511)", 实现拆解 item 1: one buffered decode
kernel for GDN and KDA; 6: equality with the conventional kernel at L = 1/4/8/16,
fp32 and bf16). Outputs and flushed fp32 checkpoints e <= 1e-4 (harness metric);
cursors bit-exact."""
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


def _small(L, act="bf16", **kw):
    d = dict(batch=6, num_v_heads=4, num_k_heads=2, num_slots=12, L=L, steps=2 * L + 3,
             act_dtype=act, wp_mode="uniform", force_rate=0.1)
    d.update(kw)
    return W.kda_decode(**d)


def _check(wl, steps, rows=None, full=False, staged=False):
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    g = Hn.run_gpu_kda(wl, steps=steps, rows=rows, full_state=full, staged=staged)
    ref = oracle.kda_run(wl, rows=rows, steps=steps, mode="full" if full else "replay")
    for t in range(steps):
        e = Hn.err(g["o"][t], ref["o"][t])
        assert e <= 1e-4, (t, e)
    if not full:
        assert np.array_equal(g["row_wp"][:, rows], ref["row_wp"])
        assert np.array_equal(g["row_flush"][:, rows], ref["row_flush"])
    ci = wl.cache_indices()[rows]
    st = g["dec"].state[torch.as_tensor(ci.astype(np.int64), device="cuda")].cpu().numpy()
    ok, e, _ = Hn.state_ok(st, ref["ckpt"], "fp32")
    assert ok, e
    return g


@pytest.mark.parametrize("L", [1, 4, 8, 16])
@pytest.mark.parametrize("act", ["bf16", "fp32"])
def test_kda_decode_matches_oracle(L, act):
    _check(_small(L, act), steps=2 * L + 3)


@pytest.mark.parametrize("act", ["bf16", "fp32"])
def test_kda_full_state_matches_oracle(act):
    _check(_small(4, act), steps=6, full=True)


def test_kda_bench_geometry_sampled_rows():
    wl = W.kda_decode(batch=64, num_slots=128, steps=17, wp_mode="uniform")
    _check(wl, steps=17, rows=[0, 21, 63])


def test_kda_staged_calls_equal_fused_step():
    wl = _small(8, force_rate=0.2)
    a = Hn.run_gpu_kda(wl, steps=10)
    b = Hn.run_gpu_kda(wl, steps=10, staged=True)
    for t in range(10):
        assert np.array_equal(a["o"][t], b["o"][t])
    assert torch.equal(a["dec"].state, b["dec"].state)
    assert torch.equal(a["dec"].ring_d, b["dec"].ring_d)


def test_kda_padding_rows_untouched_and_bad_slots_flagged():
    import ssm_linear_attention_gb300 as ssm
    wl = _small(4, wp_mode="zero", force_rate=0.0)
    dec = Hn.make_kda_decoder(wl)
    ci = wl.cache_indices().copy()
    ci[1] = -1
    ci[4] = wl.num_slots + 5
    q, k, v, be, a = Hn.kda_inputs_dev(wl, wl.step_inputs(0))
    o = torch.full((wl.batch, wl.num_v_heads, wl.head_v_dim), 7.0, device="cuda")
    before = dec.state.clone()
    dec.step(q, k, v, be, a, Hn.to_dev(ci, torch.int32), o=o)
    torch.cuda.synchronize()
    assert torch.all(o[1] == 7.0) and torch.all(o[4] == 7.0)
    assert int(dec.dev_err[0].item()) & ssm.RSSM_DEVERR_SLOT
    assert torch.equal(dec.state, before)      # w = 0, L = 4: no flush
    ref = oracle.kda_run(wl, rows=[0, 2, 3, 5], steps=1)
    assert Hn.err(o[[0, 2, 3, 5]].cpu().numpy(), ref["o"][0]) <= 1e-4
