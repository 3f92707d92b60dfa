"""CPU checks of bench.py's host-side bookkeeping: the spec cursor sequence it uses
for byte counts agrees with the oracle's cursor model, and the algorithmic byte
formulas reduce to their parts in simple cases."""
import numpy as np

import bench
import rssm_workloads as W
from oracle import cursors


def test_spec_cursor_rounds_match_the_cursor_model():
    rng = np.random.default_rng(3)
    L, T, slots = 8, 3, 10
    ci = np.array([7, 2, 5, 0], dtype=np.int32)
    seq = [rng.integers(0, T + 1, len(ci)) for _ in range(25)]
    sim, cnt_end = bench.spec_cursor_rounds(slots, ci, seq, L, T)
    cnt, base, flush = [0] * len(ci), [0] * len(ci), [0] * len(ci)
    local = np.arange(len(ci), dtype=np.int32)
    for r, acc in enumerate(seq):
        hist, fl, cr = sim[r]
        assert list(cr) == cnt and list(fl) == flush
        assert list(hist) == [0 if f else c for c, f in zip(cnt, flush)]
        cursors.spec_commit(cnt, base, flush, local, acc, L, T)
    assert list(cnt_end[ci]) == cnt


def test_byte_formulas_reduce_to_their_parts():
    wl = W.mamba2_spec(batch=2, nheads=4, ngroups=2, num_slots=4, L=8, T=2)
    zero = np.zeros(2, np.int64)
    v, f = bench.m2spec_round_bytes(wl, zero, zero, zero)
    assert f == 0
    H, P, N, G, T = 4, 64, 128, 2, 2
    entry = H * P * 2 + 4 * H + G * N * 2
    want = 2 * (H * P * N * 2 + T * (2 * H * P * 2 + 2 * G * N * 2 + 4 * H) + T * H * P * 2 + T * entry)
    assert v == want
    _, f1 = bench.m2spec_round_bytes(wl, zero, np.array([1, 0]), np.array([3, 0]))
    assert f1 == 2 * H * P * N * 2 + 3 * entry
    k = W.kda_decode(batch=2, num_v_heads=4, num_k_heads=2, num_slots=4)
    base = bench.kda_output_bytes(k, zero, zero)
    assert bench.kda_output_bytes(k, zero, np.array([1, 1])) - base == 2 * 4 * 128 * 128 * 4
    assert bench.kda_step_bytes(k, zero, zero) > base


def test_phase_complete_keeps_whole_cycles_of_in_region_samples():
    import bench
    # the last sample of each of 64 input sets, taken every 7th step: 64 consecutive
    # multiples of 7, whose residues mod 16 cover every phase 4 times
    ks = [7 * i for i in range(100, 164)]
    per = [1.0 + 0.001 * k for k in ks]
    got, src = bench._phase_complete(per, ks, None, None, 0, 0, 16, every=7)
    assert len(got) == 64 and "in the timed region" in src
    res = np.bincount(np.array([k for k, _ in got]) % 16, minlength=16)
    assert np.all(res == 4)
    # 40 samples: the last 32 are kept (two whole cycles)
    got, _ = bench._phase_complete(per[:40], ks[:40], None, None, 0, 0, 16, every=7)
    assert len(got) == 32 and [k for k, _ in got] == ks[8:40]
    assert np.all(np.bincount(np.array([k for k, _ in got]) % 16, minlength=16) == 2)


def test_source_hash_covers_the_included_headers():
    import os

    import bench
    files = set()
    bench._local_includes(os.path.join(bench.ROOT, "ssm_linear_attention_gb300", "csrc",
                                       "gdn.cu"), files)
    names = {os.path.basename(f) for f in files}
    assert {"gdn.cu", "pipeline.cuh", "common.cuh", "internal.h", "rssm.h"} <= names
    assert bench.source_hash("gdn.cu") != bench.source_hash("kda.cu")
    assert bench.source_hash("gdn.cu") == bench.source_hash("gdn.cu")
