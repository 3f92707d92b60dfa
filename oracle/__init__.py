"""Float64 CPU oracle for ReplaySSM decode (Mamba2 and gated delta net).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` import this package. The CUDA
product path (``ssm_linear_attention_gb300``) never imports, links or calls it,
and the two share no code; the only common module is ``rssm_workloads``, which
draws the seeded inputs and holds none of the method's arithmetic.

Contents:
  * ``oracle.c`` (built into ``liborc.so`` by ``build.py``): the full-state
    recurrences for Mamba2, the gated delta rule and its per-key-channel-gate
    (KDA) form, the ReplaySSM closed forms (checkpoint + ring) of all three, one
    speculative verify round for Mamba2 and for the gated delta rule, the storage
    rounding helpers, and Philox4x32-10 with the stochastic rounding to bf16.
    Every function cites the page passage (or the published definition) it
    follows.
  * ``cursors.py``: the integer cursor model (write_pos / is_flush, the circular
    spec ring).
  * The drivers below run a whole workload (history steps, then the measured
    steps) for a chosen subset of batch rows, in one of two storage modes:
      - "replay": the slot's state is rounded to its storage dtype only when the
        row flushes (ReplaySSM keeps S0 frozen between flushes and accumulates
        the rest in fp32; [M2] 风险与影响 item 2 states that ReplaySSM writes the
        state back once where the baseline rounds it every step);
      - "full": rounded every step (the conventional decode kernel).
    Rows are independent, so a subset of rows is computed exactly as it would be
    inside the full batch.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against closed forms, library routines (scipy.signal.lfilter, numpy matrix
algebra, torch's bfloat16 conversion), hand-worked examples, invariants and
published known-answer vectors (Philox4x32-10, ``tests/golden/``).
"""
import ctypes
import os
from typing import Dict, Optional, Sequence

import numpy as np

from . import build as _build
from . import cursors

__all__ = ["lib", "round_bf16", "round_f32", "softplus", "mamba2_step", "mamba2_replay",
           "gdn_step", "gdn_replay", "gdn_spec_round", "round_slots", "default_threads",
           "mamba2_run", "gdn_run", "gdn_spec_run", "cursors", "philox4x32_10", "round_bf16_sr",
           "sr_bits", "round_slots_sr", "kda_step", "kda_replay", "kda_run",
           "mamba2_spec_round", "mamba2_spec_run"]

_lib = None


class _M2Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("batch", "nheads", "headdim", "dstate", "ngroups", "num_slots")]


class _GDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("batch", "num_v_heads", "num_k_heads", "head_k_dim", "head_v_dim", "num_slots")]


_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def lib():
    """Load (building first if needed) liborc.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_round_bf16.restype = ctypes.c_double
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_round_f32.restype = ctypes.c_double
        L.orc_round_f32.argtypes = [ctypes.c_double]
        L.orc_softplus.restype = ctypes.c_double
        L.orc_softplus.argtypes = [ctypes.c_double]
        L.orc_default_threads.restype = ctypes.c_int
        L.orc_round_slots.argtypes = [_dp, ctypes.c_long, _ip, ctypes.c_int, ctypes.c_int]
        _u32p = ctypes.POINTER(ctypes.c_uint32)
        L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.orc_round_bf16_sr.restype = ctypes.c_double
        L.orc_round_bf16_sr.argtypes = [ctypes.c_double, ctypes.c_uint]
        L.orc_sr_bits.restype = ctypes.c_uint
        L.orc_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.orc_round_slots_sr.argtypes = [_dp, ctypes.c_long, _ip, ctypes.c_int, ctypes.c_uint64,
                                         ctypes.c_uint64]
        L.orc_mamba2_step.argtypes = [ctypes.POINTER(_M2Dims), _dp, _dp, _dp, _dp, ctypes.c_int,
                                      _dp, _dp, _dp, _dp, _dp, _ip, _dp, ctypes.c_int]
        L.orc_mamba2_replay.argtypes = [ctypes.POINTER(_M2Dims), ctypes.c_int, _dp, _ip, _ip,
                                        _dp, _dp, _dp, ctypes.c_int, _dp, _dp, _dp, _dp, _dp,
                                        _dp, _dp, ctypes.c_int]
        L.orc_gdn_step.argtypes = [ctypes.POINTER(_GDims), _dp, _dp, _dp, _dp, _dp, _dp, _ip,
                                   _dp, ctypes.c_int]
        L.orc_gdn_replay.argtypes = [ctypes.POINTER(_GDims), ctypes.c_int, _dp, _ip, _ip, _dp,
                                     _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
        L.orc_mamba2_spec_round.argtypes = [ctypes.POINTER(_M2Dims), ctypes.c_int, _dp, _dp, _dp,
                                            _dp, ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _ip, _ip,
                                            _dp, ctypes.c_int]
        L.orc_kda_step.argtypes = [ctypes.POINTER(_GDims), _dp, _dp, _dp, _dp, _dp, _dp, _ip,
                                   _dp, ctypes.c_int]
        L.orc_kda_replay.argtypes = [ctypes.POINTER(_GDims), ctypes.c_int, _dp, _ip, _ip, _dp,
                                     _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
        L.orc_gdn_spec_round.argtypes = [ctypes.POINTER(_GDims), ctypes.c_int, _dp, _dp, _dp,
                                         _dp, _dp, _dp, _ip, _ip, _dp, ctypes.c_int]
        _lib = L
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    if a is None:
        return None
    if a.dtype == np.float64:
        return a.ctypes.data_as(_dp)
    return a.ctypes.data_as(_ip)


def default_threads() -> int:
    return lib().orc_default_threads()


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(float(v))


def round_f32(v: float) -> float:
    return lib().orc_round_f32(float(v))


def softplus(v: float) -> float:
    return lib().orc_softplus(float(v))


def round_slots(pool: np.ndarray, slots: Sequence[int], dtype: str) -> None:
    """Round the listed slots of a float64 pool (first axis = slot) in place."""
    assert pool.dtype == np.float64 and pool.flags.c_contiguous
    sl = _i32(slots)
    if len(sl) == 0:
        return
    lib().orc_round_slots(_p(pool), int(np.prod(pool.shape[1:])), _p(sl), len(sl),
                          2 if dtype == "bf16" else 1)


def philox4x32_10(ctr: Sequence[int], key: Sequence[int]) -> list:
    """Philox4x32-10 of a 4-word counter under a 2-word key (four uint32)."""
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib().orc_philox4x32_10(c, k, o)
    return list(o)


def round_bf16_sr(v: float, r: int) -> float:
    """Stochastic rounding of v (taken to float32 first) to bf16 with 16 random bits r."""
    return lib().orc_round_bf16_sr(float(v), int(r))


def sr_bits(seed: int, offset: int, e: int) -> int:
    """The 16 random bits element e of a state pool draws at (seed, offset)."""
    return lib().orc_sr_bits(int(seed), int(offset), int(e))


def round_slots_sr(pool: np.ndarray, slots: Sequence[int], seed: int, offset: int) -> None:
    """Stochastically round the listed slots of a float64 pool (first axis = slot)
    to bf16 in place, with the bits of generator (seed, offset)."""
    assert pool.dtype == np.float64 and pool.flags.c_contiguous
    sl = _i32(slots)
    if len(sl) == 0:
        return
    lib().orc_round_slots_sr(_p(pool), int(np.prod(pool.shape[1:])), _p(sl), len(sl),
                             int(seed), int(offset))


def _check(rc):
    if rc != 0:
        raise ValueError("oracle rejected the arguments (code %d)" % rc)


# ----------------------------------------------------------------------------- #
# thin wrappers                                                                 #
# ----------------------------------------------------------------------------- #

def mamba2_step(state, x, dt_raw, A, B, C, D, z=None, dt_bias=None, dt_softplus=True,
                ci=None, nthreads=0):
    """One full-state Mamba2 step, in place on ``state`` [slots,H,P,N] (float64).
    Returns y [batch,H,P]."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    x = _f64(x)
    b, H, P = x.shape
    N = state.shape[3]
    G = np.asarray(B).shape[1]
    ci = _i32(np.arange(b) if ci is None else ci)
    y = np.zeros((b, H, P))
    d = _M2Dims(b, H, P, N, G, state.shape[0])
    arrs = [_f64(dt_raw), None if dt_bias is None else _f64(dt_bias), _f64(A), _f64(B), _f64(C),
            _f64(D), None if z is None else _f64(z)]
    _check(lib().orc_mamba2_step(ctypes.byref(d), _p(state), _p(x), _p(arrs[0]), _p(arrs[1]),
                                 int(dt_softplus), _p(arrs[2]), _p(arrs[3]), _p(arrs[4]),
                                 _p(arrs[5]), _p(arrs[6]), _p(ci), _p(y), nthreads))
    return y


def mamba2_replay(L, S0, ci, wp, ex, edt_raw, A, eB, C, D, z=None, dt_bias=None,
                  dt_softplus=True, want_fold=False, nthreads=0):
    """ReplaySSM closed form: output of the current step (ring entry wp[b]) from the
    checkpoint S0 [slots,H,P,N] and per-row entries ex [b,L,H,P], edt_raw [b,L,H],
    eB [b,L,G,N]. Returns y [b,H,P] (and the folded state [b,H,P,N])."""
    S0 = _f64(S0)
    ex = _f64(ex)
    b, _, H, P = ex.shape
    N = S0.shape[3]
    G = np.asarray(eB).shape[2]
    y = np.zeros((b, H, P))
    Sf = np.zeros((b, H, P, N)) if want_fold else None
    d = _M2Dims(b, H, P, N, G, S0.shape[0])
    a = [_i32(ci), _i32(wp), _f64(edt_raw), None if dt_bias is None else _f64(dt_bias), _f64(A),
         _f64(eB), _f64(C), _f64(D), None if z is None else _f64(z)]
    _check(lib().orc_mamba2_replay(ctypes.byref(d), L, _p(S0), _p(a[0]), _p(a[1]), _p(ex),
                                   _p(a[2]), _p(a[3]), int(dt_softplus), _p(a[4]), _p(a[5]),
                                   _p(a[6]), _p(a[7]), _p(a[8]), _p(y), _p(Sf), nthreads))
    return (y, Sf) if want_fold else y


def gdn_step(state, q, k, v, beta, g, ci=None, nthreads=0):
    """One gated-delta-rule step in place on ``state`` [slots,HV,V,K]. Returns o [b,HV,V]."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, HK, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    ci = _i32(np.arange(b) if ci is None else ci)
    o = np.zeros((b, HV, V))
    d = _GDims(b, HV, HK, K, V, state.shape[0])
    be, gg = _f64(beta), _f64(g)
    _check(lib().orc_gdn_step(ctypes.byref(d), _p(state), _p(q), _p(k), _p(v), _p(be), _p(gg),
                              _p(ci), _p(o), nthreads))
    return o


def gdn_replay(L, S0, ci, wp, ek, ev, ebeta, eg, q, want_fold=False, want_d=False, nthreads=0):
    """ReplaySSM closed form for the gated delta rule. Entries ek [b,L,HK,K],
    ev [b,L,HV,V], ebeta/eg [b,L,HV]; q = current query [b,HK,K]. Returns o
    (and the folded state [b,HV,V,K], and d [b,L,HV,V])."""
    S0 = _f64(S0)
    ek, ev = _f64(ek), _f64(ev)
    b, _, HK, K = ek.shape
    HV, V = ev.shape[2], ev.shape[3]
    o = np.zeros((b, HV, V))
    Sf = np.zeros((b, HV, V, K)) if want_fold else None
    dd = np.zeros((b, L, HV, V)) if want_d else None
    d = _GDims(b, HV, HK, K, V, S0.shape[0])
    a = [_i32(ci), _i32(wp), _f64(ebeta), _f64(eg), _f64(q)]
    _check(lib().orc_gdn_replay(ctypes.byref(d), L, _p(S0), _p(a[0]), _p(a[1]), _p(ek), _p(ev),
                                _p(a[2]), _p(a[3]), _p(a[4]), _p(o), _p(Sf), _p(dd), nthreads))
    out = [o]
    if want_fold:
        out.append(Sf)
    if want_d:
        out.append(dd)
    return out[0] if len(out) == 1 else tuple(out)


def mamba2_spec_round(state, T, x, dt_raw, A, B, C, D, acc, z=None, dt_bias=None,
                      dt_softplus=True, ci=None, nthreads=0):
    """One Mamba2 verify round over T drafts (inputs [b,T,...]); keeps the state after
    acc[b] drafts. Returns per-draft outputs y [b,T,H,P]."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    x = _f64(x)
    b, T_, H, P = x.shape
    assert T_ == T
    N = state.shape[3]
    G = np.asarray(B).shape[2]
    ci = _i32(np.arange(b) if ci is None else ci)
    y = np.zeros((b, T, H, P))
    d = _M2Dims(b, H, P, N, G, state.shape[0])
    arrs = [_f64(dt_raw), None if dt_bias is None else _f64(dt_bias), _f64(A), _f64(B), _f64(C),
            _f64(D), None if z is None else _f64(z), _i32(acc)]
    _check(lib().orc_mamba2_spec_round(ctypes.byref(d), T, _p(state), _p(x), _p(arrs[0]),
                                       _p(arrs[1]), int(dt_softplus), _p(arrs[2]), _p(arrs[3]),
                                       _p(arrs[4]), _p(arrs[5]), _p(arrs[6]), _p(ci), _p(arrs[7]),
                                       _p(y), nthreads))
    return y


def kda_step(state, q, k, v, beta, a, ci=None, nthreads=0):
    """One KDA step (per-key-channel gate a [b,HV,K]) in place on ``state``
    [slots,HV,V,K]. Returns o [b,HV,V]."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, HK, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    ci = _i32(np.arange(b) if ci is None else ci)
    o = np.zeros((b, HV, V))
    d = _GDims(b, HV, HK, K, V, state.shape[0])
    be, aa = _f64(beta), _f64(a)
    _check(lib().orc_kda_step(ctypes.byref(d), _p(state), _p(q), _p(k), _p(v), _p(be), _p(aa),
                              _p(ci), _p(o), nthreads))
    return o


def kda_replay(L, S0, ci, wp, ek, ev, ebeta, ea, q, want_fold=False, want_d=False, nthreads=0):
    """ReplaySSM closed form of the KDA step. Entries ek [b,L,HK,K], ev [b,L,HV,V],
    ebeta [b,L,HV], ea [b,L,HV,K]; q = current query [b,HK,K]. Returns o (and the
    folded state [b,HV,V,K], and d [b,L,HV,V])."""
    S0 = _f64(S0)
    ek, ev = _f64(ek), _f64(ev)
    b, _, HK, K = ek.shape
    HV, V = ev.shape[2], ev.shape[3]
    o = np.zeros((b, HV, V))
    Sf = np.zeros((b, HV, V, K)) if want_fold else None
    dd = np.zeros((b, L, HV, V)) if want_d else None
    d = _GDims(b, HV, HK, K, V, S0.shape[0])
    a = [_i32(ci), _i32(wp), _f64(ebeta), _f64(ea), _f64(q)]
    _check(lib().orc_kda_replay(ctypes.byref(d), L, _p(S0), _p(a[0]), _p(a[1]), _p(ek), _p(ev),
                                _p(a[2]), _p(a[3]), _p(a[4]), _p(o), _p(Sf), _p(dd), nthreads))
    out = [o]
    if want_fold:
        out.append(Sf)
    if want_d:
        out.append(dd)
    return out[0] if len(out) == 1 else tuple(out)


def gdn_spec_round(state, T, q, k, v, beta, g, acc, ci=None, nthreads=0):
    """One verify round over T drafts (inputs [b,T,...]); keeps the state after acc[b]
    drafts. Returns per-draft outputs o [b,T,HV,V]."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, _, HK, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    ci = _i32(np.arange(b) if ci is None else ci)
    o = np.zeros((b, T, HV, V))
    d = _GDims(b, HV, HK, K, V, state.shape[0])
    be, gg, ac = _f64(beta), _f64(g), _i32(acc)
    _check(lib().orc_gdn_spec_round(ctypes.byref(d), T, _p(state), _p(q), _p(k), _p(v), _p(be),
                                    _p(gg), _p(ci), _p(ac), _p(o), nthreads))
    return o


# ----------------------------------------------------------------------------- #
# workload drivers (row-local slots)                                            #
# ----------------------------------------------------------------------------- #

def _local_ci(ci_full: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Row i of the sample owns local slot i; padding rows stay -1."""
    sel = ci_full[rows]
    return np.where(sel >= 0, np.arange(len(rows)), -1).astype(np.int32)


def mamba2_run(wl, rows: Optional[Sequence[int]] = None, steps: Optional[int] = None,
               mode: str = "replay", nthreads: int = 0, keep_y: bool = True) -> Dict:
    """Run a Mamba2 workload (history steps, then ``steps`` measured steps) for the
    given batch rows. mode "replay" rounds a slot to the state dtype when its row
    flushes; "full" rounds after every step.

    Returns dict: y [steps][n,H,P] (measured steps), row_wp / row_flush
    [steps][n] (int), ckpt [n,H,P,N] (the slot's stored state: the pool content
    at the end), state [n,H,P,N] (current exact state), slot_wp [n]."""
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    steps = wl.steps if steps is None else steps
    n = len(rows)
    ci_full = wl.cache_indices()
    prm = wl.params()
    state = np.stack([wl.slot_state(int(ci_full[r])) for r in rows]).astype(np.float64) \
        if n else np.zeros((0, wl.nheads, wl.headdim, wl.dstate))
    state = np.ascontiguousarray(state)
    ckpt = state.copy()
    slot_wp = [0] * n

    def one(inp, ci_loc, force):
        rw, rf = cursors.advance_standard(slot_wp, ci_loc, force, wl.L)
        y = mamba2_step(state, inp["x"][rows], inp["dt_raw"][rows], prm["A"], inp["B"][rows],
                        inp["C"][rows], prm["D"], None if inp["z"] is None else inp["z"][rows],
                        prm["dt_bias"], wl.dt_softplus, ci_loc, nthreads)
        if mode == "full":
            upd = [int(s) for s in ci_loc if s >= 0]
        else:
            upd = [int(ci_loc[i]) for i in range(n) if ci_loc[i] >= 0 and rf[i]]
        round_slots(state, upd, wl.state_dtype)
        for s in upd:
            ckpt[s] = state[s]
        return y, rw, rf

    for j in range(wl.max_history()):
        one(wl.history_inputs(j), _local_ci(wl.history_ci(j), rows), None)
    ys, wps, fls = [], [], []
    for t in range(steps):
        inp = wl.step_inputs(t)
        force = wl.force_mask(t)
        y, rw, rf = one(inp, _local_ci(ci_full, rows), None if force is None else force[rows])
        if keep_y:
            ys.append(y)
        wps.append(rw)
        fls.append(rf)
    return dict(y=ys, row_wp=np.array(wps, dtype=np.int64).reshape(steps, n),
                row_flush=np.array(fls, dtype=np.int64).reshape(steps, n), ckpt=ckpt,
                state=state, slot_wp=np.array(slot_wp))


def gdn_run(wl, rows: Optional[Sequence[int]] = None, steps: Optional[int] = None,
            mode: str = "replay", nthreads: int = 0, keep_o: bool = True) -> Dict:
    """Gated delta net counterpart of mamba2_run (fp32 state)."""
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    steps = wl.steps if steps is None else steps
    n = len(rows)
    ci_full = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci_full[r])) for r in rows]).astype(np.float64))
    ckpt = state.copy()
    slot_wp = [0] * n

    def one(inp, ci_loc, force):
        rw, rf = cursors.advance_standard(slot_wp, ci_loc, force, wl.L)
        o = gdn_step(state, inp["q"][rows], inp["k"][rows], inp["v"][rows], inp["beta"][rows],
                     inp["g"][rows], ci_loc, nthreads)
        if mode == "full":
            upd = [int(s) for s in ci_loc if s >= 0]
        else:
            upd = [int(ci_loc[i]) for i in range(n) if ci_loc[i] >= 0 and rf[i]]
        round_slots(state, upd, "fp32")
        for s in upd:
            ckpt[s] = state[s]
        return o, rw, rf

    for j in range(wl.max_history()):
        one(wl.history_inputs(j), _local_ci(wl.history_ci(j), rows), None)
    os_, wps, fls = [], [], []
    for t in range(steps):
        inp = wl.step_inputs(t)
        force = wl.force_mask(t)
        o, rw, rf = one(inp, _local_ci(ci_full, rows), None if force is None else force[rows])
        if keep_o:
            os_.append(o)
        wps.append(rw)
        fls.append(rf)
    return dict(o=os_, row_wp=np.array(wps, dtype=np.int64).reshape(steps, n),
                row_flush=np.array(fls, dtype=np.int64).reshape(steps, n), ckpt=ckpt,
                state=state, slot_wp=np.array(slot_wp))


def mamba2_spec_run(wl, rows: Optional[Sequence[int]] = None, rounds: Optional[int] = None,
                    nthreads: int = 0) -> Dict:
    """Mamba2 speculative verify workload (the gdn_spec_run protocol): the checkpoint
    is stored, rounded to the state dtype, when a round starts with the slot's flush
    flag set, which is when the fold writes it. Returns dict: y [rounds][n,T,H,P],
    ckpt, state, cnt / base / flush [rounds+1][n]."""
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    rounds = wl.rounds if rounds is None else rounds
    n = len(rows)
    ci_full = wl.cache_indices()
    prm = wl.params()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci_full[r])) for r in rows]).astype(np.float64))
    ckpt = state.copy()
    cnt, base, flush = [0] * n, [0] * n, [0] * n
    ci_loc = _local_ci(ci_full, rows)
    outs, hist = [], []
    for r in range(rounds):
        hist.append((list(cnt), list(base), list(flush)))
        fold = [i for i in range(n) if ci_loc[i] >= 0 and flush[i]]
        round_slots(state, fold, wl.state_dtype)
        for s in fold:
            ckpt[s] = state[s]
        inp = wl.round_inputs(r)
        acc = wl.accepted(r)[rows]
        y = mamba2_spec_round(state, wl.T, inp["x"][rows], inp["dt_raw"][rows], prm["A"],
                              inp["B"][rows], inp["C"][rows], prm["D"], acc,
                              None if inp["z"] is None else inp["z"][rows], prm["dt_bias"],
                              wl.dt_softplus, ci_loc, nthreads)
        outs.append(y)
        cursors.spec_commit(cnt, base, flush, ci_loc, acc, wl.L, wl.T)
    hist.append((list(cnt), list(base), list(flush)))
    h = np.array(hist, dtype=np.int64)
    return dict(y=outs, ckpt=ckpt, state=state, cnt=h[:, 0], base=h[:, 1], flush=h[:, 2])


def kda_run(wl, rows: Optional[Sequence[int]] = None, steps: Optional[int] = None,
            mode: str = "replay", nthreads: int = 0, keep_o: bool = True) -> Dict:
    """KDA counterpart of gdn_run (fp32 state; inputs carry the gate vector "a")."""
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    steps = wl.steps if steps is None else steps
    n = len(rows)
    ci_full = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci_full[r])) for r in rows]).astype(np.float64))
    ckpt = state.copy()
    slot_wp = [0] * n

    def one(inp, ci_loc, force):
        rw, rf = cursors.advance_standard(slot_wp, ci_loc, force, wl.L)
        o = kda_step(state, inp["q"][rows], inp["k"][rows], inp["v"][rows], inp["beta"][rows],
                     inp["a"][rows], ci_loc, nthreads)
        if mode == "full":
            upd = [int(s) for s in ci_loc if s >= 0]
        else:
            upd = [int(ci_loc[i]) for i in range(n) if ci_loc[i] >= 0 and rf[i]]
        round_slots(state, upd, "fp32")
        for s in upd:
            ckpt[s] = state[s]
        return o, rw, rf

    for j in range(wl.max_history()):
        one(wl.history_inputs(j), _local_ci(wl.history_ci(j), rows), None)
    os_, wps, fls = [], [], []
    for t in range(steps):
        inp = wl.step_inputs(t)
        force = wl.force_mask(t)
        o, rw, rf = one(inp, _local_ci(ci_full, rows), None if force is None else force[rows])
        if keep_o:
            os_.append(o)
        wps.append(rw)
        fls.append(rf)
    return dict(o=os_, row_wp=np.array(wps, dtype=np.int64).reshape(steps, n),
                row_flush=np.array(fls, dtype=np.int64).reshape(steps, n), ckpt=ckpt,
                state=state, slot_wp=np.array(slot_wp))


def gdn_spec_run(wl, rows: Optional[Sequence[int]] = None, rounds: Optional[int] = None,
                 nthreads: int = 0) -> Dict:
    """Speculative verify workload: per round, per-draft outputs and the commit of the
    accepted prefix. The checkpoint is stored (rounded to fp32) when a round starts
    with the slot's flush flag set, which is when the exact fold writes it.

    Returns dict: o [rounds][n,T,HV,V], ckpt, state, and the cursor history
    cnt / base / flush [rounds+1][n] (before each round, and at the end)."""
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    rounds = wl.rounds if rounds is None else rounds
    n = len(rows)
    ci_full = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci_full[r])) for r in rows]).astype(np.float64))
    ckpt = state.copy()
    cnt, base, flush = [0] * n, [0] * n, [0] * n
    ci_loc = _local_ci(ci_full, rows)
    outs, hist = [], []
    for r in range(rounds):
        hist.append((list(cnt), list(base), list(flush)))
        fold = [i for i in range(n) if ci_loc[i] >= 0 and flush[i]]
        round_slots(state, fold, "fp32")
        for s in fold:
            ckpt[s] = state[s]
        inp = wl.round_inputs(r)
        acc = wl.accepted(r)[rows]
        o = gdn_spec_round(state, wl.T, inp["q"][rows], inp["k"][rows], inp["v"][rows],
                           inp["beta"][rows], inp["g"][rows], acc, ci_loc, nthreads)
        outs.append(o)
        cursors.spec_commit(cnt, base, flush, ci_loc, acc, wl.L, wl.T)
    hist.append((list(cnt), list(base), list(flush)))
    h = np.array(hist, dtype=np.int64)  # [rounds+1, 3, n]
    return dict(o=outs, ckpt=ckpt, state=state, cnt=h[:, 0], base=h[:, 1], flush=h[:, 2])
