"""Helpers for the GPU parity tests: run a seeded workload through the C ABI
(via the decode-step runners) and compare with the oracle.

Error metric (both floating-point tolerances are those of the method's stated
bar: 1e-4 for an fp32 state, 2e-3 for a bf16 state):
    e = max over elements |gpu - ref| / max(1, |ref|)
For stored bf16 states a disagreement of exactly one bf16 spacing is also
accepted: the GPU rounds an fp32 accumulation and the oracle an exact float64
value, so where the exact value lies within float32 accumulation error of a
rounding midpoint the two round to neighbouring bf16 values.
"""
import numpy as np
import torch

import oracle
from oracle import cursors


def tol_for(state_dtype: str) -> float:
    return 1e-4 if state_dtype == "fp32" else 2e-3


def torch_dt(name: str) -> torch.dtype:
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if gpu.size == 0:
        return 0.0
    return float(np.max(np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))))


def bf16_spacing(ref) -> np.ndarray:
    """Distance from |ref| (a bf16 value) to the next bf16 value away from zero."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def state_ok(gpu, ref, state_dtype: str):
    """(ok, e, flips): stored-state comparison with the one-spacing allowance for bf16."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = tol_for(state_dtype)
    d = np.abs(gpu - ref)
    lim = tol * np.maximum(1.0, np.abs(ref))
    if state_dtype == "bf16":
        within = (d <= lim) | (d <= bf16_spacing(ref) * 1.0000001)
        flips = int(np.count_nonzero(d > 0))
    else:
        within = d <= lim
        flips = 0
    e = float(np.max(d / np.maximum(1.0, np.abs(ref)))) if d.size else 0.0
    return bool(np.all(within)), e, flips


def row_chunks(rows, size):
    """Consecutive slices of `rows` of at most `size` entries, as (start, rows) pairs.
    Rows are independent, so the oracle runs one chunk at a time and its float64
    state stays bounded at the full configurations."""
    rows = np.asarray(rows)
    return [(i, rows[i:i + size]) for i in range(0, len(rows), size)]


def to_dev(a, dtype, device="cuda"):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


# --------------------------------------------------------------------------- #
# Mamba2                                                                      #
# --------------------------------------------------------------------------- #

def make_mamba2_decoder(wl, out_dtype=torch.float32, full_state=False, max_batch=None,
                        sr_seed=None):
    from ssm_linear_attention_gb300 import Mamba2FullStateDecoder, Mamba2ReplayDecoder
    prm = wl.params()
    kw = dict(A=prm["A"], D=prm["D"], dt_bias=prm["dt_bias"], dt_softplus=wl.dt_softplus,
              state_dtype=torch_dt(wl.state_dtype), act_dtype=torch_dt(wl.act_dtype),
              out_dtype=out_dtype, sr_seed=sr_seed)
    mb = wl.batch if max_batch is None else max_batch
    if full_state:
        dec = Mamba2FullStateDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.num_slots,
                                     max(mb, 1), **kw)
    else:
        dec = Mamba2ReplayDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.L,
                                  wl.num_slots, max(mb, 1), **kw)
    for s in wl.cache_indices():
        dec.state[int(s)] = to_dev(wl.slot_state(int(s)), dec.state.dtype)
    return dec


def mamba2_inputs_dev(wl, inp):
    ad = torch_dt(wl.act_dtype)
    return (to_dev(inp["x"], ad), to_dev(inp["dt_raw"], torch.float32), to_dev(inp["B"], ad),
            to_dev(inp["C"], ad), to_dev(inp["z"], ad))


def run_gpu_mamba2(wl, steps=None, out_dtype=torch.float32, full_state=False, rows=None,
                   keep_all_y=False):
    """History steps, then `steps` measured steps. Returns dict with y (per step,
    rows subset, float64 numpy), row_wp / row_flush (all rows), the decoder."""
    steps = wl.steps if steps is None else steps
    dec = make_mamba2_decoder(wl, out_dtype, full_state)
    ci = wl.cache_indices()
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    for j in range(wl.max_history()):
        x, dt, Bm, C, z = mamba2_inputs_dev(wl, wl.history_inputs(j))
        hci = to_dev(wl.history_ci(j), torch.int32)
        if full_state:
            dec.step(x, dt, Bm, C, z, hci)
        else:
            dec.step(x, dt, Bm, C, z, hci)
    ci_d = to_dev(ci, torch.int32)
    ys, wps, fls = [], [], []
    for t in range(steps):
        x, dt, Bm, C, z = mamba2_inputs_dev(wl, wl.step_inputs(t))
        if full_state:
            y = dec.step(x, dt, Bm, C, z, ci_d)
        else:
            f = wl.force_mask(t)
            y = dec.step(x, dt, Bm, C, z, ci_d, None if f is None else to_dev(f, torch.uint8))
            wps.append(dec.row_wp[: wl.batch].cpu().numpy().copy())
            fls.append(dec.row_flush[: wl.batch].cpu().numpy().copy())
        # float32 on the host (exact for fp32 and bf16 outputs); compared in float64
        ys.append((y if keep_all_y else y[torch.as_tensor(rows, device=y.device)]).float().cpu()
                  .numpy())
    torch.cuda.synchronize()
    return dict(y=ys, row_wp=np.array(wps), row_flush=np.array(fls), dec=dec)


def cursor_reference(wl, steps=None):
    """Integer cursor model over history + steps for every row (oracle side)."""
    steps = wl.steps if steps is None else steps
    slot_wp = [0] * wl.num_slots
    for j in range(wl.max_history()):
        cursors.advance_standard(slot_wp, wl.history_ci(j), None, wl.L)
    wps, fls = [], []
    ci = wl.cache_indices()
    for t in range(steps):
        rw, rf = cursors.advance_standard(slot_wp, ci, wl.force_mask(t), wl.L)
        wps.append(rw)
        fls.append(rf)
    return np.array(wps), np.array(fls), np.array(slot_wp)


# --------------------------------------------------------------------------- #
# gated delta net                                                             #
# --------------------------------------------------------------------------- #

def make_gdn_decoder(wl, out_dtype=torch.float32, full_state=False, max_batch=None):
    from ssm_linear_attention_gb300 import GDNFullStateDecoder, GDNReplayDecoder
    ad = torch_dt(wl.act_dtype)
    mb = max(wl.batch if max_batch is None else max_batch, 1)
    if full_state:
        dec = GDNFullStateDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim,
                                  wl.num_slots, mb, act_dtype=ad, out_dtype=out_dtype)
    else:
        dec = GDNReplayDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.L,
                               wl.num_slots, mb, act_dtype=ad, out_dtype=out_dtype)
    for s in wl.cache_indices():
        dec.state[int(s)] = to_dev(wl.slot_state(int(s)), torch.float32)
    return dec


def gdn_inputs_dev(wl, inp):
    ad = torch_dt(wl.act_dtype)
    return (to_dev(inp["q"], ad), to_dev(inp["k"], ad), to_dev(inp["v"], ad),
            to_dev(inp["beta"], torch.float32), to_dev(inp["g"], torch.float32))


def run_gpu_gdn(wl, steps=None, out_dtype=torch.float32, full_state=False, rows=None):
    steps = wl.steps if steps is None else steps
    dec = make_gdn_decoder(wl, out_dtype, full_state)
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    for j in range(wl.max_history()):
        q, k, v, be, g = gdn_inputs_dev(wl, wl.history_inputs(j))
        dec.step(q, k, v, be, g, to_dev(wl.history_ci(j), torch.int32))
    ci_d = to_dev(wl.cache_indices(), torch.int32)
    os_, wps, fls = [], [], []
    sel = torch.as_tensor(rows, device="cuda")
    for t in range(steps):
        q, k, v, be, g = gdn_inputs_dev(wl, wl.step_inputs(t))
        if full_state:
            o = dec.step(q, k, v, be, g, ci_d)
        else:
            f = wl.force_mask(t)
            o = dec.step(q, k, v, be, g, ci_d, None if f is None else to_dev(f, torch.uint8))
            wps.append(dec.row_wp[: wl.batch].cpu().numpy().copy())
            fls.append(dec.row_flush[: wl.batch].cpu().numpy().copy())
        os_.append(o[sel].float().cpu().numpy())
    torch.cuda.synchronize()
    return dict(o=os_, row_wp=np.array(wps), row_flush=np.array(fls), dec=dec)


def run_gpu_spec(wl, rounds=None, out_dtype=torch.float32, rows=None):
    from ssm_linear_attention_gb300 import GDNSpecVerifier
    rounds = wl.rounds if rounds is None else rounds
    ad = torch_dt(wl.act_dtype)
    ver = GDNSpecVerifier(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.L,
                          wl.T, wl.num_slots, max(wl.batch, 1), act_dtype=ad, out_dtype=out_dtype)
    ci = wl.cache_indices()
    for s in ci:
        ver.state[int(s)] = to_dev(wl.slot_state(int(s)), torch.float32)
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    sel = torch.as_tensor(rows, device="cuda")
    ci_d = to_dev(ci, torch.int32)
    cidx = torch.as_tensor(ci.astype(np.int64), device="cuda")
    outs, curs = [], []
    for r in range(rounds):
        curs.append((ver.slot_cnt[cidx].cpu().numpy(), ver.slot_base[cidx].cpu().numpy(),
                     ver.slot_flush[cidx].cpu().numpy()))
        q, k, v, be, g = gdn_inputs_dev(wl, wl.round_inputs(r))
        o = ver.verify(q, k, v, be, g, ci_d)
        outs.append(o[sel].float().cpu().numpy())
        ver.commit(ci_d, to_dev(wl.accepted(r), torch.int32))
    curs.append((ver.slot_cnt[cidx].cpu().numpy(), ver.slot_base[cidx].cpu().numpy(),
                 ver.slot_flush[cidx].cpu().numpy()))
    torch.cuda.synchronize()
    c = np.array(curs, dtype=np.int64)   # [rounds+1, 3, batch]
    return dict(o=outs, cnt=c[:, 0], base=c[:, 1], flush=c[:, 2], ver=ver)


# --------------------------------------------------------------------------- #
# KDA (per-key-channel gate)                                                  #
# --------------------------------------------------------------------------- #

def make_kda_decoder(wl, out_dtype=torch.float32, full_state=False, max_batch=None):
    from ssm_linear_attention_gb300 import KDAFullStateDecoder, KDAReplayDecoder
    ad = torch_dt(wl.act_dtype)
    mb = max(wl.batch if max_batch is None else max_batch, 1)
    if full_state:
        dec = KDAFullStateDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim,
                                  wl.num_slots, mb, act_dtype=ad, out_dtype=out_dtype)
    else:
        dec = KDAReplayDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.L,
                               wl.num_slots, mb, act_dtype=ad, out_dtype=out_dtype)
    for s in wl.cache_indices():
        dec.state[int(s)] = to_dev(wl.slot_state(int(s)), torch.float32)
    return dec


def kda_inputs_dev(wl, inp):
    ad = torch_dt(wl.act_dtype)
    return (to_dev(inp["q"], ad), to_dev(inp["k"], ad), to_dev(inp["v"], ad),
            to_dev(inp["beta"], torch.float32), to_dev(inp["a"], torch.float32))


def run_gpu_kda(wl, steps=None, out_dtype=torch.float32, full_state=False, rows=None,
                staged=False):
    steps = wl.steps if steps is None else steps
    dec = make_kda_decoder(wl, out_dtype, full_state)
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    run = dec.step_staged if staged else dec.step
    for j in range(wl.max_history()):
        q, k, v, be, a = kda_inputs_dev(wl, wl.history_inputs(j))
        (dec.step if full_state else run)(q, k, v, be, a, to_dev(wl.history_ci(j), torch.int32))
    ci_d = to_dev(wl.cache_indices(), torch.int32)
    os_, wps, fls = [], [], []
    sel = torch.as_tensor(rows, device="cuda")
    for t in range(steps):
        q, k, v, be, a = kda_inputs_dev(wl, wl.step_inputs(t))
        if full_state:
            o = dec.step(q, k, v, be, a, ci_d)
        else:
            f = wl.force_mask(t)
            o = run(q, k, v, be, a, ci_d, None if f is None else to_dev(f, torch.uint8))
            wps.append(dec.row_wp[: wl.batch].cpu().numpy().copy())
            fls.append(dec.row_flush[: wl.batch].cpu().numpy().copy())
        os_.append(o[sel].float().cpu().numpy())
    torch.cuda.synchronize()
    return dict(o=os_, row_wp=np.array(wps), row_flush=np.array(fls), dec=dec)


# --------------------------------------------------------------------------- #
# Mamba2 speculative verify                                                   #
# --------------------------------------------------------------------------- #

def run_gpu_m2spec(wl, rounds=None, out_dtype=torch.float32, rows=None):
    from ssm_linear_attention_gb300 import Mamba2SpecVerifier
    rounds = wl.rounds if rounds is None else rounds
    prm = wl.params()
    ad = torch_dt(wl.act_dtype)
    ver = Mamba2SpecVerifier(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.L, wl.T,
                             wl.num_slots, max(wl.batch, 1), prm["A"], prm["D"], prm["dt_bias"],
                             wl.dt_softplus, state_dtype=torch_dt(wl.state_dtype), act_dtype=ad,
                             out_dtype=out_dtype)
    ci = wl.cache_indices()
    for s in ci:
        ver.state[int(s)] = to_dev(wl.slot_state(int(s)), ver.state.dtype)
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    sel = torch.as_tensor(rows, device="cuda")
    ci_d = to_dev(ci, torch.int32)
    cidx = torch.as_tensor(ci.astype(np.int64), device="cuda")
    outs, curs = [], []
    for r in range(rounds):
        curs.append((ver.slot_cnt[cidx].cpu().numpy(), ver.slot_base[cidx].cpu().numpy(),
                     ver.slot_flush[cidx].cpu().numpy()))
        inp = wl.round_inputs(r)
        y = ver.verify(to_dev(inp["x"], ad), to_dev(inp["dt_raw"], torch.float32),
                       to_dev(inp["B"], ad), to_dev(inp["C"], ad), to_dev(inp["z"], ad), ci_d)
        outs.append(y[sel].float().cpu().numpy())
        ver.commit(ci_d, to_dev(wl.accepted(r), torch.int32))
    curs.append((ver.slot_cnt[cidx].cpu().numpy(), ver.slot_base[cidx].cpu().numpy(),
                 ver.slot_flush[cidx].cpu().numpy()))
    torch.cuda.synchronize()
    c = np.array(curs, dtype=np.int64)
    return dict(y=outs, cnt=c[:, 0], base=c[:, 1], flush=c[:, 2], ver=ver)
