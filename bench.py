"""Benchmark: ReplaySSM Mamba2 decode at batch 512 on GB300.

Workload (one step = one decode step of one layer for the whole batch: cursor
advance, ring append, precompute, output/flush): batch 512, nheads 128,
headdim 64, dstate 128, ngroups 8, ring L 16, bf16 checkpoint pool of 1024
slots ~ N(0, 0.1), cache indices = first 512 of a seeded permutation,
desynchronised initial write_pos ~ U{0..15}, x/z/B/C bf16, dt/A/D fp32, bf16
output. 64 distinct seeded input sets are resident in HBM and cycled.

Prints ONE JSON line (rank 0):
  value       decode rows/s over all ranks (device-timed, inputs resident)
  e2e         same metric through the public API with pinned host buffers:
              host->device copy of each step's inputs and device->host copy of
              y inside the timed region
  roofline    output kernel: algorithmic bytes per launch / CUDA-event duration
              of that kernel inside the timed region, against the measured HBM
              copy bandwidth
  cpu_baseline  the float64 oracle (full recurrence) on this host's cores over a
              bounded sample of the same workload
  full_state  the in-house conventional kernel (whole state read+written per
              step) on an identical pool, same inputs

--impl reference runs the oracle arm (the only reference implementation this
method has here) on the same metric and workload.
Multi-GPU (torchrun): every rank runs its own independent replica of the
workload (rows are independent; no collective on the data path), timing is
max over ranks, value sums the rows of all ranks.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode rows/s and µs/step at batch 512; achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "rows/s"
WORKLOAD = ("mamba2 replayssm decode: batch 512, nheads 128, headdim 64, dstate 128, ngroups 8, "
            "L 16, bf16 state pool 1024 slots, desync write_pos U{0..15}, 64 steps cycled")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--input-sets", type=int, default=64)
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-full-state", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=512)
    ap.add_argument("--num-slots", type=int, default=1024)
    return ap.parse_args()


# --------------------------------------------------------------------------- #
# distributed plumbing                                                        #
# --------------------------------------------------------------------------- #

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def shard_seed(base: int, rank: int) -> int:
    """Independent replica per rank: same workload recipe, own seed."""
    return base + 1000003 * rank


# --------------------------------------------------------------------------- #
# clocks                                                                      #
# --------------------------------------------------------------------------- #

_CLK_Q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
          "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
          "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, period_ms=100):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + _CLK_Q, "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self, bus_id=None):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 7]
        if bus_id:
            mine = [r for r in rows if bus_id.lower()[-7:] in r[0].lower()]
            rows = mine or rows
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" == r[4 + i].strip()})
        loaded = [s for s in sm if mx and s > 0.3 * max(mx)]
        return {"sm_mhz": float(np.median(loaded or sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sm)}


# --------------------------------------------------------------------------- #
# byte accounting                                                             #
# --------------------------------------------------------------------------- #

def output_kernel_bytes(wl, row_wp, row_flush, out_bytes=2):
    """Algorithmic bytes one output-kernel launch must move for the given per-row
    cursors: checkpoint read, ring x entries 0..w, C, z, y, and on flush rows the
    state write and ring B entries 0..w. The precompute tables are excluded."""
    H, P, N, G = wl.nheads, wl.headdim, wl.dstate, wl.ngroups
    sS = 2 if wl.state_dtype == "bf16" else 4
    sa = 2 if wl.act_dtype == "bf16" else 4
    w1 = row_wp.astype(np.int64) + 1
    f = row_flush.astype(np.int64)
    per_row = (H * P * N * sS + w1 * H * P * sa + G * N * sa + H * P * sa + H * P * out_bytes
               + f * (H * P * N * sS + w1 * G * N * sa))
    return int(per_row.sum())


def step_bytes(wl, row_wp, row_flush, out_bytes=2):
    """Algorithmic bytes of one whole ReplaySSM step: checkpoint read, ring entries
    before the current one (x, dt, B), this step's inputs (x, z, B, C, dt_raw),
    y, the ring append, and the flush write."""
    H, P, N, G = wl.nheads, wl.headdim, wl.dstate, wl.ngroups
    sS = 2 if wl.state_dtype == "bf16" else 4
    sa = 2 if wl.act_dtype == "bf16" else 4
    w = row_wp.astype(np.int64)
    f = row_flush.astype(np.int64)
    entry = H * P * sa + 4 * H + G * N * sa
    per_row = (H * P * N * sS + w * entry + 2 * H * P * sa + 2 * G * N * sa + 4 * H
               + H * P * out_bytes + entry + f * H * P * N * sS)
    return int(per_row.sum())


def full_state_bytes(wl, batch, out_bytes=2):
    H, P, N, G = wl.nheads, wl.headdim, wl.dstate, wl.ngroups
    sS = 2 if wl.state_dtype == "bf16" else 4
    sa = 2 if wl.act_dtype == "bf16" else 4
    return batch * (2 * H * P * N * sS + 2 * H * P * sa + 2 * G * N * sa + 4 * H + H * P * out_bytes)


def simulate_cursors(slot_wp, ci, L, k):
    """Per-step (row_wp, row_flush) for k standard steps without forced flushes
    (bookkeeping for the byte count; the kernels compute their own)."""
    wp = slot_wp.copy()
    out = []
    for _ in range(k):
        w = wp[ci]
        f = (w == L - 1).astype(np.int64)
        out.append((w.copy(), f))
        wp[ci] = np.where(f == 1, 0, w + 1)
    return out


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record(kernel_src):
    """DRAM bytes per launch of the output kernel from the committed ncu summary,
    valid only while the kernel source is unchanged (sha256 recorded beside it)."""
    src = os.path.join(ROOT, "ssm_linear_attention_gb300", "csrc", kernel_src)
    prof = os.path.join(ROOT, "profiles", "mamba2_output_kernel_batch512.md")
    if not (os.path.exists(src) and os.path.exists(prof)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    rec = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith(("source_sha256", "traffic_bytes_per_launch")):
            k, v = line.split(":", 1)
            rec[k.strip().strip("`- ")] = v.strip().strip("`")
    if rec.get("source_sha256") == sha and rec.get("traffic_bytes_per_launch"):
        return int(rec["traffic_bytes_per_launch"])
    return None


# --------------------------------------------------------------------------- #
# CPU baseline (the oracle)                                                   #
# --------------------------------------------------------------------------- #

def cpu_oracle_rate(wl, seconds, max_rows=64):
    """Time the float64 oracle recurrence on a sample of rows until `seconds` of
    work have run (at least two steps). Returns (rows/s, threads, sample text)."""
    import oracle
    nth = oracle.default_threads()
    rows = np.arange(min(max_rows, wl.batch))
    prm = wl.params()
    ci = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci[r])) for r in rows]).astype(np.float64))
    inputs = []
    for t in range(4):
        inp = wl.step_inputs(t)
        inputs.append({k: (None if v is None else np.ascontiguousarray(v[rows], dtype=np.float64))
                       for k, v in inp.items()})
    loc = np.arange(len(rows), dtype=np.int32)
    done, t0 = 0, time.perf_counter()
    while True:
        inp = inputs[done % len(inputs)]
        oracle.mamba2_step(state, inp["x"], inp["dt_raw"], prm["A"], inp["B"], inp["C"], prm["D"],
                           inp["z"], prm["dt_bias"], True, loc, nth)
        done += 1
        el = time.perf_counter() - t0
        if done >= 2 and el >= seconds:
            break
    rate = done * len(rows) / el
    sample = "%d rows x %d steps of the float64 full recurrence (%.1f s)" % (len(rows), done, el)
    return rate, nth, sample


# --------------------------------------------------------------------------- #
# main arm                                                                    #
# --------------------------------------------------------------------------- #

def run_ours(args, dist):
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    dev = torch.device("cuda", dist.local if dist.world > 1 else 0)
    torch.cuda.set_device(dev)
    ssm.lib()
    wl = W.mamba2_large(batch=args.batch, num_slots=args.num_slots,
                        seed=shard_seed(args.seed, dist.rank))
    prm = wl.params()
    bf = torch.bfloat16
    ci_np = wl.cache_indices()
    ci = torch.from_numpy(ci_np).to(dev)

    dec = ssm.Mamba2ReplayDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.L,
                                  wl.num_slots, wl.batch, prm["A"], prm["D"], prm["dt_bias"],
                                  state_dtype=bf, act_dtype=bf, out_dtype=bf, device=dev)
    for s in ci_np:
        dec.state[int(s)] = torch.from_numpy(wl.slot_state(int(s))).to(dev, bf)

    def to_dev(inp):
        return [torch.from_numpy(inp[k]).to(dev, bf if k != "dt_raw" else torch.float32)
                for k in ("x", "dt_raw", "B", "C", "z")]

    for j in range(wl.max_history()):
        x, dt, Bm, C, z = to_dev(wl.history_inputs(j))
        dec.step(x, dt, Bm, C, z, torch.from_numpy(wl.history_ci(j)).to(dev))
    sets = [to_dev(wl.step_inputs(t)) for t in range(args.input_sets)]
    torch.cuda.synchronize()

    def one_step(k):
        x, dt, Bm, C, z = sets[k % len(sets)]
        dec.advance(ci)
        dec.append(x, dt, Bm, ci)
        dec.precompute(C, ci)
        return dec.output(C, z, ci)

    for k in range(args.warmup):
        one_step(k)
    torch.cuda.synchronize()
    slot_wp0 = dec.slot_wp.cpu().numpy().astype(np.int64)

    K = args.steps
    stream = torch.cuda.current_stream()
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler()
    time.sleep(0.3)
    start.record(stream)
    for k in range(K):
        x, dt, Bm, C, z = sets[(k + args.warmup) % len(sets)]
        dec.advance(ci)
        dec.append(x, dt, Bm, ci)
        dec.precompute(C, ci)
        ev_a[k].record(stream)
        dec.output(C, z, ci)
        ev_b[k].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    bus = None
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%08x:%02x:%02x" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id, p.pci_device_id)
    except Exception:
        bus = None
    clocks = clk.stop(bus)
    elapsed_ms = start.elapsed_time(end)
    out_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]
    max_ms = dist.max(elapsed_ms)
    assert int(dec.dev_err.abs().sum().item()) == 0, "device error flag set during the bench"

    ms_step = max_ms / K
    rows_s = dist.world * wl.batch / (ms_step * 1e-3)

    # algorithmic bytes
    curs = simulate_cursors(slot_wp0, ci_np, wl.L, K)
    out_b = np.mean([output_kernel_bytes(wl, w, f) for w, f in curs])
    step_b = np.mean([step_bytes(wl, w, f) for w, f in curs])
    out_avg_ms = float(np.mean(out_ms))
    peak, peak_kind = read_peaks()
    achieved = out_b / (out_avg_ms * 1e-3) / 1e9
    traffic = traffic_record("mamba2.cu")

    # end to end through the public API with pinned host buffers
    e2e = None
    if args.e2e_steps > 0:
        host_sets = []
        for t in range(min(8, args.input_sets)):
            inp = wl.step_inputs(t)
            hs = {}
            for k2 in ("x", "dt_raw", "B", "C", "z"):
                tt = torch.from_numpy(inp[k2]).to(bf if k2 != "dt_raw" else torch.float32)
                hs[k2] = tt.pin_memory()
            host_sets.append(hs)
        dsts = {k2: v.clone() for k2, v in zip(("x", "dt_raw", "B", "C", "z"), sets[0])}
        y_host = torch.empty(wl.batch, wl.nheads, wl.headdim, dtype=bf).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host_sets[0].values())
        d2h = y_host.numel() * y_host.element_size()
        for k in range(3):
            hs = host_sets[k % len(host_sets)]
            for k2 in dsts:
                dsts[k2].copy_(hs[k2], non_blocking=True)
            y = dec.step(dsts["x"], dsts["dt_raw"], dsts["B"], dsts["C"], dsts["z"], ci)
            y_host.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(args.e2e_steps):
            hs = host_sets[k % len(host_sets)]
            for k2 in dsts:
                dsts[k2].copy_(hs[k2], non_blocking=True)
            y = dec.step(dsts["x"], dsts["dt_raw"], dsts["B"], dsts["C"], dsts["z"], ci)
            y_host.copy_(y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = dist.max(e0.elapsed_time(e1)) / args.e2e_steps
        e2e = {"value": dist.world * wl.batch / (e_ms * 1e-3), "unit": UNIT,
               "ms_per_step": e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    # the in-house conventional kernel on an identical pool
    full = None
    if not args.no_full_state:
        fdec = ssm.Mamba2FullStateDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups,
                                          wl.num_slots, wl.batch, prm["A"], prm["D"],
                                          prm["dt_bias"], state_dtype=bf, act_dtype=bf,
                                          out_dtype=bf, device=dev)
        fdec.state.copy_(dec.state)
        del dec
        for k in range(args.warmup):
            x, dt, Bm, C, z = sets[k % len(sets)]
            fdec.step(x, dt, Bm, C, z, ci)
        torch.cuda.synchronize()
        Kf = max(50, K // 4)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist.barrier()
        f0.record(stream)
        for k in range(Kf):
            x, dt, Bm, C, z = sets[k % len(sets)]
            fdec.step(x, dt, Bm, C, z, ci)
        f1.record(stream)
        torch.cuda.synchronize()
        f_ms = dist.max(f0.elapsed_time(f1)) / Kf
        fb = full_state_bytes(wl, wl.batch)
        full = {"ms_per_step": f_ms, "us_per_step": f_ms * 1e3,
                "rows_per_s": dist.world * wl.batch / (f_ms * 1e-3),
                "achieved_gbs": fb / (f_ms * 1e-3) / 1e9, "bytes_per_step": fb,
                "replay_speedup": f_ms / ms_step}

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        rate, nth, sample = cpu_oracle_rate(wl, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": nth, "kind": "oracle", "sample": sample}

    line = {
        "metric": METRIC, "value": rows_s, "unit": UNIT, "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": dist.world * wl.batch,
                   "batch_per_gpu": wl.batch, "nheads": wl.nheads, "headdim": wl.headdim,
                   "dstate": wl.dstate, "ngroups": wl.ngroups, "ring_len": wl.L,
                   "state_dtype": "bf16", "act_dtype": "bf16", "out_dtype": "bf16",
                   "parallelism": "independent replica per gpu (dp%d)" % dist.world,
                   "l2": "inputs larger than L2: 1.07 GB of checkpoint tiles streamed per step"},
        "achieved_hbm_gbs": step_b / (ms_step * 1e-3) / 1e9,
        "hbm_frac_step": step_b / (ms_step * 1e-3) / 1e9 / peak,
        "bytes_per_step": int(step_b),
        "roofline": {"bound": "hbm", "kernel": "mamba2 output_kernel<64,128,bf16>",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": int(out_b), "avg_launch_ms": out_avg_ms},
        "full_state": full,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": 4 * K,
        "clocks": clocks,
    }
    return line


def run_reference(args, dist):
    """The oracle arm: the float64 CPU recurrence on this host's cores; each step a
    bounded sample of the workload's rows."""
    import rssm_workloads as W
    import oracle
    wl = W.mamba2_large(batch=args.batch, seed=args.seed)
    prm = wl.params()
    rows = np.arange(16)
    ci = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci[r])) for r in rows]).astype(np.float64))
    nth = oracle.default_threads()
    inputs = []
    for t in range(4):
        inp = wl.step_inputs(t)
        inputs.append({k: (None if v is None else np.ascontiguousarray(v[rows], dtype=np.float64))
                       for k, v in inp.items()})
    loc = np.arange(len(rows), dtype=np.int32)

    def step(k):
        inp = inputs[k % len(inputs)]
        oracle.mamba2_step(state, inp["x"], inp["dt_raw"], prm["A"], inp["B"], inp["C"], prm["D"],
                           inp["z"], prm["dt_bias"], True, loc, nth)

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(k)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    rate = len(rows) / (ms * 1e-3)
    sample = "%d of %d rows per step, float64 full recurrence, %d threads" % (len(rows), wl.batch,
                                                                              nth)
    return {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": wl.batch,
                   "parallelism": "host cores (oracle)"},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": nth, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            if dist.rank != 0:
                return
            if args.steps > 50:
                args.steps = 50
            line = run_reference(args, dist)
        else:
            line = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
