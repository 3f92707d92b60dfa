"""Benchmark: ReplaySSM decode on GB300.

Default workload (`--workload mamba2`), the headline line: Mamba2 decode at batch
512, nheads 128, headdim 64, dstate 128, ngroups 8, ring L 16, bf16 checkpoint
pool of 1024 slots ~ N(0, 0.1), cache indices = first 512 of a seeded
permutation, desynchronised initial write_pos ~ U{0..15}, x/z/B/C bf16, dt/A/D
fp32, bf16 output; 64 distinct seeded input sets resident in HBM and cycled. One
step = cursor advance, ring append, precompute, output/flush for the whole batch.

Each step is replayed from a CUDA graph holding the fused prologue (cursor advance
+ ring append + tables, one launch) and the output kernel. Every 7th step's graph
also holds two CUDA events around the output kernel; the kernel's duration is the
mean over a phase-complete set of those samples (each residue of the step index
mod the ring length equally often: the flushing rows repeat with that period).

Keys of the JSON line (rank 0):
  value       decode rows/s over all ranks (device-timed, inputs resident)
  e2e         same metric through the public API (Mamba2ReplayDecoder.step) with
              pinned host buffers: host->device copy of each step's inputs and
              device->host copy of y inside the timed region
  roofline    output kernel: algorithmic bytes per launch / CUDA-event duration
              of that kernel inside the timed region, against the measured HBM
              copy bandwidth; traffic = DRAM bytes per launch from the committed
              ncu summary while the kernel source and its headers are unchanged
  cpu_baseline  the float64 oracle (full recurrence) on this host's cores over a
              bounded sample of the same workload
  full_state  the in-house conventional kernel (whole state read+written per
              step) on an identical pool, same inputs
  stochastic_rounding  the same steps with the bf16 state stored by stochastic
              rounding
  gdn_decode, gdn_spec, kda_decode, mamba2_spec  full lines of their own
              workloads (GDN decode batch 256, GDN spec verify batch 128 T 4, KDA
              decode batch 256, Mamba2 spec verify batch 128 T 4), each with its
              roofline, e2e, cpu_baseline and comparison
  mamba2_sweep  a compact sweep (batch 64 / 1024 x L 1 / 16 x fp32 / bf16 state),
              each point beside the full-state kernel

`--workload gdn|spec|kda|m2spec` prints one of the sub-objects as the main line;
`--workload sweep` prints one line per point of the full Mamba2 sweep (batch x L
x state dtype, 5% forced flushes), each with the full-state kernel beside it.
`--impl reference` runs the oracle arm (the only reference implementation this
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
# The kernel of interest is timed with CUDA events on every 7th step (an event record
# costs a few us). 7 is coprime with the 64 input sets and with ring lengths up to 16,
# so the sampled steps cover every input set and every cursor phase of the ring.
EVENT_EVERY = 7
LAST_SEGMENTS = []  # ms per step of each fifth of the last timed region
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
    ap.add_argument("--no-sr", action="store_true",
                    help="skip the stochastic-rounding leg of the mamba2 workload")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--num-slots", type=int, default=None)
    ap.add_argument("--workload", default="mamba2",
                    choices=["mamba2", "gdn", "spec", "kda", "m2spec", "sweep"])
    ap.add_argument("--no-gdn", action="store_true",
                    help="mamba2 line only (skip the gdn_decode / gdn_spec sub-objects)")
    ap.add_argument("--sweep-steps", type=int, default=200)
    ap.add_argument("--sweep-sub-steps", type=int, default=100,
                    help="timed steps per point of the compact sweep in the default line")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the compact Mamba2 sweep sub-object of the default line")
    ap.add_argument("--event-every", type=int, default=7,
                    help="time the kernel of interest with CUDA events on every n-th step")
    ap.add_argument("--source-hash", default=None, metavar="FILE.cu",
                    help="print the combined sha256 of a kernel source and its headers and exit")
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


def _local_includes(path, seen):
    """The file and every header it includes with #include "..." from the library's
    csrc/ or include/ folders, recursively (sorted, each once)."""
    if path in seen or not os.path.exists(path):
        return
    seen.add(path)
    dirs = [os.path.dirname(path), os.path.join(ROOT, "ssm_linear_attention_gb300", "csrc"),
            os.path.join(ROOT, "include")]
    for line in open(path, encoding="utf-8"):
        line = line.strip()
        if line.startswith("#include") and '"' in line:
            name = line.split('"')[1]
            for d in dirs:
                cand = os.path.normpath(os.path.join(d, name))
                if os.path.exists(cand):
                    _local_includes(cand, seen)
                    break


def source_hash(kernel_src):
    """sha256 over a kernel's .cu file and every local header it includes (pipeline,
    common helpers, cursor model, the C header), so that a change to any of them
    invalidates counters taken before it."""
    src = os.path.join(ROOT, "ssm_linear_attention_gb300", "csrc", kernel_src)
    files = set()
    _local_includes(src, files)
    h = hashlib.sha256()
    for f in sorted(files, key=lambda p: os.path.relpath(p, ROOT)):
        h.update(os.path.relpath(f, ROOT).encode())
        h.update(b"\0")
        h.update(open(f, "rb").read())
    return h.hexdigest()


def traffic_record(kernel_src, profile):
    """DRAM bytes per launch of a kernel from its committed ncu summary, valid only
    while the kernel source and the headers it includes are unchanged (their
    combined sha256, source_hash(), recorded beside the figure)."""
    src = os.path.join(ROOT, "ssm_linear_attention_gb300", "csrc", kernel_src)
    prof = os.path.join(ROOT, "profiles", profile)
    if not (os.path.exists(src) and os.path.exists(prof)):
        return None
    sha = source_hash(kernel_src)
    rec = {}
    for line in open(prof):
        if ":" in line and line.strip().strip("-* `").startswith(("source_sha256",
                                                                   "traffic_bytes_per_launch")):
            k, v = line.split(":", 1)
            rec[k.strip().strip("-* `")] = v.strip().strip("`")
    if rec.get("source_sha256") == sha and rec.get("traffic_bytes_per_launch"):
        return int(float(rec["traffic_bytes_per_launch"]))
    return None  # no summary, or the kernel or a header changed since the counters were taken


def gdn_output_bytes(wl, row_wp, row_flush, out_bytes=2):
    """Algorithmic bytes of one GDN output-kernel launch: checkpoint read, d entries
    0..w-1, this step's k (from the ring), q, v, the d write, o, and on flush rows
    the state write and the earlier k entries. The tables are excluded."""
    HV, HK, K, V = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim
    sa = 2 if wl.act_dtype == "bf16" else 4
    w = row_wp.astype(np.int64)
    f = row_flush.astype(np.int64)
    per_row = (HV * V * K * 4 + w * HV * V * 4 + HV * V * 4 + 2 * HK * K * sa + HV * V * sa
               + HV * V * out_bytes + f * (HV * V * K * 4 + w * HK * K * sa))
    return int(per_row.sum())


def gdn_full_bytes(wl, batch, out_bytes=2):
    HV, HK, K, V = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim
    sa = 2 if wl.act_dtype == "bf16" else 4
    return batch * (2 * HV * V * K * 4 + 2 * HK * K * sa + HV * V * sa + 2 * HV * 4
                    + HV * V * out_bytes)


def kda_output_bytes(wl, row_wp, row_flush, out_bytes=2):
    """Algorithmic bytes of one KDA output-kernel launch: checkpoint read, d entries
    0..w-1, v, o, the d write and, on flush rows, the state write. The prologue's
    gated vectors and tables are excluded (as the GDN and Mamba2 tables are)."""
    HV, V, K = wl.num_v_heads, wl.head_v_dim, wl.head_k_dim
    sa = 2 if wl.act_dtype == "bf16" else 4
    w = row_wp.astype(np.int64)
    f = row_flush.astype(np.int64)
    per_row = (HV * V * K * 4 + w * HV * V * 4 + HV * V * 4 + HV * V * sa + HV * V * out_bytes
               + f * HV * V * K * 4)
    return int(per_row.sum())


def kda_step_bytes(wl, row_wp, row_flush, out_bytes=2):
    """Algorithmic bytes of a whole KDA step: the output kernel's, plus the ring k and
    gate entries 0..w-1 the prologue reads, the step's q, k, a, beta and the k and a
    appends."""
    HV, HK, K = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim
    sa = 2 if wl.act_dtype == "bf16" else 4
    w = row_wp.astype(np.int64)
    pro = w * (HK * K * sa + HV * K * 4) + 2 * HK * K * sa + HV * K * 4 + 4 * HV \
        + HK * K * sa + HV * K * 4
    return kda_output_bytes(wl, row_wp, row_flush, out_bytes) + int(pro.sum())


def kda_full_bytes(wl, batch, out_bytes=2):
    HV, HK, K, V = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim
    sa = 2 if wl.act_dtype == "bf16" else 4
    return batch * (2 * HV * V * K * 4 + 2 * HK * K * sa + HV * V * sa + HV * K * 4 + HV * 4
                    + HV * V * out_bytes)


def spec_round_bytes(wl, hist, out_bytes=2):
    """Algorithmic bytes of one GDN verify launch over the rows, given each row's
    history count: checkpoint read, the drafts' q, k, v, beta, g, the history d
    entries, the drafts' d, raw v, k, g, beta written to the rings, o (the folds are
    counted by gdn_fold_bytes)."""
    HV, HK, K, V, T = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.T
    sa = 2 if wl.act_dtype == "bf16" else 4
    c = hist.astype(np.int64)
    verify = (HV * V * K * 4 + T * (2 * HK * K * sa + HV * V * sa + 2 * HV * 4)
              + c * HV * V * 4 + T * (HV * V * 4 + HV * V * sa + HK * K * sa + 2 * HV * 4)
              + T * HV * V * out_bytes)
    return int(verify.sum())


def spec_cursor_rounds(num_slots, ci, accepted_seq, L, T):
    """Per round (history count, pending fold flag, committed count) of the rows, for a
    sequence of accepted counts, following the commit rule (a pending fold retires
    the committed run, then cnt += accepted and flush = cnt + T > L); and the final
    cnt of every slot. Bookkeeping for the byte counts; the kernels keep their own
    cursors on the device."""
    cnt = np.zeros(num_slots, np.int64)
    base = np.zeros(num_slots, np.int64)
    flush = np.zeros(num_slots, np.int64)
    out = []
    for acc in accepted_seq:
        fl = flush[ci].copy()
        cr = cnt[ci].copy()
        out.append((np.where(fl == 1, 0, cr), fl, cr))
        base[ci] = np.where(fl == 1, (base[ci] + cr) % L, base[ci])
        cnt[ci] = np.where(fl == 1, 0, cr) + acc
        flush[ci] = (cnt[ci] + T > L).astype(np.int64)
    return out, cnt


def m2spec_round_bytes(wl, hist, fl, cr, out_bytes=2):
    """Algorithmic bytes of one Mamba2 verify round, as (verify, fold) totals over the
    rows. Verify: checkpoint read, the history x (and, in the prologue, the history B
    and dt), the drafts' x, z, dt_raw, B, C, y, and the drafts' x, dt, B appended to
    the ring. Fold (rows with a pending fold): state read and write plus the
    committed entries' x, dt, B."""
    H, P, N, G, T = wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.T
    sa = 2 if wl.act_dtype == "bf16" else 4
    ss = 2 if wl.state_dtype == "bf16" else 4
    c = hist.astype(np.int64)
    entry = H * P * sa + 4 * H + G * N * sa
    verify = (H * P * N * ss + c * entry + T * (2 * H * P * sa + 2 * G * N * sa + 4 * H)
              + T * H * P * out_bytes + T * entry)
    fold = fl.astype(np.int64) * (2 * H * P * N * ss + cr.astype(np.int64) * entry)
    return int(verify.sum()), int(fold.sum())


def gdn_fold_bytes(wl, fl, cr):
    """Algorithmic bytes of the GDN exact folds of one round: state read and write plus
    the committed entries' k, raw v, beta and g, for the rows with a pending fold."""
    HV, HK, K, V = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim
    sa = 2 if wl.act_dtype == "bf16" else 4
    return int((fl * (2 * HV * V * K * 4 + cr * (HK * K * sa + HV * V * sa + 2 * HV * 4))).sum())


# --------------------------------------------------------------------------- #
# CUDA graphs and the timed loop                                              #
# --------------------------------------------------------------------------- #

def _graphs(fns):
    """Capture each zero-argument callable into its own CUDA graph."""
    import torch
    out = []
    for fn in fns:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        out.append(g)
    torch.cuda.synchronize()
    return out


def _bus_id(dev):
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return "%08x:%02x:%02x" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id, p.pci_device_id)
    except Exception:
        return None


def _sampled_graphs(fns, kernel_fns):
    """Per input set j two graphs: whole[j] runs fns[j]; samp[j] runs the same work
    with external CUDA events recorded around kernel_fns[j] (the kernel being timed),
    so the events are nodes of the graph and time that kernel alone. kernel_fns[j] is
    a pair (before, kernel, after) of callables."""
    import torch
    whole = _graphs(fns)
    samp, evs = [], []
    for before, kern, after in kernel_fns:
        a = torch.cuda.Event(enable_timing=True, external=True)
        b = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if before is not None:
                before()
            a.record()
            kern()
            b.record()
            if after is not None:
                after()
        samp.append(g)
        evs.append((a, b))
    torch.cuda.synchronize()
    return whole, samp, evs


def _timed_graphs(whole, samp, evs, K, dist, dev, offset=0, clocks=True, every=None):
    """Replay K steps; step k runs input set j = (k + offset) % G, as samp[j] when
    k % every == 0 (events around the timed kernel) and as whole[j] otherwise.
    Returns (elapsed ms of the region, max over ranks; the timed kernel's ms from
    the last sampled replay of each input set; clock record; the step index of each
    of those samples)."""
    import torch
    every = EVENT_EVERY if every is None else every
    stream = torch.cuda.current_stream()
    G = len(whole)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # five equal segments of the region, each bracketed by events, for a median
    nseg = 5 if K >= 5 else 1
    bounds = [K * i // nseg for i in range(1, nseg)]
    seg_ev = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    last = {}
    dist.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler() if clocks else None
    if clk:
        time.sleep(0.3)
    start.record(stream)
    bi = 0
    for k in range(K):
        if bi < len(bounds) and k == bounds[bi]:
            seg_ev[bi].record(stream)
            bi += 1
        j = (k + offset) % G
        if k % every == 0:
            samp[j].replay()
            last[j] = k
        else:
            whole[j].replay()
    end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    rec = clk.stop(_bus_id(dev)) if clk else None
    js = [j for j in sorted(last) if evs[j][0] is not None]
    per = [evs[j][0].elapsed_time(evs[j][1]) for j in js]
    marks = [start] + seg_ev + [end]
    edges = [0] + bounds + [K]
    seg_ms = [marks[i].elapsed_time(marks[i + 1]) / max(edges[i + 1] - edges[i], 1)
              for i in range(len(marks) - 1)]
    global LAST_SEGMENTS
    LAST_SEGMENTS = seg_ms
    return dist.max(start.elapsed_time(end)), per, rec, [last[j] for j in js]


def _phase_complete(per, ks, samp, evs, K, offset, period, every=None):
    """Launch times of the timed kernel that cover every cursor phase equally.

    A step's cursor pattern repeats with the ring length L (every row's write_pos
    advances by one per step), so a set of samples is representative when the step
    indices cover each residue mod `period` equally often. The timed region samples
    every `every`-th step (coprime with `period`) and keeps the last sample of each
    input set, i.e. consecutive sampled steps; the last (n // period) * period of
    them cover every residue exactly n // period times. When the region holds fewer
    than `period` samples (a short --steps), a dedicated pass of consecutive steps
    right after the region, every one carrying the events, supplies them instead.
    Returns (list of (step index, ms), source description)."""
    import math

    import torch
    every = EVENT_EVERY if every is None else every
    pairs = sorted(zip(ks, per))
    if math.gcd(every, period) == 1:
        n_use = (len(pairs) // period) * period
        if n_use >= period:
            return pairs[-n_use:], "in the timed region: %d sampled launches (every %d-th step), " \
                "each cursor phase of the %d-step cycle %d times" % (n_use, every, period,
                                                                    n_use // period)
    G = len(samp)
    M = period * max(1, 32 // period)
    out, k = [], K
    while len(out) < M:
        n = min(G, M - len(out))
        js = []
        for _ in range(n):
            j = (k + offset) % G
            samp[j].replay()
            js.append((k, j))
            k += 1
        torch.cuda.synchronize()
        out += [(kk, evs[j][0].elapsed_time(evs[j][1])) for kk, j in js]
    return out, "dedicated pass of %d consecutive launches right after the timed region (the " \
        "region's %d samples did not cover the %d cursor phases)" % (M, len(pairs), period)


def _flush_split(samples, curs, bytes_fn):
    """Launch-time and byte means of the sampled launches, overall and split into
    launches whose rows flush and launches whose rows do not (rows that share one
    cursor phase flush together, every L-th step)."""
    fl = [(k, ms) for k, ms in samples if curs[k][1].any()]
    nf = [(k, ms) for k, ms in samples if not curs[k][1].any()]

    def mean(xs, f):
        return float(np.mean([f(x) for x in xs])) if xs else None

    return {
        "flush_launches": len(fl), "nonflush_launches": len(nf),
        "flush_launch_ms": mean(fl, lambda x: x[1]),
        "nonflush_launch_ms": mean(nf, lambda x: x[1]),
        "flush_bytes_per_launch": mean(fl, lambda x: bytes_fn(*curs[x[0]])),
        "nonflush_bytes_per_launch": mean(nf, lambda x: bytes_fn(*curs[x[0]])),
    }


def _e2e_pipelined(dev, dist, n_steps, host_sets, dev_template, out_template, step_fn):
    """End-to-end steps through a public API call with host buffers: every step copies
    its inputs from pinned host memory to the device and its result back, all inside
    the timed region. The copies of step k+1 (in) and k-1 (out) run on two side
    streams, with double-buffered device inputs and outputs, while step k computes.

    host_sets: list of {name: pinned host tensor}; dev_template: {name: device tensor}
    (shapes and dtypes of the device copies); out_template: a device tensor like the
    step's result; step_fn(d, out, stream) runs one step reading the device inputs d
    and writing out. Returns (ms per step, max over ranks; H2D bytes; D2H bytes)."""
    import torch
    names = list(dev_template)
    dsts = [{k: v.clone() for k, v in dev_template.items()} for _ in range(2)]
    obuf = [torch.empty_like(out_template) for _ in range(2)]
    o_host = [torch.empty(out_template.shape, dtype=out_template.dtype).pin_memory()
              for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_sets[0].values())
    d2h = o_host[0].numel() * o_host[0].element_size()
    stream = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for k in range(n):
            j = k & 1
            hs = host_sets[k % len(host_sets)]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_done[j])      # step k-2 has read buffer j
                for name in names:
                    dsts[j][name].copy_(hs[name], non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if k >= 2:
                stream.wait_event(ev_out[j])         # the result of step k-2 has left buffer j
            step_fn(dsts[j], obuf[j], stream)
            ev_done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[j])
                o_host[j].copy_(obuf[j], non_blocking=True)
                ev_out[j].record(s_out)
        stream.wait_stream(s_out)

    run(4)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    run(n_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    return dist.max(e0.elapsed_time(e1)) / n_steps, int(h2d), int(d2h)


def _pinned_sets(make_inputs, count, dtypes):
    """Pinned host copies of `count` input sets; make_inputs(t) -> {name: numpy}."""
    import torch
    out = []
    for t in range(count):
        inp = make_inputs(t)
        out.append({k: torch.from_numpy(inp[k]).to(dt).pin_memory() for k, dt in dtypes.items()})
    return out


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


def cpu_oracle_rate_gdn(wl, seconds, max_rows=16):
    """The float64 GDN recurrence on a sample of rows (rows/s, threads, sample)."""
    import oracle
    nth = oracle.default_threads()
    rows = np.arange(min(max_rows, wl.batch))
    ci = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci[r])) for r in rows]).astype(np.float64))
    inputs = []
    for t in range(4):
        inp = wl.step_inputs(t)
        inputs.append({k: np.ascontiguousarray(v[rows], dtype=np.float64) for k, v in inp.items()})
    loc = np.arange(len(rows), dtype=np.int32)
    done, t0 = 0, time.perf_counter()
    while True:
        inp = inputs[done % len(inputs)]
        oracle.gdn_step(state, inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], loc,
                        nthreads=nth)
        done += 1
        el = time.perf_counter() - t0
        if done >= 2 and el >= seconds:
            break
    rate = done * len(rows) / el
    sample = "%d rows x %d steps of the float64 gated delta recurrence (%.1f s)" % (len(rows),
                                                                                    done, el)
    return rate, nth, sample


def _cpu_rate(wl, seconds, max_rows, inputs_fn, step_fn, what):
    """Time an oracle step over a sample of rows until `seconds` of work have run (at
    least two steps). inputs_fn(t) -> {name: array over all rows}; step_fn(state,
    inputs, local slot indices, threads) runs one step of the sampled rows. Returns
    (rows/s, threads, sample text)."""
    import oracle
    nth = oracle.default_threads()
    rows = np.arange(min(max_rows, wl.batch))
    ci = wl.cache_indices()
    state = np.ascontiguousarray(
        np.stack([wl.slot_state(int(ci[r])) for r in rows]).astype(np.float64))
    inputs = []
    for t in range(4):
        inp = inputs_fn(t)
        inputs.append({k: (None if v is None else np.ascontiguousarray(v[rows]))
                       for k, v in inp.items()})
    loc = np.arange(len(rows), dtype=np.int32)
    done, t0 = 0, time.perf_counter()
    while True:
        step_fn(state, inputs[done % len(inputs)], loc, nth)
        done += 1
        el = time.perf_counter() - t0
        if done >= 2 and el >= seconds:
            break
    rate = done * len(rows) / el
    return rate, nth, "%d rows x %d %s (%.1f s)" % (len(rows), done, what, el)


def cpu_oracle_rate_kda(wl, seconds, max_rows=16):
    import oracle
    return _cpu_rate(wl, seconds, max_rows, wl.step_inputs,
                     lambda st, i, loc, n: oracle.kda_step(st, i["q"], i["k"], i["v"], i["beta"],
                                                           i["a"], loc, nthreads=n),
                     "steps of the float64 per-channel-gate delta recurrence")


def cpu_oracle_rate_spec(wl, seconds, max_rows=16):
    import oracle

    def inputs(t):
        d = dict(wl.round_inputs(t))
        d["acc"] = wl.accepted(t).astype(np.int32)
        return d

    return _cpu_rate(wl, seconds, max_rows, inputs,
                     lambda st, i, loc, n: oracle.gdn_spec_round(
                         st, wl.T, i["q"], i["k"], i["v"], i["beta"], i["g"], i["acc"], loc,
                         nthreads=n),
                     "verify rounds of the float64 gated delta recurrence (T %d drafts)" % wl.T)


def cpu_oracle_rate_m2spec(wl, seconds, max_rows=16):
    import oracle
    prm = wl.params()

    def inputs(t):
        d = dict(wl.round_inputs(t))
        d["acc"] = wl.accepted(t).astype(np.int32)
        return d

    return _cpu_rate(wl, seconds, max_rows, inputs,
                     lambda st, i, loc, n: oracle.mamba2_spec_round(
                         st, wl.T, i["x"], i["dt_raw"], prm["A"], i["B"], i["C"], prm["D"],
                         i["acc"], i["z"], prm["dt_bias"], wl.dt_softplus, loc, n),
                     "verify rounds of the float64 Mamba2 recurrence (T %d drafts)" % wl.T)


# --------------------------------------------------------------------------- #
# Mamba2 (headline)                                                           #
# --------------------------------------------------------------------------- #

def _device(dist):
    import torch
    dev = torch.device("cuda", dist.local if dist.world > 1 else 0)
    torch.cuda.set_device(dev)
    return dev


def run_mamba2(args, dist):
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    wl = W.mamba2_large(batch=args.batch or 512, num_slots=args.num_slots or 1024,
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

    K = args.steps
    G = min(len(sets), max(K, 1))

    def pre_fn(j):
        x, dt, Bm, C, z = sets[j]

        return lambda: dec.prepare(x, dt, Bm, C, ci)

    def out_fn(j):
        x, dt, Bm, C, z = sets[j]
        return lambda: dec.output(C, z, ci)

    # eager warm-up (sets shared-memory limits, first-use costs), then capture
    for k in range(max(args.warmup, 3)):
        pre_fn(k % G)()
        out_fn(k % G)()
    torch.cuda.synchronize()
    g_step, g_samp, evs = _sampled_graphs(
        [(lambda j=j: (pre_fn(j)(), out_fn(j)())) for j in range(G)],
        [(pre_fn(j), out_fn(j), None) for j in range(G)])
    # capture does not run the work: warm up the graphs themselves
    for k in range(max(args.warmup, 3)):
        g_step[k % G].replay()
    torch.cuda.synchronize()
    slot_wp0 = dec.slot_wp.cpu().numpy().astype(np.int64)
    off = args.warmup + max(args.warmup, 3)

    elapsed, out_ms, clocks, ks = _timed_graphs(g_step, g_samp, evs, K, dist, dev, offset=off)
    seg_median = float(np.median(LAST_SEGMENTS))
    samples, ksrc = _phase_complete(out_ms, ks, g_samp, evs, K, off, wl.L)
    assert int(dec.dev_err.abs().sum().item()) == 0, "device error flag set during the bench"
    del g_step, g_samp

    ms_step = elapsed / K
    rows_s = dist.world * wl.batch / (ms_step * 1e-3)

    curs = simulate_cursors(slot_wp0, ci_np, wl.L, K + 64)
    out_ms = [ms for _, ms in samples]
    out_b = np.mean([output_kernel_bytes(wl, *curs[k]) for k, _ in samples])
    step_b = np.mean([step_bytes(wl, w, f) for w, f in curs[:K]])
    out_avg_ms = float(np.mean(out_ms))
    peak, peak_kind = read_peaks()
    achieved = out_b / (out_avg_ms * 1e-3) / 1e9
    traffic = traffic_record("mamba2.cu", "mamba2_output_kernel_batch512.md")

    # end to end through the public API with pinned host buffers
    e2e = None
    if args.e2e_steps > 0:
        names = ("x", "dt_raw", "B", "C", "z")
        dts = {k2: (bf if k2 != "dt_raw" else torch.float32) for k2 in names}
        host_sets = _pinned_sets(wl.step_inputs, min(8, args.input_sets), dts)
        ybuf0 = torch.empty(wl.batch, wl.nheads, wl.headdim, device=dev, dtype=bf)

        def m2_step(d, y, stream):
            dec.step(d["x"], d["dt_raw"], d["B"], d["C"], d["z"], ci, y=y, stream=stream)

        e_ms, h2d, d2h = _e2e_pipelined(dev, dist, args.e2e_steps, host_sets,
                                        dict(zip(names, sets[0])), ybuf0, m2_step)
        e2e = {"value": dist.world * wl.batch / (e_ms * 1e-3), "unit": UNIT,
               "ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "Mamba2ReplayDecoder.step (eager; one rssm_mamba2_step call, 2 launches); "
                      "inputs and y copied on two side streams, double-buffered"}

    # the same steps with stochastic rounding of the flush stores (bf16 state)
    sr = None
    if not args.no_sr:
        dec.sr = torch.tensor([0x5EED, 0], device=dev, dtype=torch.int64)
        for k in range(max(args.warmup, 3)):
            pre_fn(k % G)()
            out_fn(k % G)()
        torch.cuda.synchronize()
        g_sr, g_srs, srevs = _sampled_graphs(
            [(lambda j=j: (pre_fn(j)(), out_fn(j)())) for j in range(G)],
            [(pre_fn(j), out_fn(j), None) for j in range(G)])
        for k in range(max(args.warmup, 3)):
            g_sr[k % G].replay()
        Ks = max(50, K // 4)
        s_el, s_per, _, _ = _timed_graphs(g_sr, g_srs, srevs, Ks, dist, dev, clocks=False)
        del g_sr, g_srs
        dec.sr = None
        s_ms = s_el / Ks
        sr = {"us_per_step": s_ms * 1e3, "rows_per_s": dist.world * wl.batch / (s_ms * 1e-3),
              "output_us": float(np.mean(s_per)) * 1e3,
              "output_us_nearest": out_avg_ms * 1e3,
              "step_overhead": s_ms / ms_step - 1.0,
              "note": "flush stores rounded stochastically (Philox4x32-10 bits); the output "
                      "launch is followed by a 1-thread launch advancing the generator offset"}

    # the in-house conventional kernel on an identical pool
    full = None
    if not args.no_full_state:
        fdec = ssm.Mamba2FullStateDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups,
                                          wl.num_slots, wl.batch, prm["A"], prm["D"],
                                          prm["dt_bias"], state_dtype=bf, act_dtype=bf,
                                          out_dtype=bf, device=dev)
        fdec.state.copy_(dec.state)
        del dec

        def full_fn(j):
            x, dt, Bm, C, z = sets[j]
            return lambda: fdec.step(x, dt, Bm, C, z, ci)

        for k in range(max(args.warmup, 3)):
            full_fn(k % G)()
        torch.cuda.synchronize()
        g_full, g_fs, fevs = _sampled_graphs([full_fn(j) for j in range(G)],
                                             [(None, full_fn(j), None) for j in range(G)])
        Kf = max(50, K // 4)
        f_el, f_per, _, _ = _timed_graphs(g_full, g_fs, fevs, Kf, dist, dev, clocks=False)
        del g_full, g_fs
        f_ms = f_el / Kf
        fb = full_state_bytes(wl, wl.batch)
        full = {"ms_per_step": f_ms, "us_per_step": f_ms * 1e3,
                "rows_per_s": dist.world * wl.batch / (f_ms * 1e-3),
                "achieved_gbs": fb / (float(np.mean(f_per)) * 1e-3) / 1e9, "bytes_per_step": fb,
                "hbm_frac": fb / (float(np.mean(f_per)) * 1e-3) / 1e9 / peak,
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
                   "timing": "one CUDA graph per step (prepare + output); on every 7th step the graph also holds CUDA events around the output kernel; the kernel figures use samples covering every cursor phase equally",
                   "l2": "inputs larger than L2: 1.07 GB of checkpoint tiles streamed per step"},
        "ms_per_step_median_of_5": seg_median,
        "achieved_hbm_gbs": step_b / (ms_step * 1e-3) / 1e9,
        "hbm_frac_step": step_b / (ms_step * 1e-3) / 1e9 / peak,
        "bytes_per_step": int(step_b),
        "roofline": {"bound": "hbm", "kernel": "mamba2 output_kernel<64,128,bf16>",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": int(out_b), "avg_launch_ms": out_avg_ms,
                     "launches_timed": len(out_ms), "min_launch_ms": float(np.min(out_ms)),
                     "max_launch_ms": float(np.max(out_ms)), "event_every": EVENT_EVERY,
                     "kernel_timing": ksrc},
        "full_state": full,
        "stochastic_rounding": sr,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    return line


# --------------------------------------------------------------------------- #
# gated delta net: decode                                                     #
# --------------------------------------------------------------------------- #

GDN_WORKLOAD = ("gdn replayssm decode: batch 256, HV 32, HK 16, K=V 128, L 16, fp32 state pool "
                "512 slots ~N(0,0.05), bf16 q/k/v, fp32 beta/g")


def run_gdn(args, dist, sub=False):
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    kw = {}
    if not sub and args.batch:
        kw["batch"] = args.batch
    if not sub and args.num_slots:
        kw["num_slots"] = args.num_slots
    wl = W.gdn_decode(seed=shard_seed(args.seed, dist.rank), **kw)
    bf = torch.bfloat16
    ci_np = wl.cache_indices()
    ci = torch.from_numpy(ci_np).to(dev)
    dec = ssm.GDNReplayDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.L,
                               wl.num_slots, wl.batch, act_dtype=bf, out_dtype=bf, device=dev)
    for s in ci_np:
        dec.state[int(s)] = torch.from_numpy(wl.slot_state(int(s))).to(dev)

    def to_dev(inp):
        return [torch.from_numpy(inp[k]).to(dev, bf if k in ("q", "k", "v") else torch.float32)
                for k in ("q", "k", "v", "beta", "g")]

    for j in range(wl.max_history()):
        dec.step(*to_dev(wl.history_inputs(j)), torch.from_numpy(wl.history_ci(j)).to(dev))
    nsets = min(args.input_sets, 32)
    sets = [to_dev(wl.step_inputs(t)) for t in range(nsets)]
    torch.cuda.synchronize()
    K = args.steps
    G = min(len(sets), max(K, 1))

    def pre_fn(j):
        q, k, v, beta, g = sets[j]

        return lambda: dec.prepare(q, k, beta, g, ci)

    def out_fn(j):
        q, k, v, beta, g = sets[j]
        return lambda: dec.output(q, v, ci)

    for k in range(max(args.warmup, 3)):
        pre_fn(k % G)()
        out_fn(k % G)()
    torch.cuda.synchronize()
    g_step, g_samp, evs = _sampled_graphs(
        [(lambda j=j: (pre_fn(j)(), out_fn(j)())) for j in range(G)],
        [(pre_fn(j), out_fn(j), None) for j in range(G)])
    for k in range(max(args.warmup, 3)):
        g_step[k % G].replay()
    torch.cuda.synchronize()
    slot_wp0 = dec.slot_wp.cpu().numpy().astype(np.int64)
    off = args.warmup + max(args.warmup, 3)
    elapsed, out_ms, clocks, ks = _timed_graphs(g_step, g_samp, evs, K, dist, dev, offset=off,
                                                clocks=not sub)
    samples, ksrc = _phase_complete(out_ms, ks, g_samp, evs, K, off, wl.L)
    assert int(dec.dev_err.abs().sum().item()) == 0, "device error flag set during the gdn bench"
    del g_step, g_samp
    ms_step = elapsed / K
    rows_s = dist.world * wl.batch / (ms_step * 1e-3)
    curs = simulate_cursors(slot_wp0, ci_np, wl.L, K + 64)
    out_ms = [ms for _, ms in samples]
    out_b = np.mean([gdn_output_bytes(wl, *curs[k]) for k, _ in samples])
    split = _flush_split(samples, curs, lambda w, f: gdn_output_bytes(wl, w, f))
    out_avg_ms = float(np.mean(out_ms))
    peak, peak_kind = read_peaks()
    achieved = out_b / (out_avg_ms * 1e-3) / 1e9

    e2e = None
    if args.e2e_steps > 0:
        names = ("q", "k", "v", "beta", "g")
        dts = {n_: (bf if n_ in ("q", "k", "v") else torch.float32) for n_ in names}
        host_sets = _pinned_sets(wl.step_inputs, min(8, nsets), dts)
        obuf0 = torch.empty(wl.batch, wl.num_v_heads, wl.head_v_dim, device=dev, dtype=bf)

        def gdn_step(d, o, stream):
            dec.step(d["q"], d["k"], d["v"], d["beta"], d["g"], ci, o=o, stream=stream)

        e_ms, h2d, d2h = _e2e_pipelined(dev, dist, args.e2e_steps, host_sets,
                                        dict(zip(names, sets[0])), obuf0, gdn_step)
        e2e = {"value": dist.world * wl.batch / (e_ms * 1e-3), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "GDNReplayDecoder.step (eager; one rssm_gdn_step call, 2 launches); inputs "
                      "and o copied on two side streams, double-buffered"}

    full = None
    if not args.no_full_state:
        fdec = ssm.GDNFullStateDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim,
                                       wl.head_v_dim, wl.num_slots, wl.batch, act_dtype=bf,
                                       out_dtype=bf, device=dev)
        fdec.state.copy_(dec.state)
        del dec

        def full_fn(j):
            q, k, v, beta, g = sets[j]
            return lambda: fdec.step(q, k, v, beta, g, ci)

        for k in range(max(args.warmup, 3)):
            full_fn(k % G)()
        torch.cuda.synchronize()
        g_full, g_fs, fevs = _sampled_graphs([full_fn(j) for j in range(G)],
                                             [(None, full_fn(j), None) for j in range(G)])
        Kf = max(50, K // 4)
        f_el, f_per, _, _ = _timed_graphs(g_full, g_fs, fevs, Kf, dist, dev, clocks=False)
        del g_full, g_fs
        f_ms = f_el / Kf
        fb = gdn_full_bytes(wl, wl.batch)
        full = {"ms_per_step": f_ms, "us_per_step": f_ms * 1e3,
                "rows_per_s": dist.world * wl.batch / (f_ms * 1e-3),
                "achieved_gbs": fb / (float(np.mean(f_per)) * 1e-3) / 1e9, "bytes_per_step": fb,
                "hbm_frac": fb / (float(np.mean(f_per)) * 1e-3) / 1e9 / peak,
                "replay_speedup": f_ms / ms_step}

    line = {
        "metric": "gdn decode rows/s and µs/step at batch %d; achieved HBM GB/s" % wl.batch,
        "value": rows_s, "unit": UNIT, "n_gpus": dist.world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "us_per_step": ms_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": GDN_WORKLOAD, "global_batch": dist.world * wl.batch,
                   "batch_per_gpu": wl.batch, "HV": wl.num_v_heads, "HK": wl.num_k_heads,
                   "K": wl.head_k_dim, "V": wl.head_v_dim, "ring_len": wl.L,
                   "timing": "one CUDA graph per step (prepare + output); on every 7th step the graph also holds CUDA events around the output kernel; the kernel figures use samples covering every cursor phase equally",
                   "l2": "inputs larger than L2: 537 MB of fp32 checkpoint tiles per step"},
        "roofline": dict({"bound": "hbm", "kernel": "gdn output kernel (fp32 state, 32-row tiles)",
                          "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak, "peak_source": peak_kind,
                          "traffic": traffic_record("gdn.cu", "gdn_output_kernel_batch256.md"),
                          "algorithmic_bytes_per_launch": int(out_b), "avg_launch_ms": out_avg_ms,
                          "launches_timed": len(out_ms), "kernel_timing": ksrc}, **split),
        "full_state": full,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        rate, nth, sample = cpu_oracle_rate_gdn(wl, args.cpu_seconds / 3 if sub else args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": nth, "kind": "oracle",
                                "sample": sample}
    return line


KDA_WORKLOAD = ("kda replayssm decode: batch 256, HV 32, HK 16, K=V 128, L 16, fp32 state pool "
                "512 slots ~N(0,0.05), bf16 q/k/v, fp32 beta, per-channel gates a [HV, K] in (0,1)")


def run_kda(args, dist, sub=False):
    """The KDA (per-key-channel gate) decode step against the conventional KDA kernel."""
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    kw = {}
    if not sub and args.batch:
        kw["batch"] = args.batch
    if not sub and args.num_slots:
        kw["num_slots"] = args.num_slots
    wl = W.kda_decode(seed=shard_seed(args.seed, dist.rank), **kw)
    bf = torch.bfloat16
    ci_np = wl.cache_indices()
    ci = torch.from_numpy(ci_np).to(dev)
    dec = ssm.KDAReplayDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, wl.L,
                               wl.num_slots, wl.batch, act_dtype=bf, out_dtype=bf, device=dev)
    for s in ci_np:
        dec.state[int(s)] = torch.from_numpy(wl.slot_state(int(s))).to(dev)

    def to_dev(inp):
        return [torch.from_numpy(inp[k]).to(dev, bf if k in ("q", "k", "v") else torch.float32)
                for k in ("q", "k", "v", "beta", "a")]

    for j in range(wl.max_history()):
        dec.step(*to_dev(wl.history_inputs(j)), torch.from_numpy(wl.history_ci(j)).to(dev))
    nsets = min(args.input_sets, 32)
    sets = [to_dev(wl.step_inputs(t)) for t in range(nsets)]
    torch.cuda.synchronize()
    K = args.steps
    G = min(len(sets), max(K, 1))

    def pre_fn(j):
        q, k, v, beta, a = sets[j]

        def f():
            dec.advance(ci)
            dec.prepare(q, k, a, beta, ci)
        return f

    def out_fn(j):
        q, k, v, beta, a = sets[j]
        return lambda: dec.output(v, ci)

    for k in range(max(args.warmup, 3)):
        pre_fn(k % G)()
        out_fn(k % G)()
    torch.cuda.synchronize()
    g_step, g_samp, evs = _sampled_graphs(
        [(lambda j=j: (pre_fn(j)(), out_fn(j)())) for j in range(G)],
        [(pre_fn(j), out_fn(j), None) for j in range(G)])
    for k in range(max(args.warmup, 3)):
        g_step[k % G].replay()
    torch.cuda.synchronize()
    slot_wp0 = dec.slot_wp.cpu().numpy().astype(np.int64)
    off = args.warmup + max(args.warmup, 3)
    elapsed, out_ms, clocks, ks = _timed_graphs(g_step, g_samp, evs, K, dist, dev, offset=off,
                                                clocks=not sub)
    samples, ksrc = _phase_complete(out_ms, ks, g_samp, evs, K, off, wl.L)
    assert int(dec.dev_err.abs().sum().item()) == 0, "device error flag set during the kda bench"
    del g_step, g_samp
    ms_step = elapsed / K
    rows_s = dist.world * wl.batch / (ms_step * 1e-3)
    curs = simulate_cursors(slot_wp0, ci_np, wl.L, K + 64)
    out_ms = [ms for _, ms in samples]
    out_b = np.mean([kda_output_bytes(wl, *curs[k]) for k, _ in samples])
    split = _flush_split(samples, curs, lambda w, f: kda_output_bytes(wl, w, f))
    step_b = np.mean([kda_step_bytes(wl, w, f) for w, f in curs[:K]])
    out_avg_ms = float(np.mean(out_ms))
    peak, peak_kind = read_peaks()
    achieved = out_b / (out_avg_ms * 1e-3) / 1e9

    e2e = None
    if args.e2e_steps > 0:
        names = ("q", "k", "v", "beta", "a")
        dts = {n_: (bf if n_ in ("q", "k", "v") else torch.float32) for n_ in names}
        host_sets = _pinned_sets(wl.step_inputs, min(8, nsets), dts)
        obuf0 = torch.empty(wl.batch, wl.num_v_heads, wl.head_v_dim, device=dev, dtype=bf)

        def kda_step(d, o, stream):
            dec.step(d["q"], d["k"], d["v"], d["beta"], d["a"], ci, o=o, stream=stream)

        e_ms, h2d, d2h = _e2e_pipelined(dev, dist, args.e2e_steps, host_sets,
                                        dict(zip(names, sets[0])), obuf0, kda_step)
        e2e = {"value": dist.world * wl.batch / (e_ms * 1e-3), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "KDAReplayDecoder.step (eager; one rssm_kda_step call, 3 launches); inputs "
                      "and o copied on two side streams, double-buffered"}

    full = None
    if not args.no_full_state:
        fdec = ssm.KDAFullStateDecoder(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim,
                                       wl.head_v_dim, wl.num_slots, wl.batch, act_dtype=bf,
                                       out_dtype=bf, device=dev)
        fdec.state.copy_(dec.state)
        del dec

        def full_fn(j):
            q, k, v, beta, a = sets[j]
            return lambda: fdec.step(q, k, v, beta, a, ci)

        for k in range(max(args.warmup, 3)):
            full_fn(k % G)()
        torch.cuda.synchronize()
        g_full, g_fs, fevs = _sampled_graphs([full_fn(j) for j in range(G)],
                                             [(None, full_fn(j), None) for j in range(G)])
        Kf = max(50, K // 4)
        f_el, f_per, _, _ = _timed_graphs(g_full, g_fs, fevs, Kf, dist, dev, clocks=False)
        del g_full, g_fs
        f_ms = f_el / Kf
        fb = kda_full_bytes(wl, wl.batch)
        full = {"ms_per_step": f_ms, "us_per_step": f_ms * 1e3,
                "rows_per_s": dist.world * wl.batch / (f_ms * 1e-3),
                "achieved_gbs": fb / (float(np.mean(f_per)) * 1e-3) / 1e9, "bytes_per_step": fb,
                "hbm_frac": fb / (float(np.mean(f_per)) * 1e-3) / 1e9 / peak,
                "replay_speedup": f_ms / ms_step}

    line = {
        "metric": "kda decode rows/s and µs/step at batch %d; achieved HBM GB/s" % wl.batch,
        "value": rows_s, "unit": UNIT, "n_gpus": dist.world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "us_per_step": ms_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": KDA_WORKLOAD, "global_batch": dist.world * wl.batch,
                   "batch_per_gpu": wl.batch, "HV": wl.num_v_heads, "HK": wl.num_k_heads,
                   "K": wl.head_k_dim, "V": wl.head_v_dim, "ring_len": wl.L,
                   "timing": "one CUDA graph per step (cursor + prepare + output); on every 7th step the graph also holds CUDA events around the output kernel; the kernel figures use samples covering every cursor phase equally",
                   "l2": "inputs larger than L2: 537 MB of fp32 checkpoint tiles per step"},
        "achieved_hbm_gbs": step_b / (ms_step * 1e-3) / 1e9,
        "hbm_frac_step": step_b / (ms_step * 1e-3) / 1e9 / peak,
        "bytes_per_step": int(step_b),
        "roofline": dict({"bound": "hbm", "kernel": "kda output kernel (fp32 state, 32-row tiles)",
                          "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak, "peak_source": peak_kind,
                          "traffic": traffic_record("kda.cu", "kda_output_kernel_batch256.md"),
                          "algorithmic_bytes_per_launch": int(out_b), "avg_launch_ms": out_avg_ms,
                          "launches_timed": len(out_ms), "kernel_timing": ksrc}, **split),
        "full_state": full,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clocks,
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        rate, nth, sample = cpu_oracle_rate_kda(wl, args.cpu_seconds / 3 if sub else args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": nth, "kind": "oracle",
                                "sample": sample}
    return line


M2SPEC_WORKLOAD = ("mamba2 replayssm spec verify: batch 128, T 4 drafts, H 128, P 64, N 128, G 8, "
                   "L 16, bf16 state pool 256 slots ~N(0,0.1), accepted ~U{0..4}")


def run_m2spec(args, dist, sub=False):
    """Mamba2 speculative verify rounds (prologue + verify + commit per round)."""
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    kw = {}
    if not sub and args.batch:
        kw["batch"] = args.batch
    if not sub and args.num_slots:
        kw["num_slots"] = args.num_slots
    wl = W.mamba2_spec(seed=shard_seed(args.seed, dist.rank), **kw)
    prm = wl.params()
    bf = torch.bfloat16
    T, L = wl.T, wl.L
    ci_np = wl.cache_indices()
    ci = torch.from_numpy(ci_np).to(dev)
    ver = ssm.Mamba2SpecVerifier(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, L, T, wl.num_slots,
                                 wl.batch, prm["A"], prm["D"], prm["dt_bias"], state_dtype=bf,
                                 act_dtype=bf, out_dtype=bf, device=dev)
    for s in ci_np:
        ver.state[int(s)] = torch.from_numpy(wl.slot_state(int(s))).to(dev, bf)
    nsets = min(args.input_sets, 32)
    sets, accs = [], []
    for r in range(nsets):
        inp = wl.round_inputs(r)
        sets.append([torch.from_numpy(inp[k]).to(dev, bf if k != "dt_raw" else torch.float32)
                     for k in ("x", "dt_raw", "B", "C", "z")])
        accs.append(wl.accepted(r))
    acc_dev = [torch.from_numpy(a).to(dev) for a in accs]
    torch.cuda.synchronize()
    K = args.steps
    G = min(nsets, max(K, 1))

    def round_fn(j):
        x, dt, Bm, C, z = sets[j]

        def f():
            ver.verify(x, dt, Bm, C, z, ci)
            ver.commit(ci, acc_dev[j])
        return f

    W0 = max(args.warmup, 3)
    for k in range(W0):
        round_fn(k % G)()
    torch.cuda.synchronize()
    graphs, g_rs, revs = _sampled_graphs([round_fn(j) for j in range(G)],
                                         [(None, round_fn(j), None) for j in range(G)])
    for k in range(W0):
        graphs[(W0 + k) % G].replay()
    torch.cuda.synchronize()
    offset = 2 * W0
    elapsed, per, clocks, ks = _timed_graphs(graphs, g_rs, revs, K, dist, dev, offset=offset,
                                             clocks=not sub)
    samples, ksrc = _phase_complete(per, ks, g_rs, revs, K, offset, 16)
    assert int(ver.dev_err.abs().sum().item()) == 0, "device error flag set during the m2 spec bench"
    del graphs, g_rs
    ms_round = elapsed / K
    n_run = max(K, max(k for k, _ in samples) + 1)
    seq = [accs[k % G] for k in range(offset + n_run)]
    sim, cnt_end = spec_cursor_rounds(wl.num_slots, ci_np, seq, L, T)
    dev_cnt = ver.slot_cnt.cpu().numpy().astype(np.int64)
    assert np.array_equal(dev_cnt[ci_np], cnt_end[ci_np]), "spec cursor bookkeeping disagrees"
    vb, fb = [], []
    for k, _ in samples:
        hist, fl, cr = sim[offset + k]
        v_b, f_b = m2spec_round_bytes(wl, hist, fl, cr)
        vb.append(v_b)
        fb.append(f_b)
    round_b = float(np.mean(vb)) + float(np.mean(fb))
    peak, peak_kind = read_peaks()
    per_ms = float(np.mean([ms for _, ms in samples]))

    e2e = None
    if args.e2e_steps > 0:
        names = ("x", "dt_raw", "B", "C", "z", "acc")
        dts = {n_: (torch.float32 if n_ == "dt_raw" else torch.int32 if n_ == "acc" else bf)
               for n_ in names}

        def inputs(t):
            d = dict(wl.round_inputs(t))
            d["acc"] = wl.accepted(t).astype(np.int32)
            return d

        host_sets = _pinned_sets(inputs, min(8, nsets), dts)
        ybuf0 = torch.empty(wl.batch, T, wl.nheads, wl.headdim, device=dev, dtype=bf)

        def m2spec_round(d, y, stream):
            ver.verify(d["x"], d["dt_raw"], d["B"], d["C"], d["z"], ci, y=y, stream=stream)
            ver.commit(ci, d["acc"], stream=stream)

        e_ms, h2d, d2h = _e2e_pipelined(dev, dist, args.e2e_steps, host_sets,
                                        dict(zip(names, sets[0] + [acc_dev[0]])), ybuf0,
                                        m2spec_round)
        e2e = {"value": dist.world * wl.batch / (e_ms * 1e-3), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "Mamba2SpecVerifier.verify + commit (eager; 3 launches per round); drafts, "
                      "accepted counts and y copied on two side streams, double-buffered"}
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        rate, nth, sample = cpu_oracle_rate_m2spec(wl, args.cpu_seconds / 3 if sub else
                                                   args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": nth, "kind": "oracle", "sample": sample}
    return {
        "metric": "mamba2 spec verify rows/s and µs/round at batch %d, T %d" % (wl.batch, T),
        "value": dist.world * wl.batch / (ms_round * 1e-3), "unit": UNIT,
        "draft_tokens_per_s": dist.world * wl.batch * T / (ms_round * 1e-3),
        "n_gpus": dist.world, "steps": K, "warmup": W0, "ms_per_step": ms_round,
        "us_per_round": ms_round * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": M2SPEC_WORKLOAD, "global_batch": dist.world * wl.batch,
                   "batch_per_gpu": wl.batch, "T": T, "ring_len": L,
                   "timing": "one CUDA graph per round (prologue, verify, commit)",
                   "l2": "inputs larger than L2: 268 MB of bf16 checkpoint per round"},
        "roofline": {"bound": "hbm", "kernel": "mamba2 spec round (prologue + verify + commit)",
                     "achieved": round_b / (per_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": round_b / (per_ms * 1e-3) / 1e9 / peak, "peak_source": peak_kind,
                     "traffic": traffic_record("mamba2_spec.cu", "mamba2_spec_verify_batch128_T4.md"),
                     "algorithmic_bytes_per_round": int(round_b), "avg_round_ms": per_ms,
                     "verify_bytes": float(np.mean(vb)), "fold_bytes": float(np.mean(fb)),
                     "rounds_timed": len(samples), "kernel_timing": ksrc},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": 3 * K,
        "clocks": clocks,
    }


# --------------------------------------------------------------------------- #
# gated delta net: speculative verify                                         #
# --------------------------------------------------------------------------- #

SPEC_WORKLOAD = ("gdn replayssm spec verify: batch 128, T 4 drafts, HV 32, HK 16, K=V 128, L 16, "
                 "fp32 state pool 256 slots, accepted ~U{0..4}")


def run_spec(args, dist, sub=False):
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    kw = {}
    if not sub and args.batch:
        kw["batch"] = args.batch
    if not sub and args.num_slots:
        kw["num_slots"] = args.num_slots
    wl = W.gdn_spec(seed=shard_seed(args.seed, dist.rank), **kw)
    bf = torch.bfloat16
    T, L = wl.T, wl.L
    ci_np = wl.cache_indices()
    ci = torch.from_numpy(ci_np).to(dev)
    ver = ssm.GDNSpecVerifier(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim, L, T,
                              wl.num_slots, wl.batch, act_dtype=bf, out_dtype=bf, device=dev)
    for s in ci_np:
        ver.state[int(s)] = torch.from_numpy(wl.slot_state(int(s))).to(dev)
    nsets = min(args.input_sets, 32)
    sets, accs = [], []
    for r in range(nsets):
        inp = wl.round_inputs(r)
        sets.append([torch.from_numpy(inp[k]).to(dev, bf if k in ("q", "k", "v") else torch.float32)
                     for k in ("q", "k", "v", "beta", "g")])
        accs.append(wl.accepted(r))
    acc_dev = [torch.from_numpy(a).to(dev) for a in accs]
    torch.cuda.synchronize()
    K = args.steps
    G = min(nsets, max(K, 1))

    def round_fn(j):
        q, k, v, beta, g = sets[j]

        def f():
            ver.verify(q, k, v, beta, g, ci)
            ver.commit(ci, acc_dev[j])
        return f

    W0 = max(args.warmup, 3)
    for k in range(W0):
        round_fn(k % G)()
    torch.cuda.synchronize()
    graphs, g_rs, revs = _sampled_graphs([round_fn(j) for j in range(G)],
                                         [(None, round_fn(j), None) for j in range(G)])
    for k in range(W0):
        graphs[(W0 + k) % G].replay()
    torch.cuda.synchronize()
    offset = 2 * W0
    elapsed, per, clocks, ks = _timed_graphs(graphs, g_rs, revs, K, dist, dev, offset=offset,
                                             clocks=not sub)
    samples, ksrc = _phase_complete(per, ks, g_rs, revs, K, offset, 16)
    assert int(ver.dev_err.abs().sum().item()) == 0, "device error flag set during the spec bench"
    del graphs, g_rs
    ms_round = elapsed / K
    # byte count from the cursor sequence of all rounds run so far
    n_run = max(K, max(k for k, _ in samples) + 1)
    seq = [accs[k % G] for k in range(offset + n_run)]
    sim, cnt_end = spec_cursor_rounds(wl.num_slots, ci_np, seq, L, T)
    dev_cnt = ver.slot_cnt.cpu().numpy().astype(np.int64)
    assert np.array_equal(dev_cnt[ci_np], cnt_end[ci_np]), "spec cursor bookkeeping disagrees"
    vb, fb = [], []
    for hist, fl, cr in [sim[offset + k] for k, _ in samples]:  # the sampled rounds
        vb.append(spec_round_bytes(wl, hist))
        fb.append(gdn_fold_bytes(wl, fl, cr))
    round_b = float(np.mean(vb)) + float(np.mean(fb))
    peak, peak_kind = read_peaks()
    per_ms = float(np.mean([ms for _, ms in samples]))

    e2e = None
    if args.e2e_steps > 0:
        names = ("q", "k", "v", "beta", "g", "acc")
        dts = {n_: (bf if n_ in ("q", "k", "v") else torch.int32 if n_ == "acc" else
                    torch.float32) for n_ in names}

        def inputs(t):
            d = dict(wl.round_inputs(t))
            d["acc"] = wl.accepted(t).astype(np.int32)
            return d

        host_sets = _pinned_sets(inputs, min(8, nsets), dts)
        obuf0 = torch.empty(wl.batch, T, wl.num_v_heads, wl.head_v_dim, device=dev, dtype=bf)

        def spec_round(d, o, stream):
            ver.verify(d["q"], d["k"], d["v"], d["beta"], d["g"], ci, o=o, stream=stream)
            ver.commit(ci, d["acc"], stream=stream)

        e_ms, h2d, d2h = _e2e_pipelined(dev, dist, args.e2e_steps, host_sets,
                                        dict(zip(names, sets[0] + [acc_dev[0]])), obuf0,
                                        spec_round)
        e2e = {"value": dist.world * wl.batch / (e_ms * 1e-3), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "GDNSpecVerifier.verify + commit (eager; 3 launches per round); drafts, "
                      "accepted counts and o copied on two side streams, double-buffered"}

    # the in-house conventional verify (a full-state snapshot per draft, commit copies
    # the accepted one) on an identical pool, same drafts and accepted counts
    full = None
    if not args.no_full_state:
        fver = ssm.GDNSpecFullStateVerifier(wl.num_v_heads, wl.num_k_heads, wl.head_k_dim,
                                            wl.head_v_dim, T, wl.num_slots, wl.batch, act_dtype=bf,
                                            out_dtype=bf, device=dev)
        fver.state.copy_(ver.state)
        del ver

        def full_fn(j):
            q, k, v, beta, g = sets[j]

            def f():
                fver.verify(q, k, v, beta, g, ci)
                fver.commit(ci, acc_dev[j])
            return f

        for k in range(W0):
            full_fn(k % G)()
        torch.cuda.synchronize()
        g_full, g_fs, fevs = _sampled_graphs([full_fn(j) for j in range(G)],
                                             [(None, full_fn(j), None) for j in range(G)])
        Kf = max(50, K // 4)
        f_el, _, _, _ = _timed_graphs(g_full, g_fs, fevs, Kf, dist, dev, clocks=False)
        assert int(fver.dev_err.abs().sum().item()) == 0
        del g_full, g_fs, fver
        f_ms = f_el / Kf
        HV, HK, Kd, Vd = wl.num_v_heads, wl.num_k_heads, wl.head_k_dim, wl.head_v_dim
        sab = 2 if wl.act_dtype == "bf16" else 4
        acc_mean = float(np.mean([(accs[k % G] > 0).mean() for k in range(Kf)]))
        fsb = wl.batch * (HV * Vd * Kd * 4 * (1 + T + 2 * acc_mean)
                          + T * (2 * HK * Kd * sab + HV * Vd * sab + 8 * HV + HV * Vd * 2))
        full = {"ms_per_round": f_ms, "us_per_round": f_ms * 1e3,
                "rows_per_s": dist.world * wl.batch / (f_ms * 1e-3),
                "bytes_per_round": int(fsb), "achieved_gbs": fsb / (f_ms * 1e-3) / 1e9,
                "hbm_frac": fsb / (f_ms * 1e-3) / 1e9 / peak,
                "replay_speedup": f_ms / ms_round,
                "snapshot_bytes": int(wl.batch * T * HV * Vd * Kd * 4)}

    line = {
        "metric": "gdn spec verify rows/s and µs/round at batch %d, T %d" % (wl.batch, T),
        "value": dist.world * wl.batch / (ms_round * 1e-3), "unit": UNIT,
        "draft_tokens_per_s": dist.world * wl.batch * T / (ms_round * 1e-3),
        "n_gpus": dist.world, "steps": K, "warmup": W0, "ms_per_step": ms_round,
        "us_per_round": ms_round * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": SPEC_WORKLOAD, "global_batch": dist.world * wl.batch,
                   "batch_per_gpu": wl.batch, "T": T, "ring_len": L,
                   "timing": "one CUDA graph per round (fold + tables, verify, commit)",
                   "l2": "inputs larger than L2: 268 MB of fp32 checkpoint per round"},
        "roofline": {"bound": "hbm", "kernel": "spec round (prologue + verify + commit)",
                     "achieved": round_b / (per_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": round_b / (per_ms * 1e-3) / 1e9 / peak, "peak_source": peak_kind,
                     "traffic": traffic_record("gdn_spec.cu", "gdn_spec_verify_batch128_T4.md"),
                     "algorithmic_bytes_per_round": int(round_b), "avg_round_ms": per_ms,
                     "verify_bytes": float(np.mean(vb)), "fold_bytes": float(np.mean(fb)),
                     "rounds_timed": len(samples), "kernel_timing": ksrc},
        "full_state": full,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clocks,
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        rate, nth, sample = cpu_oracle_rate_spec(wl, args.cpu_seconds / 3 if sub else
                                                 args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": nth, "kind": "oracle",
                                "sample": sample}
    return line


# --------------------------------------------------------------------------- #
# Mamba2 sweep                                                                #
# --------------------------------------------------------------------------- #

SWEEP_BATCH = (1, 16, 64, 128, 256, 512, 1024)
SWEEP_L = (1, 4, 8, 16)
SWEEP_DT = ("fp32", "bf16")


def sweep_point(args, dist, dev, batch, L, sdt, K):
    """One Mamba2 sweep point (config-2 geometry: H 128, P 64, N 128, G 8, 5% of rows
    force-flushed per step): the ReplaySSM step (one CUDA graph per step) and the
    full-state kernel on an identical pool, K timed steps each. The pool is filled on
    the device from a seeded generator."""
    import torch

    import rssm_workloads as W
    import ssm_linear_attention_gb300 as ssm

    peak, _ = read_peaks()
    bf = torch.bfloat16
    st = torch.float32 if sdt == "fp32" else bf
    wl = W.mamba2_sweep(batch, L, sdt, seed=shard_seed(args.seed, dist.rank))
    prm = wl.params()
    ci_np = wl.cache_indices()
    ci = torch.from_numpy(ci_np).to(dev)
    dec = ssm.Mamba2ReplayDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups, L,
                                  wl.num_slots, batch, prm["A"], prm["D"],
                                  prm["dt_bias"], state_dtype=st, act_dtype=bf,
                                  out_dtype=bf, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(shard_seed(args.seed, dist.rank) + batch * 131 + L)
    dec.state.normal_(0.0, 0.1, generator=gen)
    nsets = 8
    sets = []
    for t in range(nsets):
        inp = wl.step_inputs(t)
        xs = [torch.from_numpy(inp[k]).to(dev, bf if k != "dt_raw" else torch.float32)
              for k in ("x", "dt_raw", "B", "C", "z")]
        fm = wl.force_mask(t)
        xs.append(None if fm is None else torch.from_numpy(fm).to(dev))
        sets.append(xs)
    torch.cuda.synchronize()

    def rep_fn(j):
        x, dt, Bm, C, z, fm = sets[j]
        return lambda: dec.step(x, dt, Bm, C, z, ci, force_flush=fm)

    for k in range(3):
        rep_fn(k % nsets)()
    g_rep = _graphs([rep_fn(j) for j in range(nsets)])
    for k in range(3):
        g_rep[k].replay()
    el, _, _, _ = _timed_graphs(g_rep, g_rep, [(None, None)] * nsets, K, dist, dev,
                                clocks=False, every=K + 1)
    assert int(dec.dev_err.abs().sum().item()) == 0
    del g_rep
    rep_ms = el / K
    fdec = ssm.Mamba2FullStateDecoder(wl.nheads, wl.headdim, wl.dstate, wl.ngroups,
                                      wl.num_slots, batch, prm["A"], prm["D"],
                                      prm["dt_bias"], state_dtype=st, act_dtype=bf,
                                      out_dtype=bf, device=dev)
    fdec.state.copy_(dec.state)
    del dec

    def full_fn(j):
        x, dt, Bm, C, z, fm = sets[j]
        return lambda: fdec.step(x, dt, Bm, C, z, ci)

    for k in range(3):
        full_fn(k % nsets)()
    g_full = _graphs([full_fn(j) for j in range(nsets)])
    for k in range(3):
        g_full[k].replay()
    fel, _, _, _ = _timed_graphs(g_full, g_full, [(None, None)] * nsets, K, dist, dev,
                                 clocks=False, every=K + 1)
    del g_full, fdec
    full_ms = fel / K
    fb = full_state_bytes(wl, batch)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
    tile_bytes = batch * wl.nheads * wl.headdim * wl.dstate * (4 if sdt == "fp32" else 2)
    del sets
    torch.cuda.empty_cache()
    return {"batch": batch, "ring_len": L, "state_dtype": sdt, "steps": K,
            "state_bytes_per_step": tile_bytes,
            "possibly_l2_resident": bool(l2 and tile_bytes <= l2),
            "replay_us_per_step": rep_ms * 1e3,
            "replay_rows_per_s": dist.world * batch / (rep_ms * 1e-3),
            "full_state_us_per_step": full_ms * 1e3,
            "full_state_gbs": fb / (full_ms * 1e-3) / 1e9,
            "full_state_hbm_frac": fb / (full_ms * 1e-3) / 1e9 / peak,
            "replay_speedup": full_ms / rep_ms}


SWEEP_BATCH = (1, 16, 64, 128, 256, 512, 1024)
SWEEP_L = (1, 4, 8, 16)
SWEEP_DT = ("fp32", "bf16")
# the points the default line carries: the batches the bar names (>= 64) at both ends
# of the ring lengths, both state dtypes
SWEEP_DEFAULT = [(b, L, d) for d in SWEEP_DT for L in (1, 16) for b in (64, 1024)]


def run_sweep(args, dist):
    """One JSON line per (batch, L, state dtype) of the Mamba2 sweep, each point beside
    the full-state kernel."""
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    for sdt in SWEEP_DT:
        for L in SWEEP_L:
            for batch in SWEEP_BATCH:
                pt = sweep_point(args, dist, dev, batch, L, sdt, args.sweep_steps)
                line = dict({"metric": "mamba2 sweep point", "workload": "sweep",
                             "n_gpus": dist.world,
                             "timing": "one CUDA graph per step (2 launches); full state one graph"},
                            **pt)
                if dist.rank == 0:
                    print(json.dumps(line), flush=True)
    return None


def run_sweep_sub(args, dist):
    """The compact sweep of the default line: SWEEP_DEFAULT's points."""
    import ssm_linear_attention_gb300 as ssm

    dev = _device(dist)
    ssm.lib()
    pts = [sweep_point(args, dist, dev, b, L, d, args.sweep_sub_steps) for b, L, d in SWEEP_DEFAULT]
    return {"workload": "mamba2 sweep (H 128, P 64, N 128, G 8, 5% forced flushes per step), "
                        "ReplaySSM step beside the full-state kernel on an identical pool",
            "timing": "one CUDA graph per step; %d timed steps per point and kernel"
                      % args.sweep_sub_steps,
            "points": pts}


def run_reference(args, dist):
    """The oracle arm: the float64 CPU recurrence on this host's cores; each step a
    bounded sample of the workload's rows."""
    import rssm_workloads as W
    import oracle
    wl = W.mamba2_large(batch=args.batch or 512, seed=args.seed)
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
    global EVENT_EVERY
    args = parse()
    if args.source_hash:
        print(source_hash(args.source_hash))
        return
    EVENT_EVERY = max(1, args.event_every)
    dist = Dist()
    try:
        if args.impl == "reference":
            if dist.rank != 0:
                return
            if args.steps > 50:
                args.steps = 50
            line = run_reference(args, dist)
        elif args.workload == "gdn":
            line = run_gdn(args, dist)
        elif args.workload == "spec":
            line = run_spec(args, dist)
        elif args.workload == "kda":
            line = run_kda(args, dist)
        elif args.workload == "m2spec":
            line = run_m2spec(args, dist)
        elif args.workload == "sweep":
            line = run_sweep(args, dist)
        else:
            line = run_mamba2(args, dist)
            if not args.no_gdn:
                line["gdn_decode"] = run_gdn(args, dist, sub=True)
                line["gdn_spec"] = run_spec(args, dist, sub=True)
                line["kda_decode"] = run_kda(args, dist, sub=True)
                line["mamba2_spec"] = run_m2spec(args, dist, sub=True)
            if not args.no_sweep:
                line["mamba2_sweep"] = run_sweep_sub(args, dist)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
