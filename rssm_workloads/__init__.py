"""Seeded synthetic inputs for ReplaySSM decode workloads.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA side
(tests, benchmark, smoke check). It holds the input recipe only: shapes, value
distributions, slot maps, initial cursors and force-flush masks. None of the
method's arithmetic lives here: softplus of dt, decays, dot products and state
updates belong to the two implementations.

Every array is drawn from numpy's PCG64 through a SeedSequence keyed by
(seed, stream tag, index), so any step or slot can be regenerated on its own and
both sides see identical numbers. Values are returned as float32 arrays that are
exactly representable in their storage dtype ("bf16" values are rounded to
bfloat16, ties to even, before they are returned).

Workload recipes (the pages print no benchmark inputs; these follow the
distributions of the decode workloads the pages describe: Mamba2 state
[nheads, headdim, dstate] per slot with ngroups shared B/C, and gated delta net
state [HV, V, K] with grouped key heads):
  mamba2_tiny   batch 4, nheads 8, headdim 64, dstate 128, ngroups 1, L 4,
                16 steps, fp32 state and activations, zero state, slots 0..3.
  mamba2_large  batch 512, nheads 128, headdim 64, dstate 128, ngroups 8, L 16,
                64 steps, bf16 state N(0, 0.1), 1024 slots, cache indices the first
                512 of a seeded permutation, initial write_pos ~ U{0..15}.
  mamba2_sweep  batch in {1,16,64,128,256,512,1024} x L in {1,4,8,16} x state
                {fp32, bf16}, 32 steps, 5% seeded forced flushes per step.
  gdn_decode    batch 256, HV 32, HK 16, K = V = 128, L 16, 64 steps, fp32 state
                N(0, 0.05), 512 slots, q and k L2-normalised per head.
  gdn_spec      batch 128, T 4 drafts per round, L 16, 32 rounds, accepted drafts
                ~ U{0..4} per row and round.
  kda_decode    gdn_decode's geometry with a per-key-channel gate a [HV, K] per
                step instead of the scalar g.
  mamba2_spec   mamba2_large's geometry, batch 128, 256 slots, T 4 drafts per verify
                round, L 16, accepted drafts ~ U{0..4}.
"""
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

__all__ = [
    "round_bf16_f32", "Mamba2Workload", "GDNWorkload", "GDNSpecWorkload",
    "mamba2_tiny", "mamba2_large", "mamba2_sweep", "gdn_decode", "gdn_spec", "kda_decode",
    "KDAWorkload", "Mamba2SpecWorkload", "mamba2_spec",
]

# stream tags
_T_PARAMS, _T_STATE, _T_STEP, _T_HIST, _T_FORCE, _T_CI, _T_WP, _T_ACC = range(1, 9)


def _rng(seed: int, tag: int, idx: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, idx])))


def round_bf16_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.
    Finite values and infinities only (the sum below stays inside 32 bits for every
    such bit pattern; the inputs never hold NaN)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    r = (u >> 16) & 1
    r += 0x7FFF
    r += u
    r &= 0xFFFF0000
    return r.view(np.float32)


def _to_grid(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    return round_bf16_f32(a) if dtype == "bf16" else a


def _normal(rng, shape, std=1.0):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


# --------------------------------------------------------------------------- #
# Mamba2                                                                      #
# --------------------------------------------------------------------------- #

@dataclass
class Mamba2Workload:
    batch: int
    nheads: int = 128
    headdim: int = 64
    dstate: int = 128
    ngroups: int = 8
    L: int = 16
    num_slots: int = 1024
    steps: int = 64
    state_dtype: str = "bf16"     # "fp32" | "bf16"
    act_dtype: str = "bf16"       # x, z, B, C
    state_init: str = "normal"    # "zero" | "normal"
    state_std: float = 0.1
    ci_mode: str = "perm"         # "perm" | "arange"
    wp_mode: str = "uniform"      # "zero" | "uniform"
    force_rate: float = 0.0
    with_z: bool = True
    dt_softplus: bool = True
    seed: int = 0
    name: str = "mamba2"
    _cache: Dict = field(default_factory=dict, repr=False)

    # per-head parameters: A = -exp(U(0, ln 16)), D ~ N(0, 1), dt_bias ~ U(-4, -2)
    def params(self):
        if "params" not in self._cache:
            r = _rng(self.seed, _T_PARAMS)
            H = self.nheads
            A = -np.exp(r.uniform(0.0, np.log(16.0), H)).astype(np.float32)
            D = r.standard_normal(H).astype(np.float32)
            dt_bias = r.uniform(-4.0, -2.0, H).astype(np.float32)
            self._cache["params"] = dict(A=A, D=D, dt_bias=dt_bias)
        return self._cache["params"]

    def cache_indices(self) -> np.ndarray:
        if "ci" not in self._cache:
            if self.ci_mode == "arange":
                ci = np.arange(self.batch, dtype=np.int32)
            else:
                ci = _rng(self.seed, _T_CI).permutation(self.num_slots)[: self.batch].astype(np.int32)
            self._cache["ci"] = ci
        return self._cache["ci"]

    def history_len(self) -> np.ndarray:
        """Per-row number of steps already in the ring when the measured steps start
        (the row's initial write_pos)."""
        if "wp" not in self._cache:
            if self.wp_mode == "zero" or self.L == 1:
                wp = np.zeros(self.batch, dtype=np.int32)
            else:
                wp = _rng(self.seed, _T_WP).integers(0, self.L, self.batch).astype(np.int32)
            self._cache["wp"] = wp
        return self._cache["wp"]

    def slot_state(self, s: int) -> np.ndarray:
        """Initial state of slot s: [nheads, headdim, dstate] on the state dtype grid."""
        shp = (self.nheads, self.headdim, self.dstate)
        if self.state_init == "zero":
            return np.zeros(shp, dtype=np.float32)
        return _to_grid(_normal(_rng(self.seed, _T_STATE, s), shp, self.state_std), self.state_dtype)

    def _inputs(self, rng):
        B_, H, P, N, G = self.batch, self.nheads, self.headdim, self.dstate, self.ngroups
        x = _to_grid(_normal(rng, (B_, H, P)), self.act_dtype)
        dt_raw = rng.standard_normal((B_, H), dtype=np.float32)
        Bm = _to_grid(_normal(rng, (B_, G, N), 1.0 / np.sqrt(N)), self.act_dtype)
        Cm = _to_grid(_normal(rng, (B_, G, N), 1.0 / np.sqrt(N)), self.act_dtype)
        z = _to_grid(_normal(rng, (B_, H, P)), self.act_dtype) if self.with_z else None
        return dict(x=x, dt_raw=dt_raw, B=Bm, C=Cm, z=z)

    def step_inputs(self, t: int):
        """Inputs of measured step t: x [b,H,P], dt_raw [b,H], B, C [b,G,N], z [b,H,P]."""
        return self._inputs(_rng(self.seed, _T_STEP, t))

    def history_inputs(self, j: int):
        """Inputs of history step j (only rows with history_len > j take part)."""
        return self._inputs(_rng(self.seed, _T_HIST, j))

    def history_ci(self, j: int) -> np.ndarray:
        """Cache indices for history step j: rows without a j-th history entry are
        padding (-1)."""
        ci = self.cache_indices().copy()
        ci[self.history_len() <= j] = -1
        return ci

    def force_mask(self, t: int) -> Optional[np.ndarray]:
        if self.force_rate <= 0.0:
            return None
        r = _rng(self.seed, _T_FORCE, t)
        return (r.random(self.batch) < self.force_rate).astype(np.uint8)

    def max_history(self) -> int:
        return int(self.history_len().max()) if self.batch else 0


def mamba2_tiny(**kw) -> Mamba2Workload:
    d = dict(batch=4, nheads=8, headdim=64, dstate=128, ngroups=1, L=4, num_slots=4, steps=16,
             state_dtype="fp32", act_dtype="fp32", state_init="zero", ci_mode="arange",
             wp_mode="zero", name="mamba2_tiny")
    d.update(kw)
    return Mamba2Workload(**d)


def mamba2_large(**kw) -> Mamba2Workload:
    d = dict(batch=512, nheads=128, headdim=64, dstate=128, ngroups=8, L=16, num_slots=1024,
             steps=64, state_dtype="bf16", act_dtype="bf16", state_init="normal", state_std=0.1,
             ci_mode="perm", wp_mode="uniform", name="mamba2_large")
    d.update(kw)
    return Mamba2Workload(**d)


def mamba2_sweep(batch: int, L: int, state_dtype: str, **kw) -> Mamba2Workload:
    d = dict(batch=batch, nheads=128, headdim=64, dstate=128, ngroups=8, L=L, num_slots=1024,
             steps=32, state_dtype=state_dtype, act_dtype="bf16", state_init="normal",
             state_std=0.1, ci_mode="perm", wp_mode="uniform", force_rate=0.05,
             name="mamba2_sweep_b%d_L%d_%s" % (batch, L, state_dtype))
    d.update(kw)
    return Mamba2Workload(**d)


# --------------------------------------------------------------------------- #
# Gated delta net                                                             #
# --------------------------------------------------------------------------- #

def _unit_rows(a: np.ndarray) -> np.ndarray:
    """L2-normalise the last axis in float64 (q and k recipe)."""
    a = a.astype(np.float64)
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


@dataclass
class GDNWorkload:
    batch: int
    num_v_heads: int = 32
    num_k_heads: int = 16
    head_k_dim: int = 128
    head_v_dim: int = 128
    L: int = 16
    num_slots: int = 512
    steps: int = 64
    act_dtype: str = "bf16"       # q, k, v
    state_std: float = 0.05
    ci_mode: str = "perm"
    wp_mode: str = "zero"
    force_rate: float = 0.0
    seed: int = 0
    name: str = "gdn"
    _cache: Dict = field(default_factory=dict, repr=False)

    def cache_indices(self) -> np.ndarray:
        if "ci" not in self._cache:
            if self.ci_mode == "arange":
                ci = np.arange(self.batch, dtype=np.int32)
            else:
                ci = _rng(self.seed, _T_CI).permutation(self.num_slots)[: self.batch].astype(np.int32)
            self._cache["ci"] = ci
        return self._cache["ci"]

    def history_len(self) -> np.ndarray:
        if "wp" not in self._cache:
            if self.wp_mode == "zero" or self.L == 1:
                wp = np.zeros(self.batch, dtype=np.int32)
            else:
                wp = _rng(self.seed, _T_WP).integers(0, self.L, self.batch).astype(np.int32)
            self._cache["wp"] = wp
        return self._cache["wp"]

    def max_history(self) -> int:
        return int(self.history_len().max()) if self.batch else 0

    def slot_state(self, s: int) -> np.ndarray:
        """Initial fp32 state of slot s: [HV, V, K] ~ N(0, state_std)."""
        shp = (self.num_v_heads, self.head_v_dim, self.head_k_dim)
        return _normal(_rng(self.seed, _T_STATE, s), shp, self.state_std)

    def _token_inputs(self, rng, lead):
        HV, HK, K, V = self.num_v_heads, self.num_k_heads, self.head_k_dim, self.head_v_dim
        q = _to_grid(_unit_rows(rng.standard_normal(lead + (HK, K))), self.act_dtype)
        k = _to_grid(_unit_rows(rng.standard_normal(lead + (HK, K))), self.act_dtype)
        v = _to_grid(rng.standard_normal(lead + (HV, V), dtype=np.float32), self.act_dtype)
        beta = (1.0 / (1.0 + np.exp(-rng.standard_normal(lead + (HV,))))).astype(np.float32)
        a = rng.standard_normal(lead + (HV,)) + 1.0
        softplus_a = np.where(a > 0, a + np.log1p(np.exp(-np.abs(a))), np.log1p(np.exp(a)))
        g = np.exp(-softplus_a).astype(np.float32)
        return dict(q=q, k=k, v=v, beta=beta, g=g)

    def step_inputs(self, t: int):
        """q, k [b,HK,K]; v [b,HV,V]; beta, g [b,HV] (g is the gate value in (0, 1))."""
        return self._token_inputs(_rng(self.seed, _T_STEP, t), (self.batch,))

    def history_inputs(self, j: int):
        return self._token_inputs(_rng(self.seed, _T_HIST, j), (self.batch,))

    def history_ci(self, j: int) -> np.ndarray:
        ci = self.cache_indices().copy()
        ci[self.history_len() <= j] = -1
        return ci

    def force_mask(self, t: int) -> Optional[np.ndarray]:
        if self.force_rate <= 0.0:
            return None
        r = _rng(self.seed, _T_FORCE, t)
        return (r.random(self.batch) < self.force_rate).astype(np.uint8)


@dataclass
class GDNSpecWorkload(GDNWorkload):
    T: int = 4
    rounds: int = 32

    def round_inputs(self, r: int):
        """Draft inputs of verify round r: q, k [b,T,HK,K]; v [b,T,HV,V]; beta, g [b,T,HV]."""
        return self._token_inputs(_rng(self.seed, _T_STEP, r), (self.batch, self.T))

    def accepted(self, r: int) -> np.ndarray:
        """Accepted draft count per row for round r, U{0..T}."""
        return _rng(self.seed, _T_ACC, r).integers(0, self.T + 1, self.batch).astype(np.int32)


@dataclass
class Mamba2SpecWorkload(Mamba2Workload):
    """Mamba2 geometry with T draft tokens per verify round; accepted ~ U{0..T}."""
    T: int = 4
    rounds: int = 32

    def round_inputs(self, r: int):
        """Draft inputs of round r: x, z [b,T,H,P]; dt_raw [b,T,H]; B, C [b,T,G,N]."""
        rng = _rng(self.seed, _T_STEP, r)
        B_, T, H, P, N, G = self.batch, self.T, self.nheads, self.headdim, self.dstate, self.ngroups
        x = _to_grid(_normal(rng, (B_, T, H, P)), self.act_dtype)
        dt_raw = rng.standard_normal((B_, T, H), dtype=np.float32)
        Bm = _to_grid(_normal(rng, (B_, T, G, N), 1.0 / np.sqrt(N)), self.act_dtype)
        Cm = _to_grid(_normal(rng, (B_, T, G, N), 1.0 / np.sqrt(N)), self.act_dtype)
        z = _to_grid(_normal(rng, (B_, T, H, P)), self.act_dtype) if self.with_z else None
        return dict(x=x, dt_raw=dt_raw, B=Bm, C=Cm, z=z)

    def accepted(self, r: int) -> np.ndarray:
        return _rng(self.seed, _T_ACC, r).integers(0, self.T + 1, self.batch).astype(np.int32)


def mamba2_spec(**kw) -> Mamba2SpecWorkload:
    d = dict(batch=128, nheads=128, headdim=64, dstate=128, ngroups=8, L=16, num_slots=256,
             T=4, rounds=32, steps=0, state_dtype="bf16", act_dtype="bf16", state_init="normal",
             state_std=0.1, ci_mode="perm", wp_mode="zero", name="mamba2_spec")
    d.update(kw)
    return Mamba2SpecWorkload(**d)


@dataclass
class KDAWorkload(GDNWorkload):
    """GDN geometry with a per-key-channel gate a [.., HV, K] in (0, 1) instead of the
    scalar g: a = exp(-softplus(N(0, 1) - 2)) per element (mean ~0.87, so ring
    entries several steps old still matter)."""
    name: str = "kda"

    def _token_inputs(self, rng, lead):
        d = GDNWorkload._token_inputs(self, rng, lead)
        x = rng.standard_normal(lead + (self.num_v_heads, self.head_k_dim)) - 2.0
        sp = np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(x)))
        d["a"] = np.exp(-sp).astype(np.float32)
        return d


def kda_decode(**kw) -> KDAWorkload:
    d = dict(batch=256, num_v_heads=32, num_k_heads=16, head_k_dim=128, head_v_dim=128, L=16,
             num_slots=512, steps=64, act_dtype="bf16", state_std=0.05, name="kda_decode")
    d.update(kw)
    return KDAWorkload(**d)


def gdn_decode(**kw) -> GDNWorkload:
    d = dict(batch=256, num_v_heads=32, num_k_heads=16, head_k_dim=128, head_v_dim=128, L=16,
             num_slots=512, steps=64, act_dtype="bf16", state_std=0.05, name="gdn_decode")
    d.update(kw)
    return GDNWorkload(**d)


def gdn_spec(**kw) -> GDNSpecWorkload:
    d = dict(batch=128, num_v_heads=32, num_k_heads=16, head_k_dim=128, head_v_dim=128, L=16,
             num_slots=256, T=4, rounds=32, steps=0, act_dtype="bf16", state_std=0.05,
             name="gdn_spec")
    d.update(kw)
    return GDNSpecWorkload(**d)
