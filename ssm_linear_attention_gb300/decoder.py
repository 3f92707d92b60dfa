"""Decode-step runners over the C ABI.

Each runner owns the device buffers of one layer's ReplaySSM state on the current
CUDA device (allocated with torch: the slot-indexed checkpoint pool, the input
rings, the per-slot cursors, the per-row cursor outputs, the workspace), and a
step is the sequence of librssm calls the method needs, in stream order:

  Mamba2 decode:  rssm_mamba2_step = rssm_mamba2_prepare (cursor advance,
                  ring append, tables: one launch) -> rssm_mamba2_output; or the
                  four calls rssm_advance_cursors (STANDARD) -> rssm_ring_append ->
                  rssm_mamba2_precompute -> rssm_mamba2_output
  GDN decode:     rssm_gdn_step = rssm_gdn_prepare (one launch) ->
                  rssm_gdn_output; or the four calls rssm_advance_cursors
                  (STANDARD) -> rssm_gdn_ring_append -> rssm_gdn_precompute ->
                  rssm_gdn_output
  GDN spec:       rssm_gdn_spec_verify (fold + verify), then
                  rssm_advance_cursors (SPEC_COMMIT) with the accepted counts

No host synchronisation happens inside a step, so a step can be captured in a
CUDA graph. Several layers that share slots can share one cursor advance
(``advance=False`` on all but one layer, with ``row_wp`` / ``row_flush`` shared).
"""
import torch

from . import _binding as B

__all__ = ["torch_dtype_code", "Mamba2ReplayDecoder", "Mamba2FullStateDecoder",
           "GDNReplayDecoder", "GDNFullStateDecoder", "GDNSpecVerifier",
           "GDNSpecFullStateVerifier"]


def _sr_state(seed, device):
    """Device {seed, offset} pair (uint64 bits kept in int64) for stochastic rounding,
    or None for round-to-nearest."""
    if seed is None:
        return None
    s = int(seed) & (2 ** 64 - 1)
    s = s - 2 ** 64 if s >= 2 ** 63 else s
    return torch.tensor([s, 0], device=device, dtype=torch.int64)


def torch_dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return B.RSSM_F32
    if dt == torch.bfloat16:
        return B.RSSM_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % dt)


class Mamba2ReplayDecoder:
    """ReplaySSM Mamba2 decode for one layer.

    Buffers: state [num_slots, H, P, N] (state_dtype), ring_x [num_slots, H, L, P],
    ring_dt [num_slots, H, L] float32, ring_B [num_slots, G, L, N], slot_wp
    [num_slots] int32, and per-row row_wp / row_flush / workspace / y for up to
    max_batch rows. With sr_seed set, bf16 state stores round stochastically
    (Philox4x32-10 bits from {sr_seed, offset}; the offset advances each call)."""

    def __init__(self, nheads, headdim, dstate, ngroups, ring_len, num_slots, max_batch, A, D,
                 dt_bias=None, dt_softplus=True, state_dtype=torch.bfloat16,
                 act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None, sr_seed=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.H, self.P, self.N, self.G, self.L = nheads, headdim, dstate, ngroups, ring_len
        self.num_slots, self.max_batch = num_slots, max_batch
        self.state_dtype, self.act_dtype, self.out_dtype = state_dtype, act_dtype, out_dtype
        self.dt_softplus = dt_softplus
        f32 = dict(device=dev, dtype=torch.float32)
        self.A = torch.as_tensor(A, **f32).contiguous()
        self.D = torch.as_tensor(D, **f32).contiguous()
        self.dt_bias = None if dt_bias is None else torch.as_tensor(dt_bias, **f32).contiguous()
        self.state = torch.zeros(num_slots, nheads, headdim, dstate, device=dev, dtype=state_dtype)
        self.ring_x = torch.zeros(num_slots, nheads, ring_len, headdim, device=dev, dtype=act_dtype)
        self.ring_dt = torch.zeros(num_slots, nheads, ring_len, **f32)
        self.ring_B = torch.zeros(num_slots, ngroups, ring_len, dstate, device=dev, dtype=act_dtype)
        self.slot_wp = torch.zeros(num_slots, device=dev, dtype=torch.int32)
        self.row_wp = torch.zeros(max_batch, device=dev, dtype=torch.int32)
        self.row_flush = torch.zeros(max_batch, device=dev, dtype=torch.uint8)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.ws_bytes = B.rssm_mamba2_workspace_size(self.dims(max_batch))
        # zero-filled: the one-launch small-batch step keeps per-row counters here
        self.workspace = torch.zeros(max(self.ws_bytes, 16), device=dev, dtype=torch.uint8)
        self.y = torch.empty(max_batch, nheads, headdim, device=dev, dtype=out_dtype)
        self.sr = _sr_state(sr_seed, dev)

    def dims(self, batch):
        return B.Mamba2Dims(batch, self.H, self.P, self.N, self.G, self.L, self.num_slots,
                            torch_dtype_code(self.state_dtype), torch_dtype_code(self.act_dtype),
                            torch_dtype_code(self.out_dtype))

    # individual stages (bench.py times them separately)
    def advance(self, cache_indices, force_flush=None, stream=None):
        b = cache_indices.shape[0]
        B.rssm_advance_cursors(B.RSSM_CURSOR_STANDARD, self.slot_wp, None, None, cache_indices,
                               force_flush, None, b, self.num_slots, self.L, 0, self.row_wp,
                               self.row_flush, self.dev_err, stream)

    def append(self, x, dt_raw, Bm, cache_indices, stream=None):
        B.rssm_ring_append(self.dims(x.shape[0]), x, dt_raw, self.dt_bias, self.dt_softplus, Bm,
                           cache_indices, self.row_wp, self.ring_x, self.ring_dt, self.ring_B,
                           self.dev_err, stream)

    def precompute(self, C, cache_indices, stream=None):
        B.rssm_mamba2_precompute(self.dims(C.shape[0]), self.A, C, self.ring_dt, self.ring_B,
                                 cache_indices, self.row_wp, self.workspace, self.ws_bytes,
                                 self.dev_err, stream)

    def output(self, C, z, cache_indices, y=None, stream=None):
        b = C.shape[0]
        y = self.y[:b] if y is None else y
        if self.sr is not None:
            B.rssm_mamba2_output_sr(self.dims(b), self.state, C, self.D, z, self.ring_x,
                                    self.ring_B, cache_indices, self.row_wp, self.row_flush,
                                    self.workspace, self.ws_bytes, y, self.sr, self.dev_err,
                                    stream)
            return y
        B.rssm_mamba2_output(self.dims(b), self.state, C, self.D, z, self.ring_x, self.ring_B,
                             cache_indices, self.row_wp, self.row_flush, self.workspace,
                             self.ws_bytes, y, self.dev_err, stream)
        return y

    def prepare(self, x, dt_raw, Bm, C, cache_indices, force_flush=None, stream=None,
                advance=True):
        """Cursor advance (unless advance=False), ring append and tables in one launch."""
        B.rssm_mamba2_prepare(self.dims(x.shape[0]), advance, force_flush, self.slot_wp,
                              self.row_wp, self.row_flush, x, dt_raw, self.dt_bias,
                              self.dt_softplus, Bm, self.A, C, cache_indices, self.ring_x,
                              self.ring_dt, self.ring_B, self.workspace, self.ws_bytes,
                              self.dev_err, stream)

    def step(self, x, dt_raw, Bm, C, z, cache_indices, force_flush=None, y=None, stream=None,
             advance=True):
        """One decode step for rows cache_indices (padding rows: -1), as one
        rssm_mamba2_step call (two launches). Returns y [b, H, P]."""
        b = x.shape[0]
        y = self.y[:b] if y is None else y
        if self.sr is not None:
            B.rssm_mamba2_step_sr(self.dims(b), advance, force_flush, self.slot_wp, self.row_wp,
                                  self.row_flush, self.state, x, dt_raw, self.dt_bias,
                                  self.dt_softplus, self.A, Bm, C, self.D, z, cache_indices,
                                  self.ring_x, self.ring_dt, self.ring_B, self.workspace,
                                  self.ws_bytes, y, self.sr, self.dev_err, stream)
            return y
        B.rssm_mamba2_step(self.dims(b), advance, force_flush, self.slot_wp, self.row_wp,
                           self.row_flush, self.state, x, dt_raw, self.dt_bias, self.dt_softplus,
                           self.A, Bm, C, self.D, z, cache_indices, self.ring_x, self.ring_dt,
                           self.ring_B, self.workspace, self.ws_bytes, y, self.dev_err, stream)
        return y

    def step_staged(self, x, dt_raw, Bm, C, z, cache_indices, force_flush=None, y=None,
                    stream=None, advance=True):
        """The same step as four calls (cursor, append, precompute, output)."""
        if advance:
            self.advance(cache_indices, force_flush, stream)
        self.append(x, dt_raw, Bm, cache_indices, stream)
        self.precompute(C, cache_indices, stream)
        return self.output(C, z, cache_indices, y, stream)

    def reset_slots(self, slots, stream=None):
        B.rssm_advance_cursors(B.RSSM_CURSOR_RESET, self.slot_wp, None, None, slots, None, None,
                               slots.shape[0], self.num_slots, self.L, 0, None, None, self.dev_err,
                               stream)

    def copy_slots(self, src, dst, stream=None):
        """Fork: slot dst[i] becomes a copy of slot src[i] (checkpoint, rings, cursor)."""
        B.rssm_copy_slots([self.state, self.ring_x, self.ring_dt, self.ring_B, self.slot_wp],
                          src, dst, src.shape[0], self.num_slots, self.dev_err, stream)

    def materialize(self, slots, out=None, stream=None):
        """Current fp32 state of the listed slots [n, H, P, N] (checkpoint folded with the
        live ring entries); pool, rings and cursors are left untouched."""
        n = slots.shape[0]
        if out is None:
            out = torch.empty(n, self.H, self.P, self.N, device=self.state.device,
                              dtype=torch.float32)
        B.rssm_mamba2_materialize_state(self.dims(n), self.state, self.A, self.ring_x,
                                        self.ring_dt, self.ring_B, slots, self.slot_wp, out,
                                        self.dev_err, stream)
        return out


class Mamba2FullStateDecoder:
    """The conventional Mamba2 decode step (whole state read and written every step);
    sr_seed as in Mamba2ReplayDecoder."""

    def __init__(self, nheads, headdim, dstate, ngroups, num_slots, max_batch, A, D, dt_bias=None,
                 dt_softplus=True, state_dtype=torch.bfloat16, act_dtype=torch.bfloat16,
                 out_dtype=torch.bfloat16, device=None, sr_seed=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.H, self.P, self.N, self.G = nheads, headdim, dstate, ngroups
        self.num_slots = num_slots
        self.state_dtype, self.act_dtype, self.out_dtype = state_dtype, act_dtype, out_dtype
        self.dt_softplus = dt_softplus
        f32 = dict(device=dev, dtype=torch.float32)
        self.A = torch.as_tensor(A, **f32).contiguous()
        self.D = torch.as_tensor(D, **f32).contiguous()
        self.dt_bias = None if dt_bias is None else torch.as_tensor(dt_bias, **f32).contiguous()
        self.state = torch.zeros(num_slots, nheads, headdim, dstate, device=dev, dtype=state_dtype)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.y = torch.empty(max_batch, nheads, headdim, device=dev, dtype=out_dtype)
        self.sr = _sr_state(sr_seed, dev)

    def dims(self, batch):
        return B.Mamba2Dims(batch, self.H, self.P, self.N, self.G, 1, self.num_slots,
                            torch_dtype_code(self.state_dtype), torch_dtype_code(self.act_dtype),
                            torch_dtype_code(self.out_dtype))

    def step(self, x, dt_raw, Bm, C, z, cache_indices, y=None, stream=None):
        b = x.shape[0]
        y = self.y[:b] if y is None else y
        if self.sr is not None:
            B.rssm_mamba2_full_state_update_sr(self.dims(b), self.state, x, dt_raw, self.dt_bias,
                                               self.dt_softplus, self.A, Bm, C, self.D, z,
                                               cache_indices, y, self.sr, self.dev_err, stream)
            return y
        B.rssm_mamba2_full_state_update(self.dims(b), self.state, x, dt_raw, self.dt_bias,
                                        self.dt_softplus, self.A, Bm, C, self.D, z, cache_indices,
                                        y, self.dev_err, stream)
        return y


class GDNReplayDecoder:
    """ReplaySSM gated-delta-net decode for one layer.

    Buffers: state [num_slots, HV, V, K] float32, ring_d [num_slots, HV, V/32, L, 32]
    float32 (value rows in blocks of 32), ring_k [num_slots, HK, L, K] (act dtype), ring_g [num_slots, HV, L]
    float32, slot_wp [num_slots] int32."""

    def __init__(self, num_v_heads, num_k_heads, head_k_dim, head_v_dim, ring_len, num_slots,
                 max_batch, act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.HV, self.HK, self.K, self.V, self.L = (num_v_heads, num_k_heads, head_k_dim,
                                                    head_v_dim, ring_len)
        self.num_slots, self.max_batch = num_slots, max_batch
        self.act_dtype, self.out_dtype = act_dtype, out_dtype
        f32 = dict(device=dev, dtype=torch.float32)
        self.state = torch.zeros(num_slots, num_v_heads, head_v_dim, head_k_dim, **f32)
        self.ring_d = torch.zeros(num_slots, num_v_heads, head_v_dim // 32, ring_len, 32, **f32)
        self.ring_k = torch.zeros(num_slots, num_k_heads, ring_len, head_k_dim, device=dev,
                                  dtype=act_dtype)
        self.ring_g = torch.zeros(num_slots, num_v_heads, ring_len, **f32)
        self.slot_wp = torch.zeros(num_slots, device=dev, dtype=torch.int32)
        self.row_wp = torch.zeros(max_batch, device=dev, dtype=torch.int32)
        self.row_flush = torch.zeros(max_batch, device=dev, dtype=torch.uint8)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.ws_bytes = B.rssm_gdn_workspace_size(self.dims(max_batch))
        self.workspace = torch.empty(max(self.ws_bytes, 16), device=dev, dtype=torch.uint8)
        self.o = torch.empty(max_batch, num_v_heads, head_v_dim, device=dev, dtype=out_dtype)

    def dims(self, batch):
        return B.GDNDims(batch, self.HV, self.HK, self.K, self.V, self.L, self.num_slots,
                         torch_dtype_code(self.act_dtype), torch_dtype_code(self.out_dtype))

    def advance(self, cache_indices, force_flush=None, stream=None):
        b = cache_indices.shape[0]
        B.rssm_advance_cursors(B.RSSM_CURSOR_STANDARD, self.slot_wp, None, None, cache_indices,
                               force_flush, None, b, self.num_slots, self.L, 0, self.row_wp,
                               self.row_flush, self.dev_err, stream)

    def append(self, k, g, cache_indices, stream=None):
        B.rssm_gdn_ring_append(self.dims(k.shape[0]), k, g, cache_indices, self.row_wp,
                               self.ring_k, self.ring_g, self.dev_err, stream)

    def precompute(self, q, k, beta, g, cache_indices, stream=None):
        B.rssm_gdn_precompute(self.dims(q.shape[0]), q, k, beta, g, self.ring_k, self.ring_g,
                              cache_indices, self.row_wp, self.workspace, self.ws_bytes,
                              self.dev_err, stream)

    def output(self, q, v, cache_indices, o=None, stream=None):
        b = v.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_gdn_output(self.dims(b), self.state, q, v, self.ring_k, self.ring_d, cache_indices,
                          self.row_wp, self.row_flush, self.workspace, self.ws_bytes, o,
                          self.dev_err, stream)
        return o

    def prepare(self, q, k, beta, g, cache_indices, force_flush=None, stream=None, advance=True):
        """Cursor advance (unless advance=False), ring append and tables in one launch."""
        B.rssm_gdn_prepare(self.dims(q.shape[0]), advance, force_flush, self.slot_wp, self.row_wp,
                           self.row_flush, q, k, beta, g, cache_indices, self.ring_k, self.ring_g,
                           self.workspace, self.ws_bytes, self.dev_err, stream)

    def step(self, q, k, v, beta, g, cache_indices, force_flush=None, o=None, stream=None,
             advance=True):
        """One decode step as one rssm_gdn_step call (two launches). Returns o [b, HV, V]."""
        b = q.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_gdn_step(self.dims(b), advance, force_flush, self.slot_wp, self.row_wp,
                        self.row_flush, self.state, q, k, v, beta, g, cache_indices, self.ring_k,
                        self.ring_g, self.ring_d, self.workspace, self.ws_bytes, o, self.dev_err,
                        stream)
        return o

    def step_staged(self, q, k, v, beta, g, cache_indices, force_flush=None, o=None, stream=None,
                    advance=True):
        """The same step as four calls (cursor, append, precompute, output)."""
        if advance:
            self.advance(cache_indices, force_flush, stream)
        self.append(k, g, cache_indices, stream)
        self.precompute(q, k, beta, g, cache_indices, stream)
        return self.output(q, v, cache_indices, o, stream)

    def reset_slots(self, slots, stream=None):
        B.rssm_advance_cursors(B.RSSM_CURSOR_RESET, self.slot_wp, None, None, slots, None, None,
                               slots.shape[0], self.num_slots, self.L, 0, None, None, self.dev_err,
                               stream)

    def copy_slots(self, src, dst, stream=None):
        """Fork: slot dst[i] becomes a copy of slot src[i] (checkpoint, rings, cursor)."""
        B.rssm_copy_slots([self.state, self.ring_d, self.ring_k, self.ring_g, self.slot_wp],
                          src, dst, src.shape[0], self.num_slots, self.dev_err, stream)

    def materialize(self, slots, out=None, stream=None):
        """Current fp32 state of the listed slots [n, HV, V, K]."""
        n = slots.shape[0]
        if out is None:
            out = torch.empty(n, self.HV, self.V, self.K, device=self.state.device,
                              dtype=torch.float32)
        B.rssm_gdn_materialize_state(self.dims(n), self.state, self.ring_k, self.ring_g,
                                     self.ring_d, slots, self.slot_wp, None, out, self.dev_err,
                                     stream)
        return out


class GDNFullStateDecoder:
    """The conventional gated-delta-net decode step (state read and written every step)."""

    def __init__(self, num_v_heads, num_k_heads, head_k_dim, head_v_dim, num_slots, max_batch,
                 act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.HV, self.HK, self.K, self.V = num_v_heads, num_k_heads, head_k_dim, head_v_dim
        self.num_slots = num_slots
        self.act_dtype, self.out_dtype = act_dtype, out_dtype
        self.state = torch.zeros(num_slots, num_v_heads, head_v_dim, head_k_dim, device=dev,
                                 dtype=torch.float32)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.o = torch.empty(max_batch, num_v_heads, head_v_dim, device=dev, dtype=out_dtype)

    def dims(self, batch):
        return B.GDNDims(batch, self.HV, self.HK, self.K, self.V, 1, self.num_slots,
                         torch_dtype_code(self.act_dtype), torch_dtype_code(self.out_dtype))

    def step(self, q, k, v, beta, g, cache_indices, o=None, stream=None):
        b = q.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_gdn_full_state_decode(self.dims(b), self.state, q, k, v, beta, g, cache_indices, o,
                                     self.dev_err, stream)
        return o


class KDAReplayDecoder(GDNReplayDecoder):
    """ReplaySSM decode of the gated delta rule with a per-key-channel gate (KDA) for
    one layer. Buffers as GDNReplayDecoder, with the gate ring ring_a [num_slots, HV,
    L, K] float32 in place of ring_g. A step is rssm_kda_step (cursor advance,
    prepare, output: three launches)."""

    def __init__(self, num_v_heads, num_k_heads, head_k_dim, head_v_dim, ring_len, num_slots,
                 max_batch, act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None):
        super().__init__(num_v_heads, num_k_heads, head_k_dim, head_v_dim, ring_len, num_slots,
                         max_batch, act_dtype, out_dtype, device)
        dev = self.state.device
        self.ring_g = None
        self.ring_a = torch.zeros(num_slots, num_v_heads, ring_len, head_k_dim, device=dev,
                                  dtype=torch.float32)
        self.ws_bytes = B.rssm_kda_workspace_size(self.dims(max_batch))
        self.workspace = torch.empty(max(self.ws_bytes, 16), device=dev, dtype=torch.uint8)

    def prepare(self, q, k, a, beta, cache_indices, stream=None):
        """Ring append and tables (the cursors of the step must be set: advance())."""
        B.rssm_kda_prepare(self.dims(q.shape[0]), q, k, a, beta, cache_indices, self.row_wp,
                           self.row_flush, self.ring_k, self.ring_a, self.workspace,
                           self.ws_bytes, self.dev_err, stream)

    def output(self, v, cache_indices, o=None, stream=None):
        b = v.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_kda_output(self.dims(b), self.state, v, self.ring_d, cache_indices, self.row_wp,
                          self.row_flush, self.workspace, self.ws_bytes, o, self.dev_err, stream)
        return o

    def step(self, q, k, v, beta, a, cache_indices, force_flush=None, o=None, stream=None,
             advance=True):
        """One decode step (gate vectors a [b, HV, K]). Returns o [b, HV, V]."""
        b = q.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_kda_step(self.dims(b), advance, force_flush, self.slot_wp, self.row_wp,
                        self.row_flush, self.state, q, k, v, beta, a, cache_indices, self.ring_k,
                        self.ring_a, self.ring_d, self.workspace, self.ws_bytes, o, self.dev_err,
                        stream)
        return o

    def step_staged(self, q, k, v, beta, a, cache_indices, force_flush=None, o=None, stream=None,
                    advance=True):
        """The same step as three calls (cursor, prepare, output)."""
        if advance:
            self.advance(cache_indices, force_flush, stream)
        self.prepare(q, k, a, beta, cache_indices, stream)
        return self.output(v, cache_indices, o, stream)

    def copy_slots(self, src, dst, stream=None):
        B.rssm_copy_slots([self.state, self.ring_d, self.ring_k, self.ring_a, self.slot_wp],
                          src, dst, src.shape[0], self.num_slots, self.dev_err, stream)

    def append(self, *args, **kw):
        raise NotImplementedError("KDA appends inside prepare()")

    def precompute(self, *args, **kw):
        raise NotImplementedError("KDA builds its tables inside prepare()")

    def materialize(self, *args, **kw):
        raise NotImplementedError("no KDA materialize entry point")


class KDAFullStateDecoder(GDNFullStateDecoder):
    """The conventional KDA decode step (state read and written every step)."""

    def step(self, q, k, v, beta, a, cache_indices, o=None, stream=None):
        b = q.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_kda_full_state_decode(self.dims(b), self.state, q, k, v, beta, a, cache_indices, o,
                                     self.dev_err, stream)
        return o


class Mamba2SpecVerifier:
    """ReplaySSM speculative verify for Mamba2: T draft tokens per row and round on the
    circular ring (cursors cnt / base / flush per slot), then a commit of the accepted
    prefix that only moves cursors. Buffers as Mamba2ReplayDecoder plus slot_base and
    slot_flush; y [max_batch, T, H, P]."""

    def __init__(self, nheads, headdim, dstate, ngroups, ring_len, T, num_slots, max_batch, A, D,
                 dt_bias=None, dt_softplus=True, state_dtype=torch.bfloat16,
                 act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.H, self.P, self.N, self.G, self.L, self.T = (nheads, headdim, dstate, ngroups,
                                                          ring_len, T)
        self.num_slots, self.max_batch = num_slots, max_batch
        self.state_dtype, self.act_dtype, self.out_dtype = state_dtype, act_dtype, out_dtype
        self.dt_softplus = dt_softplus
        f32 = dict(device=dev, dtype=torch.float32)
        self.A = torch.as_tensor(A, **f32).contiguous()
        self.D = torch.as_tensor(D, **f32).contiguous()
        self.dt_bias = None if dt_bias is None else torch.as_tensor(dt_bias, **f32).contiguous()
        self.state = torch.zeros(num_slots, nheads, headdim, dstate, device=dev, dtype=state_dtype)
        self.ring_x = torch.zeros(num_slots, nheads, ring_len, headdim, device=dev, dtype=act_dtype)
        self.ring_dt = torch.zeros(num_slots, nheads, ring_len, **f32)
        self.ring_B = torch.zeros(num_slots, ngroups, ring_len, dstate, device=dev, dtype=act_dtype)
        self.slot_cnt = torch.zeros(num_slots, device=dev, dtype=torch.int32)
        self.slot_base = torch.zeros(num_slots, device=dev, dtype=torch.int32)
        self.slot_flush = torch.zeros(num_slots, device=dev, dtype=torch.uint8)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.ws_bytes = B.rssm_mamba2_spec_workspace_size(self.dims(max_batch), T)
        self.workspace = torch.empty(max(self.ws_bytes, 16), device=dev, dtype=torch.uint8)
        self.y = torch.empty(max_batch, T, nheads, headdim, device=dev, dtype=out_dtype)

    def dims(self, batch):
        return B.Mamba2Dims(batch, self.H, self.P, self.N, self.G, self.L, self.num_slots,
                            torch_dtype_code(self.state_dtype), torch_dtype_code(self.act_dtype),
                            torch_dtype_code(self.out_dtype))

    def verify(self, x, dt_raw, Bm, C, z, cache_indices, y=None, stream=None):
        """Per-draft outputs y [b, T, H, P] for draft inputs [b, T, ...]."""
        b = x.shape[0]
        y = self.y[:b] if y is None else y
        B.rssm_mamba2_spec_verify(self.dims(b), self.T, self.state, x, dt_raw, self.dt_bias,
                                  self.dt_softplus, self.A, Bm, C, self.D, z, self.ring_x,
                                  self.ring_dt, self.ring_B, cache_indices, self.slot_cnt,
                                  self.slot_base, self.slot_flush, self.workspace, self.ws_bytes,
                                  y, self.dev_err, stream)
        return y

    def commit(self, cache_indices, num_accepted, stream=None):
        B.rssm_advance_cursors(B.RSSM_CURSOR_SPEC_COMMIT, self.slot_cnt, self.slot_base,
                               self.slot_flush, cache_indices, None, num_accepted,
                               cache_indices.shape[0], self.num_slots, self.L, self.T, None, None,
                               self.dev_err, stream)

    def reset_slots(self, slots, stream=None):
        B.rssm_advance_cursors(B.RSSM_CURSOR_RESET, self.slot_cnt, self.slot_base,
                               self.slot_flush, slots, None, None, slots.shape[0], self.num_slots,
                               self.L, self.T, None, None, self.dev_err, stream)

    def copy_slots(self, src, dst, stream=None):
        B.rssm_copy_slots([self.state, self.ring_x, self.ring_dt, self.ring_B, self.slot_cnt,
                           self.slot_base, self.slot_flush], src, dst, src.shape[0],
                          self.num_slots, self.dev_err, stream)


class GDNSpecVerifier:
    """ReplaySSM speculative verify for the gated delta net (linear draft chain of T).

    Buffers: state [num_slots, HV, V, K] float32; rings d [.., HV, V/32, L, 32] f32,
    k [.., HK, L, K], g [.., HV, L] f32, raw v [.., HV, L, V], beta [.., HV, L] f32;
    per-slot cursors cnt (slot_wp), base, flush."""

    def __init__(self, num_v_heads, num_k_heads, head_k_dim, head_v_dim, ring_len, T, num_slots,
                 max_batch, act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.HV, self.HK, self.K, self.V, self.L, self.T = (num_v_heads, num_k_heads, head_k_dim,
                                                           head_v_dim, ring_len, T)
        self.num_slots = num_slots
        self.act_dtype, self.out_dtype = act_dtype, out_dtype
        f32 = dict(device=dev, dtype=torch.float32)
        self.state = torch.zeros(num_slots, num_v_heads, head_v_dim, head_k_dim, **f32)
        self.ring_d = torch.zeros(num_slots, num_v_heads, head_v_dim // 32, ring_len, 32, **f32)
        self.ring_k = torch.zeros(num_slots, num_k_heads, ring_len, head_k_dim, device=dev,
                                  dtype=act_dtype)
        self.ring_g = torch.zeros(num_slots, num_v_heads, ring_len, **f32)
        self.ring_v = torch.zeros(num_slots, num_v_heads, ring_len, head_v_dim, device=dev,
                                  dtype=act_dtype)
        self.ring_beta = torch.zeros(num_slots, num_v_heads, ring_len, **f32)
        self.slot_cnt = torch.zeros(num_slots, device=dev, dtype=torch.int32)
        self.slot_base = torch.zeros(num_slots, device=dev, dtype=torch.int32)
        self.slot_flush = torch.zeros(num_slots, device=dev, dtype=torch.uint8)
        self.row_cnt = torch.zeros(max_batch, device=dev, dtype=torch.int32)
        self.row_flush = torch.zeros(max_batch, device=dev, dtype=torch.uint8)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.o = torch.empty(max_batch, T, num_v_heads, head_v_dim, device=dev, dtype=out_dtype)
        self.ws_bytes = B.rssm_gdn_spec_workspace_size(self.dims(max_batch), T)
        self.workspace = torch.empty(max(self.ws_bytes, 16), device=dev, dtype=torch.uint8)

    def dims(self, batch):
        return B.GDNDims(batch, self.HV, self.HK, self.K, self.V, self.L, self.num_slots,
                         torch_dtype_code(self.act_dtype), torch_dtype_code(self.out_dtype))

    def verify(self, q, k, v, beta, g, cache_indices, o=None, stream=None):
        """Per-draft outputs o [b, T, HV, V] for draft inputs [b, T, ...]."""
        b = q.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_gdn_spec_verify(self.dims(b), self.T, self.state, q, k, v, beta, g, self.ring_d,
                               self.ring_k, self.ring_g, self.ring_v, self.ring_beta,
                               cache_indices, self.slot_cnt, self.slot_base, self.slot_flush,
                               self.workspace, self.ws_bytes, o, self.dev_err, stream)
        return o

    def commit(self, cache_indices, num_accepted, stream=None):
        b = cache_indices.shape[0]
        B.rssm_advance_cursors(B.RSSM_CURSOR_SPEC_COMMIT, self.slot_cnt, self.slot_base,
                               self.slot_flush, cache_indices, None, num_accepted, b,
                               self.num_slots, self.L, self.T, self.row_cnt[:b], self.row_flush[:b],
                               self.dev_err, stream)

    def reset_slots(self, slots, stream=None):
        B.rssm_advance_cursors(B.RSSM_CURSOR_RESET, self.slot_cnt, self.slot_base,
                               self.slot_flush, slots, None, None, slots.shape[0], self.num_slots,
                               self.L, self.T, None, None, self.dev_err, stream)

    def copy_slots(self, src, dst, stream=None):
        """Fork: slot dst[i] becomes a copy of slot src[i] (checkpoint, the five rings
        and the three cursors, a pending fold included)."""
        B.rssm_copy_slots([self.state, self.ring_d, self.ring_k, self.ring_g, self.ring_v,
                           self.ring_beta, self.slot_cnt, self.slot_base, self.slot_flush],
                          src, dst, src.shape[0], self.num_slots, self.dev_err, stream)

    def materialize(self, slots, out=None, stream=None):
        """Current fp32 state of the listed slots [n, HV, V, K]: the checkpoint folded with
        the committed entries (including those of a pending fold)."""
        n = slots.shape[0]
        if out is None:
            out = torch.empty(n, self.HV, self.V, self.K, device=self.state.device,
                              dtype=torch.float32)
        B.rssm_gdn_materialize_state(self.dims(n), self.state, self.ring_k, self.ring_g,
                                     self.ring_d, slots, self.slot_cnt, self.slot_base, out,
                                     self.dev_err, stream)
        return out


class GDNSpecFullStateVerifier:
    """The conventional speculative verify (in-house comparison): every draft's full
    state is stored as a snapshot [max_batch, T, HV, V, K] float32; the commit copies the
    accepted draft's snapshot into the slot."""

    def __init__(self, num_v_heads, num_k_heads, head_k_dim, head_v_dim, T, num_slots, max_batch,
                 act_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.HV, self.HK, self.K, self.V, self.T = (num_v_heads, num_k_heads, head_k_dim,
                                                    head_v_dim, T)
        self.num_slots = num_slots
        self.act_dtype, self.out_dtype = act_dtype, out_dtype
        self.state = torch.zeros(num_slots, num_v_heads, head_v_dim, head_k_dim, device=dev,
                                 dtype=torch.float32)
        self.snap_bytes = B.rssm_gdn_spec_full_state_snapshot_bytes(self.dims(max_batch), T)
        self.snapshots = torch.empty(max_batch, T, num_v_heads, head_v_dim, head_k_dim,
                                     device=dev, dtype=torch.float32)
        self.dev_err = torch.zeros(4, device=dev, dtype=torch.int32)
        self.o = torch.empty(max_batch, T, num_v_heads, head_v_dim, device=dev, dtype=out_dtype)

    def dims(self, batch):
        return B.GDNDims(batch, self.HV, self.HK, self.K, self.V, 1, self.num_slots,
                         torch_dtype_code(self.act_dtype), torch_dtype_code(self.out_dtype))

    def verify(self, q, k, v, beta, g, cache_indices, o=None, stream=None):
        b = q.shape[0]
        o = self.o[:b] if o is None else o
        B.rssm_gdn_spec_full_state_verify(self.dims(b), self.T, self.state, q, k, v, beta, g,
                                          cache_indices, self.snapshots, self.snap_bytes, o,
                                          self.dev_err, stream)
        return o

    def commit(self, cache_indices, num_accepted, stream=None):
        B.rssm_gdn_spec_full_state_commit(self.dims(cache_indices.shape[0]), self.T, self.state,
                                          self.snapshots, cache_indices, num_accepted,
                                          self.dev_err, stream)
