"""ctypes binding over librssm.so: one Python function per C-ABI entry point,
same names, argument marshalling only (tensors -> device pointers, None -> NULL,
the current torch stream when none is given). Every computation happens in the
library's CUDA kernels; there is no fallback path. A non-zero status raises
RSSMError.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librssm.so")

RSSM_OK, RSSM_ERR_INVALID_ARG, RSSM_ERR_UNSUPPORTED, RSSM_ERR_CONFIG, RSSM_ERR_CUDA = range(5)
RSSM_F32, RSSM_BF16 = 0, 1
RSSM_DEVERR_SLOT, RSSM_DEVERR_CURSOR, RSSM_DEVERR_TIMEOUT = 1, 2, 4
RSSM_CURSOR_STANDARD, RSSM_CURSOR_SPEC_COMMIT, RSSM_CURSOR_RESET = 0, 1, 2
RSSM_NOALLOC_WORKSPACE_BYTES = 16 << 20
RSSM_MAX_SLOT_BUFFERS = 12

# every symbol include/rssm.h declares
EXPORTS = (
    "rssm_status_string", "rssm_abi_version", "rssm_advance_cursors", "rssm_copy_slots",
    "rssm_ring_append",
    "rssm_mamba2_workspace_size", "rssm_mamba2_precompute", "rssm_mamba2_output",
    "rssm_mamba2_decode", "rssm_mamba2_decode_noalloc", "rssm_mamba2_prepare", "rssm_mamba2_step",
    "rssm_mamba2_full_state_update", "rssm_mamba2_output_sr", "rssm_mamba2_step_sr",
    "rssm_mamba2_full_state_update_sr", "rssm_philox4x32_fill", "rssm_mamba2_spec_workspace_size",
    "rssm_mamba2_spec_verify",
    "rssm_gdn_ring_append",
    "rssm_gdn_workspace_size", "rssm_gdn_precompute", "rssm_gdn_output", "rssm_gdn_decode",
    "rssm_gdn_prepare", "rssm_gdn_step",
    "rssm_gdn_full_state_decode", "rssm_gdn_spec_workspace_size", "rssm_gdn_spec_verify",
    "rssm_mamba2_materialize_state", "rssm_gdn_materialize_state",
    "rssm_gdn_spec_full_state_snapshot_bytes", "rssm_gdn_spec_full_state_verify",
    "rssm_gdn_spec_full_state_commit", "rssm_kda_workspace_size", "rssm_kda_prepare",
    "rssm_kda_output", "rssm_kda_step", "rssm_kda_full_state_decode",
    "rssm_debug_pipeline_copy", "rssm_debug_umma_fold",
)


class RSSMError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = _lib.rssm_status_string(status).decode() if _lib else str(status)
        super().__init__("%s failed: %s (status %d)" % (fn, msg, status))


class SlotBuffer(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("slot_bytes", ctypes.c_size_t)]


class Mamba2Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "nheads", "headdim", "dstate", "ngroups", "ring_len", "num_slots",
        "state_dtype", "act_dtype", "out_dtype")]


class GDNDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_v_heads", "num_k_heads", "head_k_dim", "head_v_dim", "ring_len",
        "num_slots", "act_dtype", "out_dtype")]


_lib = None
_VP = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t


def _declare(L):
    m2 = ctypes.POINTER(Mamba2Dims)
    gd = ctypes.POINTER(GDNDims)
    sig = {
        "rssm_status_string": (ctypes.c_char_p, [_I]),
        "rssm_abi_version": (_I, []),
        "rssm_advance_cursors": (_I, [_I, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32,
                                      _VP, _VP, _VP, _VP]),
        "rssm_copy_slots": (_I, [ctypes.POINTER(SlotBuffer), _I32, _VP, _VP, _I32, _I32, _VP, _VP]),
        "rssm_ring_append": (_I, [m2, _VP, _VP, _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
        "rssm_mamba2_workspace_size": (_SZ, [m2]),
        "rssm_mamba2_precompute": (_I, [m2, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
        "rssm_mamba2_output": (_I, [m2, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                                    _VP, _VP, _VP]),
        "rssm_mamba2_decode": (_I, [m2, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                    _VP, _SZ, _VP, _VP, _VP]),
        "rssm_mamba2_decode_noalloc": (_I, [m2, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            _VP, _VP, _VP, _VP]),
        "rssm_mamba2_prepare": (_I, [m2, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP,
                                     _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
        "rssm_mamba2_step": (_I, [m2, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP, _VP,
                                  _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP, _VP]),
        "rssm_mamba2_full_state_update": (_I, [m2, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP, _VP,
                                               _VP, _VP, _VP, _VP, _VP]),
        "rssm_mamba2_output_sr": (_I, [m2, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                       _SZ, _VP, _VP, _VP, _VP]),
        "rssm_mamba2_step_sr": (_I, [m2, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP, _VP,
                                     _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP, _VP,
                                     _VP]),
        "rssm_mamba2_full_state_update_sr": (_I, [m2, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP,
                                                  _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
        "rssm_philox4x32_fill": (_I, [ctypes.c_uint64, ctypes.c_uint64, _VP, _SZ, _VP]),
        "rssm_mamba2_spec_workspace_size": (_SZ, [m2, _I32]),
        "rssm_mamba2_spec_verify": (_I, [m2, _I32, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP, _VP, _VP,
                                         _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP,
                                         _VP]),
        "rssm_gdn_ring_append": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
        "rssm_gdn_workspace_size": (_SZ, [gd]),
        "rssm_gdn_precompute": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP,
                                     _VP]),
        "rssm_gdn_output": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP,
                                 _VP]),
        "rssm_gdn_decode": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                 _VP, _SZ, _VP, _VP, _VP]),
        "rssm_gdn_prepare": (_I, [gd, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                  _VP, _SZ, _VP, _VP]),
        "rssm_gdn_step": (_I, [gd, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                               _VP, _VP, _VP, _VP, _SZ, _VP, _VP, _VP]),
        "rssm_gdn_full_state_decode": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            _VP]),
        "rssm_gdn_spec_workspace_size": (_SZ, [gd, _I32]),
        "rssm_gdn_spec_full_state_snapshot_bytes": (_SZ, [gd, _I32]),
        "rssm_gdn_spec_full_state_verify": (_I, [gd, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                 _SZ, _VP, _VP, _VP]),
        "rssm_gdn_spec_full_state_commit": (_I, [gd, _I32, _VP, _VP, _VP, _VP, _VP, _VP]),
        "rssm_mamba2_materialize_state": (_I, [m2, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                               _VP]),
        "rssm_gdn_materialize_state": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            _VP]),
        "rssm_kda_workspace_size": (_SZ, [gd]),
        "rssm_kda_prepare": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP,
                                  _VP]),
        "rssm_kda_output": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP, _VP]),
        "rssm_kda_step": (_I, [gd, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                               _VP, _VP, _VP, _VP, _SZ, _VP, _VP, _VP]),
        "rssm_kda_full_state_decode": (_I, [gd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            _VP]),
        "rssm_gdn_spec_verify": (_I, [gd, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                      _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP, _VP]),
        "rssm_debug_pipeline_copy": (_I, [_VP, _VP, _I, _I, _I, _VP, _VP]),
        "rssm_debug_umma_fold": (_I, [_VP, _VP, _I, _I, _VP, _VP, _VP]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def lib():
    """The loaded librssm.so. Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("librssm.so is not built (run ssm_linear_attention_gb300/build.py "
                              "or __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != RSSM_OK:
        raise RSSMError(name, rc)


def rssm_status_string(status):
    return lib().rssm_status_string(status).decode()


def rssm_abi_version():
    return lib().rssm_abi_version()


def rssm_advance_cursors(mode, slot_wp, slot_base, slot_flush, cache_indices, force_flush,
                         num_accepted, batch, num_slots, L, T, row_wp, row_flush, dev_err=None,
                         stream=None):
    _call("rssm_advance_cursors", mode, _ptr(slot_wp), _ptr(slot_base), _ptr(slot_flush),
          _ptr(cache_indices), _ptr(force_flush), _ptr(num_accepted), batch, num_slots, L, T,
          _ptr(row_wp), _ptr(row_flush), _ptr(dev_err), _stream(stream))


def rssm_copy_slots(buffers, src_slots, dst_slots, n, num_slots, dev_err=None, stream=None):
    """buffers: per-slot buffers, each a slot-major tensor (its first dimension is
    the slot; slot_bytes = bytes of one slot) or a (pointer or tensor, slot_bytes)
    pair."""
    descs = []
    for b in buffers:
        if isinstance(b, tuple):
            ptr, sb = b
        else:
            ptr, sb = b, b[0].numel() * b.element_size()
        descs.append(SlotBuffer(_ptr(ptr), int(sb)))
    arr = (SlotBuffer * max(len(descs), 1))(*descs)
    _call("rssm_copy_slots", arr if descs else None, len(descs), _ptr(src_slots),
          _ptr(dst_slots), int(n), int(num_slots), _ptr(dev_err), _stream(stream))


def rssm_ring_append(dims, x, dt_raw, dt_bias, dt_softplus, B, cache_indices, row_wp, ring_x,
                     ring_dt, ring_B, dev_err=None, stream=None):
    _call("rssm_ring_append", ctypes.byref(dims), _ptr(x), _ptr(dt_raw), _ptr(dt_bias),
          int(dt_softplus), _ptr(B), _ptr(cache_indices), _ptr(row_wp), _ptr(ring_x),
          _ptr(ring_dt), _ptr(ring_B), _ptr(dev_err), _stream(stream))


def rssm_mamba2_workspace_size(dims):
    return lib().rssm_mamba2_workspace_size(ctypes.byref(dims))


def rssm_mamba2_precompute(dims, A, C, ring_dt, ring_B, cache_indices, row_wp, workspace,
                           workspace_bytes, dev_err=None, stream=None):
    _call("rssm_mamba2_precompute", ctypes.byref(dims), _ptr(A), _ptr(C), _ptr(ring_dt),
          _ptr(ring_B), _ptr(cache_indices), _ptr(row_wp), _ptr(workspace), workspace_bytes,
          _ptr(dev_err), _stream(stream))


def rssm_mamba2_output(dims, state, C, D, z, ring_x, ring_B, cache_indices, row_wp, row_flush,
                       workspace, workspace_bytes, y, dev_err=None, stream=None):
    _call("rssm_mamba2_output", ctypes.byref(dims), _ptr(state), _ptr(C), _ptr(D), _ptr(z),
          _ptr(ring_x), _ptr(ring_B), _ptr(cache_indices), _ptr(row_wp), _ptr(row_flush),
          _ptr(workspace), workspace_bytes, _ptr(y), _ptr(dev_err), _stream(stream))


def rssm_mamba2_decode(dims, state, A, C, D, z, ring_x, ring_dt, ring_B, cache_indices, row_wp,
                       row_flush, workspace, workspace_bytes, y, dev_err=None, stream=None):
    _call("rssm_mamba2_decode", ctypes.byref(dims), _ptr(state), _ptr(A), _ptr(C), _ptr(D),
          _ptr(z), _ptr(ring_x), _ptr(ring_dt), _ptr(ring_B), _ptr(cache_indices), _ptr(row_wp),
          _ptr(row_flush), _ptr(workspace), workspace_bytes, _ptr(y), _ptr(dev_err),
          _stream(stream))


def rssm_mamba2_decode_noalloc(dims, state, A, C, D, z, ring_x, ring_dt, ring_B, cache_indices,
                               row_wp, row_flush, y, dev_err=None, stream=None):
    """rssm_mamba2_decode without a workspace argument, for callers that cannot
    allocate device memory: the tables live in the library's fixed device array
    (RSSM_NOALLOC_WORKSPACE_BYTES). Calls that overlap on the GPU share that array."""
    _call("rssm_mamba2_decode_noalloc", ctypes.byref(dims), _ptr(state), _ptr(A), _ptr(C), _ptr(D),
          _ptr(z), _ptr(ring_x), _ptr(ring_dt), _ptr(ring_B), _ptr(cache_indices), _ptr(row_wp),
          _ptr(row_flush), _ptr(y), _ptr(dev_err), _stream(stream))


def rssm_mamba2_prepare(dims, advance, force_flush, slot_wp, row_wp, row_flush, x, dt_raw,
                        dt_bias, dt_softplus, B, A, C, cache_indices, ring_x, ring_dt, ring_B,
                        workspace, workspace_bytes, dev_err=None, stream=None):
    _call("rssm_mamba2_prepare", ctypes.byref(dims), int(advance), _ptr(force_flush),
          _ptr(slot_wp), _ptr(row_wp), _ptr(row_flush), _ptr(x), _ptr(dt_raw), _ptr(dt_bias),
          int(dt_softplus), _ptr(B), _ptr(A), _ptr(C), _ptr(cache_indices), _ptr(ring_x),
          _ptr(ring_dt), _ptr(ring_B), _ptr(workspace), workspace_bytes, _ptr(dev_err),
          _stream(stream))


def rssm_mamba2_step(dims, advance, force_flush, slot_wp, row_wp, row_flush, state, x, dt_raw,
                     dt_bias, dt_softplus, A, B, C, D, z, cache_indices, ring_x, ring_dt, ring_B,
                     workspace, workspace_bytes, y, dev_err=None, stream=None):
    _call("rssm_mamba2_step", ctypes.byref(dims), int(advance), _ptr(force_flush), _ptr(slot_wp),
          _ptr(row_wp), _ptr(row_flush), _ptr(state), _ptr(x), _ptr(dt_raw), _ptr(dt_bias),
          int(dt_softplus), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(cache_indices),
          _ptr(ring_x), _ptr(ring_dt), _ptr(ring_B), _ptr(workspace), workspace_bytes, _ptr(y),
          _ptr(dev_err), _stream(stream))


def rssm_mamba2_full_state_update(dims, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z,
                                  cache_indices, y, dev_err=None, stream=None):
    _call("rssm_mamba2_full_state_update", ctypes.byref(dims), _ptr(state), _ptr(x),
          _ptr(dt_raw), _ptr(dt_bias), int(dt_softplus), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
          _ptr(z), _ptr(cache_indices), _ptr(y), _ptr(dev_err), _stream(stream))


def rssm_mamba2_output_sr(dims, state, C, D, z, ring_x, ring_B, cache_indices, row_wp, row_flush,
                          workspace, workspace_bytes, y, sr_state, dev_err=None, stream=None):
    """rssm_mamba2_output with stochastic rounding of the bf16 flush stores; sr_state
    is a device uint64 pair {seed, offset} whose offset the call advances."""
    _call("rssm_mamba2_output_sr", ctypes.byref(dims), _ptr(state), _ptr(C), _ptr(D), _ptr(z),
          _ptr(ring_x), _ptr(ring_B), _ptr(cache_indices), _ptr(row_wp), _ptr(row_flush),
          _ptr(workspace), workspace_bytes, _ptr(y), _ptr(sr_state), _ptr(dev_err),
          _stream(stream))


def rssm_mamba2_step_sr(dims, advance, force_flush, slot_wp, row_wp, row_flush, state, x, dt_raw,
                        dt_bias, dt_softplus, A, B, C, D, z, cache_indices, ring_x, ring_dt,
                        ring_B, workspace, workspace_bytes, y, sr_state, dev_err=None,
                        stream=None):
    """rssm_mamba2_step with stochastic rounding of the bf16 flush stores."""
    _call("rssm_mamba2_step_sr", ctypes.byref(dims), int(advance), _ptr(force_flush),
          _ptr(slot_wp), _ptr(row_wp), _ptr(row_flush), _ptr(state), _ptr(x), _ptr(dt_raw),
          _ptr(dt_bias), int(dt_softplus), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
          _ptr(cache_indices), _ptr(ring_x), _ptr(ring_dt), _ptr(ring_B), _ptr(workspace),
          workspace_bytes, _ptr(y), _ptr(sr_state), _ptr(dev_err), _stream(stream))


def rssm_mamba2_full_state_update_sr(dims, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z,
                                     cache_indices, y, sr_state, dev_err=None, stream=None):
    """rssm_mamba2_full_state_update with stochastic rounding of the bf16 state store."""
    _call("rssm_mamba2_full_state_update_sr", ctypes.byref(dims), _ptr(state), _ptr(x),
          _ptr(dt_raw), _ptr(dt_bias), int(dt_softplus), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
          _ptr(z), _ptr(cache_indices), _ptr(y), _ptr(sr_state), _ptr(dev_err), _stream(stream))


def rssm_philox4x32_fill(seed, offset, out, n_groups, stream=None):
    """out (device uint32/int32 [4 n_groups]) = the Philox4x32-10 blocks the stochastic
    rounding of groups 0..n_groups-1 draws at (seed, offset)."""
    _call("rssm_philox4x32_fill", int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1),
          _ptr(out), int(n_groups), _stream(stream))


def rssm_debug_pipeline_copy(src, dst, n_tiles, stall_tile, wait_us, dev_err=None, stream=None):
    """Copy n_tiles 16 KB tiles src -> dst through the streaming pipeline; stall_tile >= 0
    makes that tile's stage wait run out after wait_us (test of the bounded waits)."""
    _call("rssm_debug_pipeline_copy", _ptr(src), _ptr(dst), int(n_tiles), int(stall_tile),
          int(wait_us), _ptr(dev_err), _stream(stream))


def rssm_debug_umma_fold(A, B, w, N, D, dev_err=None, stream=None):
    """D [128][N] = A[:, :w+1] @ B[:w+1] on the tensor cores (A float32 [128][16], B bf16
    [16][N]); test of the fold building block."""
    _call("rssm_debug_umma_fold", _ptr(A), _ptr(B), int(w), int(N), _ptr(D), _ptr(dev_err),
          _stream(stream))


def rssm_gdn_ring_append(dims, k, g, cache_indices, row_wp, ring_k, ring_g, dev_err=None,
                         stream=None):
    _call("rssm_gdn_ring_append", ctypes.byref(dims), _ptr(k), _ptr(g), _ptr(cache_indices),
          _ptr(row_wp), _ptr(ring_k), _ptr(ring_g), _ptr(dev_err), _stream(stream))


def rssm_gdn_workspace_size(dims):
    return lib().rssm_gdn_workspace_size(ctypes.byref(dims))


def rssm_gdn_precompute(dims, q, k, beta, g, ring_k, ring_g, cache_indices, row_wp, workspace,
                        workspace_bytes, dev_err=None, stream=None):
    _call("rssm_gdn_precompute", ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(beta), _ptr(g),
          _ptr(ring_k), _ptr(ring_g), _ptr(cache_indices), _ptr(row_wp), _ptr(workspace),
          workspace_bytes, _ptr(dev_err), _stream(stream))


def rssm_gdn_output(dims, state, q, v, ring_k, ring_d, cache_indices, row_wp, row_flush,
                    workspace, workspace_bytes, o, dev_err=None, stream=None):
    _call("rssm_gdn_output", ctypes.byref(dims), _ptr(state), _ptr(q), _ptr(v), _ptr(ring_k),
          _ptr(ring_d), _ptr(cache_indices), _ptr(row_wp), _ptr(row_flush), _ptr(workspace),
          workspace_bytes, _ptr(o), _ptr(dev_err), _stream(stream))


def rssm_gdn_decode(dims, state, q, k, v, beta, g, ring_k, ring_g, ring_d, cache_indices, row_wp,
                    row_flush, workspace, workspace_bytes, o, dev_err=None, stream=None):
    _call("rssm_gdn_decode", ctypes.byref(dims), _ptr(state), _ptr(q), _ptr(k), _ptr(v),
          _ptr(beta), _ptr(g), _ptr(ring_k), _ptr(ring_g), _ptr(ring_d), _ptr(cache_indices),
          _ptr(row_wp), _ptr(row_flush), _ptr(workspace), workspace_bytes, _ptr(o),
          _ptr(dev_err), _stream(stream))


def rssm_gdn_prepare(dims, advance, force_flush, slot_wp, row_wp, row_flush, q, k, beta, g,
                     cache_indices, ring_k, ring_g, workspace, workspace_bytes, dev_err=None,
                     stream=None):
    _call("rssm_gdn_prepare", ctypes.byref(dims), int(advance), _ptr(force_flush), _ptr(slot_wp),
          _ptr(row_wp), _ptr(row_flush), _ptr(q), _ptr(k), _ptr(beta), _ptr(g),
          _ptr(cache_indices), _ptr(ring_k), _ptr(ring_g), _ptr(workspace), workspace_bytes,
          _ptr(dev_err), _stream(stream))


def rssm_gdn_step(dims, advance, force_flush, slot_wp, row_wp, row_flush, state, q, k, v, beta, g,
                  cache_indices, ring_k, ring_g, ring_d, workspace, workspace_bytes, o,
                  dev_err=None, stream=None):
    _call("rssm_gdn_step", ctypes.byref(dims), int(advance), _ptr(force_flush), _ptr(slot_wp),
          _ptr(row_wp), _ptr(row_flush), _ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
          _ptr(g), _ptr(cache_indices), _ptr(ring_k), _ptr(ring_g), _ptr(ring_d), _ptr(workspace),
          workspace_bytes, _ptr(o), _ptr(dev_err), _stream(stream))


def rssm_gdn_full_state_decode(dims, state, q, k, v, beta, g, cache_indices, o, dev_err=None,
                               stream=None):
    _call("rssm_gdn_full_state_decode", ctypes.byref(dims), _ptr(state), _ptr(q), _ptr(k),
          _ptr(v), _ptr(beta), _ptr(g), _ptr(cache_indices), _ptr(o), _ptr(dev_err),
          _stream(stream))


def rssm_gdn_spec_workspace_size(dims, T):
    return lib().rssm_gdn_spec_workspace_size(ctypes.byref(dims), T)


def rssm_gdn_spec_verify(dims, T, state, q, k, v, beta, g, ring_d, ring_k, ring_g, ring_v,
                         ring_beta, cache_indices, slot_wp, slot_base, slot_flush, workspace,
                         workspace_bytes, o, dev_err=None, stream=None):
    _call("rssm_gdn_spec_verify", ctypes.byref(dims), T, _ptr(state), _ptr(q), _ptr(k), _ptr(v),
          _ptr(beta), _ptr(g), _ptr(ring_d), _ptr(ring_k), _ptr(ring_g), _ptr(ring_v),
          _ptr(ring_beta), _ptr(cache_indices), _ptr(slot_wp), _ptr(slot_base), _ptr(slot_flush),
          _ptr(workspace), workspace_bytes, _ptr(o), _ptr(dev_err), _stream(stream))


def rssm_mamba2_materialize_state(dims, state, A, ring_x, ring_dt, ring_B, slots, slot_wp, out,
                                  dev_err=None, stream=None):
    _call("rssm_mamba2_materialize_state", ctypes.byref(dims), _ptr(state), _ptr(A), _ptr(ring_x),
          _ptr(ring_dt), _ptr(ring_B), _ptr(slots), _ptr(slot_wp), _ptr(out), _ptr(dev_err),
          _stream(stream))


def rssm_gdn_materialize_state(dims, state, ring_k, ring_g, ring_d, slots, slot_wp, slot_base,
                               out, dev_err=None, stream=None):
    _call("rssm_gdn_materialize_state", ctypes.byref(dims), _ptr(state), _ptr(ring_k),
          _ptr(ring_g), _ptr(ring_d), _ptr(slots), _ptr(slot_wp), _ptr(slot_base), _ptr(out),
          _ptr(dev_err), _stream(stream))


def rssm_gdn_spec_full_state_snapshot_bytes(dims, T):
    return lib().rssm_gdn_spec_full_state_snapshot_bytes(ctypes.byref(dims), T)


def rssm_gdn_spec_full_state_verify(dims, T, state, q, k, v, beta, g, cache_indices, snapshots,
                                    snapshot_bytes, o, dev_err=None, stream=None):
    _call("rssm_gdn_spec_full_state_verify", ctypes.byref(dims), T, _ptr(state), _ptr(q), _ptr(k),
          _ptr(v), _ptr(beta), _ptr(g), _ptr(cache_indices), _ptr(snapshots), snapshot_bytes,
          _ptr(o), _ptr(dev_err), _stream(stream))


def rssm_gdn_spec_full_state_commit(dims, T, state, snapshots, cache_indices, num_accepted,
                                    dev_err=None, stream=None):
    _call("rssm_gdn_spec_full_state_commit", ctypes.byref(dims), T, _ptr(state), _ptr(snapshots),
          _ptr(cache_indices), _ptr(num_accepted), _ptr(dev_err), _stream(stream))


def rssm_kda_workspace_size(dims):
    return lib().rssm_kda_workspace_size(ctypes.byref(dims))


def rssm_kda_prepare(dims, q, k, a, beta, cache_indices, row_wp, row_flush, ring_k, ring_a,
                     workspace, workspace_bytes, dev_err=None, stream=None):
    _call("rssm_kda_prepare", ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(a), _ptr(beta),
          _ptr(cache_indices), _ptr(row_wp), _ptr(row_flush), _ptr(ring_k), _ptr(ring_a),
          _ptr(workspace), workspace_bytes, _ptr(dev_err), _stream(stream))


def rssm_kda_output(dims, state, v, ring_d, cache_indices, row_wp, row_flush, workspace,
                    workspace_bytes, o, dev_err=None, stream=None):
    _call("rssm_kda_output", ctypes.byref(dims), _ptr(state), _ptr(v), _ptr(ring_d),
          _ptr(cache_indices), _ptr(row_wp), _ptr(row_flush), _ptr(workspace), workspace_bytes,
          _ptr(o), _ptr(dev_err), _stream(stream))


def rssm_kda_step(dims, advance, force_flush, slot_wp, row_wp, row_flush, state, q, k, v, beta, a,
                  cache_indices, ring_k, ring_a, ring_d, workspace, workspace_bytes, o,
                  dev_err=None, stream=None):
    _call("rssm_kda_step", ctypes.byref(dims), int(advance), _ptr(force_flush), _ptr(slot_wp),
          _ptr(row_wp), _ptr(row_flush), _ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
          _ptr(a), _ptr(cache_indices), _ptr(ring_k), _ptr(ring_a), _ptr(ring_d), _ptr(workspace),
          workspace_bytes, _ptr(o), _ptr(dev_err), _stream(stream))


def rssm_kda_full_state_decode(dims, state, q, k, v, beta, a, cache_indices, o, dev_err=None,
                               stream=None):
    _call("rssm_kda_full_state_decode", ctypes.byref(dims), _ptr(state), _ptr(q), _ptr(k),
          _ptr(v), _ptr(beta), _ptr(a), _ptr(cache_indices), _ptr(o), _ptr(dev_err),
          _stream(stream))


def rssm_mamba2_spec_workspace_size(dims, T):
    return lib().rssm_mamba2_spec_workspace_size(ctypes.byref(dims), int(T))


def rssm_mamba2_spec_verify(dims, T, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z, ring_x,
                            ring_dt, ring_B, cache_indices, slot_cnt, slot_base, slot_flush,
                            workspace, workspace_bytes, y, dev_err=None, stream=None):
    _call("rssm_mamba2_spec_verify", ctypes.byref(dims), int(T), _ptr(state), _ptr(x),
          _ptr(dt_raw), _ptr(dt_bias), int(dt_softplus), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
          _ptr(z), _ptr(ring_x), _ptr(ring_dt), _ptr(ring_B), _ptr(cache_indices), _ptr(slot_cnt),
          _ptr(slot_base), _ptr(slot_flush), _ptr(workspace), workspace_bytes, _ptr(y),
          _ptr(dev_err), _stream(stream))
