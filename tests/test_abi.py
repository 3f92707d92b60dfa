"""The C-ABI library loads, exports every symbol include/rssm.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import ssm_linear_attention_gb300 as ssm
from ssm_linear_attention_gb300 import _binding as B
from ssm_linear_attention_gb300 import build as rbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "rssm.h")


@pytest.fixture(scope="module")
def lib():
    rbuild.build()
    return ssm.lib()


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rssm_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_abi_version_and_status_strings(lib):
    assert ssm.rssm_abi_version() == 1
    for st in range(5):
        assert ssm.rssm_status_string(st)
    assert ssm.rssm_status_string(99) == "unknown status"


def _m2(**kw):
    d = dict(batch=4, nheads=8, headdim=64, dstate=128, ngroups=2, ring_len=4, num_slots=8,
             state_dtype=B.RSSM_BF16, act_dtype=B.RSSM_BF16, out_dtype=B.RSSM_F32)
    d.update(kw)
    return B.Mamba2Dims(**d)


FAKE = 0x10000  # aligned non-null address; never dereferenced (validation fails first)


def _rc(name, *args):
    return getattr(ssm.lib(), name)(*args)


def test_cursor_validation(lib):
    L = ssm.lib()
    assert L.rssm_advance_cursors(9, FAKE, None, None, FAKE, None, None, 4, 8, 4, 0, FAKE, FAKE,
                                  None, None) == B.RSSM_ERR_INVALID_ARG
    assert L.rssm_advance_cursors(0, FAKE, None, None, FAKE, None, None, 4, 8, 0, 0, FAKE, FAKE,
                                  None, None) == B.RSSM_ERR_CONFIG
    assert L.rssm_advance_cursors(0, None, None, None, FAKE, None, None, 4, 8, 4, 0, FAKE, FAKE,
                                  None, None) == B.RSSM_ERR_INVALID_ARG
    assert L.rssm_advance_cursors(0, FAKE, None, None, FAKE, None, None, 4, 8, 4, 0, None, FAKE,
                                  None, None) == B.RSSM_ERR_INVALID_ARG
    # spec commit: ring must hold twice the drafts
    assert L.rssm_advance_cursors(1, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, 8, 7, 4, None, None,
                                  None, None) == B.RSSM_ERR_CONFIG
    assert L.rssm_advance_cursors(1, FAKE, None, FAKE, FAKE, None, FAKE, 4, 8, 8, 4, None, None,
                                  None, None) == B.RSSM_ERR_INVALID_ARG
    # empty batch is a no-op, even with null buffers
    assert L.rssm_advance_cursors(0, None, None, None, None, None, None, 0, 8, 4, 0, None, None,
                                  None, None) == B.RSSM_OK


def test_mamba2_validation(lib):
    d = _m2()
    by = ctypes.byref
    # tables (4 rows x 8 heads x round4(2 * 4 + 1) floats), then the 256-byte work counter
    # at a 256-byte boundary
    assert B.rssm_mamba2_workspace_size(d) == (4 * 8 * 12 * 4 + 255) // 256 * 256 + 256
    assert B.rssm_mamba2_workspace_size(_m2(ngroups=3)) == 0
    # shapes
    for bad, code in [(dict(ngroups=3), B.RSSM_ERR_CONFIG), (dict(ring_len=0), B.RSSM_ERR_CONFIG),
                      (dict(headdim=32), B.RSSM_ERR_UNSUPPORTED),
                      (dict(dstate=96), B.RSSM_ERR_UNSUPPORTED),
                      (dict(state_dtype=7), B.RSSM_ERR_INVALID_ARG),
                      (dict(batch=-1), B.RSSM_ERR_INVALID_ARG)]:
        dd = _m2(**bad)
        assert _rc("rssm_ring_append", by(dd), FAKE, FAKE, None, 1, FAKE, FAKE, FAKE, FAKE, FAKE,
                   FAKE, None, None) == code
        assert _rc("rssm_mamba2_output", by(dd), FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE,
                   FAKE, FAKE, 1 << 20, FAKE, None, None) == code
    # null / misaligned pointers
    assert _rc("rssm_ring_append", by(d), None, FAKE, None, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
               None, None) == B.RSSM_ERR_INVALID_ARG
    assert _rc("rssm_mamba2_output", by(d), FAKE + 4, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE,
               FAKE, FAKE, 1 << 20, FAKE, None, None) == B.RSSM_ERR_INVALID_ARG
    # workspace too small
    assert _rc("rssm_mamba2_decode", by(d), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE,
               FAKE, FAKE, FAKE, 16, FAKE, None, None) == B.RSSM_ERR_INVALID_ARG
    assert _rc("rssm_mamba2_full_state_update", by(d), FAKE, FAKE, FAKE, None, 1, FAKE, FAKE, None,
               FAKE, None, FAKE, FAKE, None, None) == B.RSSM_ERR_INVALID_ARG


def test_binding_raises_with_status(lib):
    with pytest.raises(ssm.RSSMError) as ei:
        ssm.rssm_advance_cursors(0, FAKE, None, None, FAKE, None, None, 4, 8, 0, 0, FAKE, FAKE,
                                 None, stream=0)
    assert ei.value.status == B.RSSM_ERR_CONFIG


def test_copy_slots_validation(lib):
    L = ssm.lib()
    one = (B.SlotBuffer * 1)(B.SlotBuffer(FAKE, 64))
    many = (B.SlotBuffer * 13)(*[B.SlotBuffer(FAKE, 64) for _ in range(13)])
    zero = (B.SlotBuffer * 1)(B.SlotBuffer(FAKE, 0))
    nul = (B.SlotBuffer * 1)(B.SlotBuffer(None, 64))
    INV = B.RSSM_ERR_INVALID_ARG
    assert L.rssm_copy_slots(None, 1, FAKE, FAKE, 2, 8, None, None) == INV
    assert L.rssm_copy_slots(one, 0, FAKE, FAKE, 2, 8, None, None) == INV
    assert L.rssm_copy_slots(many, 13, FAKE, FAKE, 2, 8, None, None) == INV
    assert L.rssm_copy_slots(zero, 1, FAKE, FAKE, 2, 8, None, None) == INV
    assert L.rssm_copy_slots(nul, 1, FAKE, FAKE, 2, 8, None, None) == INV
    assert L.rssm_copy_slots(one, 1, FAKE, FAKE, -1, 8, None, None) == INV
    assert L.rssm_copy_slots(one, 1, FAKE, FAKE, 2, 0, None, None) == INV
    assert L.rssm_copy_slots(one, 1, None, FAKE, 2, 8, None, None) == INV
    assert L.rssm_copy_slots(one, 1, FAKE, FAKE + 4, 2, 8, None, None) == INV
    # nothing to copy: valid, launches nothing
    assert L.rssm_copy_slots(one, 1, None, None, 0, 8, None, None) == B.RSSM_OK


def test_binding_arity_matches_header(lib):
    # every ctypes signature has as many arguments as the C declaration
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "rssm.h")).read()
    decl = {}
    for m in re.finditer(r"\n[a-z_ 0-9*]+?\b(rssm_\w+)\(([^;]*?)\);", hdr):
        args = m.group(2).strip()
        decl[m.group(1)] = 0 if args in ("void", "") else args.count(",") + 1
    L = ssm.lib()
    for name in B.EXPORTS:
        assert len(getattr(L, name).argtypes or []) == decl[name], name


def _gdims(**kw):
    d = dict(batch=4, num_v_heads=8, num_k_heads=4, head_k_dim=128, head_v_dim=128, ring_len=8,
             num_slots=8, act_dtype=B.RSSM_BF16, out_dtype=B.RSSM_F32)
    d.update(kw)
    return B.GDNDims(**d)


def test_mamba2_spec_validation(lib):
    by = ctypes.byref
    d = _m2(ring_len=8)
    assert B.rssm_mamba2_spec_workspace_size(d, 0) == 0
    assert B.rssm_mamba2_spec_workspace_size(d, 5) == 0
    assert B.rssm_mamba2_spec_workspace_size(d, 3) == 4 * 8 * ((3 * 8 + 6 + 3) // 4 * 4) * 4

    def call(dd, T, state=FAKE, ws_bytes=1 << 20):
        return _rc("rssm_mamba2_spec_verify", by(dd), T, state, FAKE, FAKE, None, 1, FAKE, FAKE,
                   FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes, FAKE,
                   None, None)
    assert call(d, 5) == B.RSSM_ERR_UNSUPPORTED          # T > 4
    assert call(_m2(ring_len=40), 2) == B.RSSM_ERR_UNSUPPORTED   # L > 32
    assert call(_m2(ring_len=5), 3) == B.RSSM_ERR_CONFIG          # L < 2T
    assert call(d, 2, state=None) == B.RSSM_ERR_INVALID_ARG
    assert call(d, 2, ws_bytes=16) == B.RSSM_ERR_INVALID_ARG       # workspace too small
    assert call(_m2(ring_len=8, batch=0), 2) == B.RSSM_OK          # nothing to do


def test_kda_validation(lib):
    by = ctypes.byref
    assert B.rssm_kda_workspace_size(_gdims()) > 0
    assert B.rssm_kda_workspace_size(_gdims(head_k_dim=64)) == 0
    assert B.rssm_kda_workspace_size(_gdims(ring_len=65)) == 0
    out = lambda dd, st=FAKE: _rc("rssm_kda_output", by(dd), st, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, 1 << 30, FAKE, None, None)
    assert out(_gdims(), st=None) == B.RSSM_ERR_INVALID_ARG
    assert out(_gdims(num_k_heads=3)) == B.RSSM_ERR_CONFIG
    assert out(_gdims(head_v_dim=48)) == B.RSSM_ERR_UNSUPPORTED
    pre = _rc("rssm_kda_prepare", by(_gdims()), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
              FAKE, FAKE, 16, None, None)
    assert pre == B.RSSM_ERR_INVALID_ARG                            # workspace too small
    full = _rc("rssm_kda_full_state_decode", by(_gdims()), FAKE, FAKE, FAKE, FAKE, FAKE, None,
               FAKE, FAKE, None, None)
    assert full == B.RSSM_ERR_INVALID_ARG                           # gates missing


def test_stochastic_rounding_validation(lib):
    by = ctypes.byref
    d = _m2()
    rc = _rc("rssm_mamba2_output_sr", by(d), FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
             FAKE, 1 << 20, FAKE, None, None, None)
    assert rc == B.RSSM_ERR_INVALID_ARG                             # no generator state
    rc = _rc("rssm_mamba2_full_state_update_sr", by(d), FAKE, FAKE, FAKE, None, 1, FAKE, FAKE,
             FAKE, FAKE, None, FAKE, FAKE, FAKE + 8, None, None)
    assert rc == B.RSSM_ERR_INVALID_ARG                             # misaligned generator state
    assert _rc("rssm_philox4x32_fill", 1, 2, None, 0, None) == B.RSSM_OK
    assert _rc("rssm_philox4x32_fill", 1, 2, None, 4, None) == B.RSSM_ERR_INVALID_ARG


def test_debug_pipeline_copy_validation(lib):
    f = "rssm_debug_pipeline_copy"
    bad = ssm.RSSM_ERR_INVALID_ARG
    assert _rc(f, FAKE, FAKE, -1, -1, 1000, None, None) == bad          # negative count
    assert _rc(f, FAKE, FAKE, 4, 4, 1000, None, None) == bad            # stall tile out of range
    assert _rc(f, FAKE, FAKE, 4, -1, 0, None, None) == bad              # wait limit too short
    assert _rc(f, FAKE, FAKE, 4, -1, 2000001, None, None) == bad        # wait limit too long
    assert _rc(f, None, FAKE, 4, -1, 1000, None, None) == bad           # null source
    assert _rc(f, FAKE, FAKE + 4, 4, -1, 1000, None, None) == bad       # misaligned destination
    assert _rc(f, FAKE, FAKE, 0, -1, 1000, None, None) == ssm.RSSM_OK   # nothing to copy


def test_debug_umma_fold_validation(lib):
    f = "rssm_debug_umma_fold"
    bad = ssm.RSSM_ERR_INVALID_ARG
    assert _rc(f, FAKE, FAKE, 16, 128, FAKE, None, None) == bad     # w beyond the 16 entries
    assert _rc(f, FAKE, FAKE, -1, 128, FAKE, None, None) == bad
    assert _rc(f, FAKE, FAKE, 3, 96, FAKE, None, None) == bad       # N not 64 or 128
    assert _rc(f, None, FAKE, 3, 64, FAKE, None, None) == bad
    assert _rc(f, FAKE, FAKE, 3, 64, FAKE + 8, None, None) == bad   # misaligned D
