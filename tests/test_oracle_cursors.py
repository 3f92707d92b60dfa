"""Pins for the integer cursor model (standard decode and the circular spec ring)."""
import itertools
import random

import pytest

from oracle import cursors


@pytest.mark.parametrize("L", [1, 2, 3, 4, 7, 16])
def test_standard_cursor_closed_form(L):
    # Without forced flushes, a slot that starts at write_pos w0 has write_pos
    # (w0 + k) mod L at step k and flushes exactly when that is L - 1.
    for w0 in range(L):
        slot_wp = [w0]
        for k in range(3 * L + 2):
            rw, rf = cursors.advance_standard(slot_wp, [0], None, L)
            assert rw == [(w0 + k) % L]
            assert rf == [1 if (w0 + k) % L == L - 1 else 0]


def test_standard_cursor_exhaustive_force():
    # every (w, force) pair for L = 5: flush iff w == L-1 or force; next wp 0 on flush
    L = 5
    for w, force in itertools.product(range(L), (0, 1)):
        slot_wp = [w]
        rw, rf = cursors.advance_standard(slot_wp, [0], [force], L)
        assert rw == [w]
        assert rf == [int(w == L - 1 or force)]
        assert slot_wp == [0 if rf[0] else w + 1]


def test_standard_cursor_padding_and_slot_map():
    slot_wp = [3, 1, 0, 2]
    rw, rf = cursors.advance_standard(slot_wp, [2, -1, 0, 7], None, 4)
    assert rw == [0, 0, 3, 0] and rf == [0, 0, 1, 0]
    assert slot_wp == [0, 1, 1, 2]


def test_spec_ring_never_overwrites_live_entries():
    # Simulate the ring contents: committed tokens must sit at base..base+cnt-1 (mod L),
    # in commit order, and a round's drafts must never land on a live entry.
    rnd = random.Random(0)
    for L, T in [(8, 4), (16, 4), (9, 3), (4, 2)]:
        cnt, base, flush = [0], [0], [0]
        ring = [None] * L
        live = []          # committed, unfolded token ids in order
        folded = []
        tok = 0
        for _ in range(400):
            if flush[0]:
                folded.extend(live)
                live = []
                c_eff, b_eff = 0, (base[0] + cnt[0]) % L
            else:
                c_eff, b_eff = cnt[0], base[0]
            for i, t in enumerate(live):
                assert ring[(b_eff + i) % L] == t
            pos = cursors.spec_draft_positions(cnt[0], base[0], L, T)
            assert c_eff + T <= L
            live_pos = {(b_eff + i) % L for i in range(c_eff)}
            assert not live_pos.intersection(pos)
            drafts = list(range(tok, tok + T))
            tok += T
            for p, t in zip(pos, drafts):
                ring[p] = t
            a = rnd.randint(0, T)
            cursors.spec_commit(cnt, base, flush, [0], [a], L, T)
            live.extend(drafts[:a])
            assert cnt[0] == len(live)
            assert flush[0] == int(cnt[0] + T > L)


def test_spec_reset():
    cnt, base, flush = [3, 4], [5, 6], [1, 1]
    cursors.spec_reset(cnt, base, flush, [1])
    assert (cnt, base, flush) == ([3, 0], [5, 0], [1, 0])
