"""Integer cursor model of ReplaySSM (oracle side).

TEST INFRASTRUCTURE: only the tests, the smoke check and the CPU-baseline leg of
the benchmark import this module.

Sources:
  [M2]   "ReplaySSM: cache SSM inputs for faster Mamba2 standard decode" (vLLM PR
         48018 report), 实现拆解 item 3: the metadata builder gives every decode
         row a write_pos and an is_flush flag; 关键源码片段: write_pos / is_flush
         are passed to the output kernel per row.
  [GDN]  "GDN ReplaySSM decode (Part A of RFC 28511)" (SGLang PR 28451 report),
         实现拆解 item 2: a static force-flush mask forces a flush on chosen rows.
  [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify" (SGLang PR 28695 report),
         实现拆解 item 2: per-slot cursors write_pos, cache_base, is_flush of a
         circular ring; 关键源码片段 (server_args): the ring must hold at least
         twice the maximum number of draft tokens.

Readings (the pages give no formula for the cursors):
  * Standard decode. w = write_pos is the ring index of the current step's
    entry. Entries 0..w are live once the step is appended. The row flushes when
    w == L-1 or its force-flush bit is set; a flush folds entries 0..w into the
    checkpoint and the slot's next write_pos is 0, otherwise w+1.
  * Speculative verify (circular ring). Per slot: cnt (committed, unfolded
    entries; stored in the write_pos array), base (ring position of the oldest
    unfolded entry) and flush. A verify round first folds the cnt committed
    entries into the checkpoint when flush is set; its T drafts go to ring
    positions (base + cnt + j) mod L. The commit with a accepted drafts first
    retires a fold done by that verify (base <- (base + cnt) mod L, cnt <- 0),
    then sets cnt <- cnt + a and flush <- (cnt + T > L), so the next round's
    drafts always fit in the ring.
  * Reset: the listed slots restart with cnt = base = 0 and no flush.
"""
from typing import List, Optional, Sequence, Tuple


def advance_standard(slot_wp: List[int], ci: Sequence[int], force: Optional[Sequence[int]],
                     L: int) -> Tuple[List[int], List[int]]:
    """One standard decode step. Mutates slot_wp; returns (row_wp, row_flush).

    Rows with a negative cache index are padding: row_wp = 0, row_flush = 0 and
    no slot changes."""
    row_wp, row_flush = [], []
    for b, s in enumerate(ci):
        if s < 0 or s >= len(slot_wp):
            row_wp.append(0)
            row_flush.append(0)
            continue
        w = slot_wp[s]
        f = 1 if (w == L - 1 or (force is not None and force[b])) else 0
        row_wp.append(w)
        row_flush.append(f)
        slot_wp[s] = 0 if f else w + 1
    return row_wp, row_flush


def spec_commit(slot_cnt: List[int], slot_base: List[int], slot_flush: List[int],
                ci: Sequence[int], accepted: Sequence[int], L: int, T: int) -> None:
    """Commit after a verify round (mutates the three per-slot cursor arrays)."""
    for b, s in enumerate(ci):
        if s < 0 or s >= len(slot_cnt):
            continue
        if slot_flush[s]:
            slot_base[s] = (slot_base[s] + slot_cnt[s]) % L
            slot_cnt[s] = 0
        slot_cnt[s] += accepted[b]
        slot_flush[s] = 1 if slot_cnt[s] + T > L else 0


def spec_reset(slot_cnt: List[int], slot_base: List[int], slot_flush: List[int],
               slots: Sequence[int]) -> None:
    for s in slots:
        if 0 <= s < len(slot_cnt):
            slot_cnt[s] = 0
            slot_base[s] = 0
            slot_flush[s] = 0


def spec_draft_positions(cnt: int, base: int, L: int, T: int) -> List[int]:
    """Ring positions of the T drafts of one verify round."""
    return [(base + cnt + j) % L for j in range(T)]
