"""Host model of the tensor-core kernel's Q6_K raw-row loader (CPU only).

The loader warp's 32 lanes fill a 128-row slot with 16-byte cp.async copies:
lane l takes chunks l, l + 32, ... of the slot, chunk c = 14 r + q being
bytes 16 q .. 16 q + 15 of row r's 224-byte window, which starts at the
16-byte boundary at or below the row's 210-byte super-block (Q6_K blocks,
ggml layout: 128 B ql, 64 B qh, 16 B scales, f16 d). The lane walks (r, q)
incrementally (c + 32 is r + 2, q + 4 with a carry). A chunk is read only for
rows of the matrix and only up to the end of W; the rest is zero-filled.

This model replays that walk and checks, for many shapes and base
alignments, that every chunk of the slot is written exactly once, that the
shared-memory offsets stay inside the slot (rows of 240 bytes), that no read
leaves W, and that the bytes read cover each row's whole super-block.
"""
import random

import pytest

KBM, KCH, ROW_PITCH, SB_BYTES = 128, 14, 240, 210


def walk(wbase, row_bytes, w_rows, wrow, sbg):
    """Yield (lane, smem_offset, src, valid) for every copy of one slot."""
    wend = wbase + row_bytes * w_rows
    rows_ok = min(KBM, w_rows - wrow)
    per_lane = KBM * KCH // 32
    dr, dq = 32 // KCH, 32 % KCH
    for lane in range(32):
        r, q = lane // KCH, lane % KCH
        rb = wbase + (wrow + r) * row_bytes + SB_BYTES * sbg
        for _ in range(per_lane):
            a = (rb & ~15) + 16 * q
            src, valid = wbase, 0
            if r < rows_ok and a < wend:
                src, valid = a, min(16, wend - a)
            yield lane, r * ROW_PITCH + 16 * q, src, valid, r, q
            r += dr
            q += dq
            rb += dr * row_bytes
            if q >= KCH:
                q -= KCH
                r += 1
                rb += row_bytes


def check_slot(wbase, k, w_rows, wrow, sbg):
    row_bytes = (k // 256) * SB_BYTES
    wend = wbase + row_bytes * w_rows
    seen = set()
    covered = {}
    for lane, off, src, valid, r, q in walk(wbase, row_bytes, w_rows, wrow, sbg):
        assert 0 <= r < KBM and 0 <= q < KCH
        assert (r, q) not in seen, "chunk written twice"
        seen.add((r, q))
        assert off % 16 == 0 and off + 16 <= KBM * ROW_PITCH, "outside the slot"
        assert src % 16 == 0, "cp.async source must be 16-byte aligned"
        assert 0 <= valid <= 16
        if valid:
            assert wbase <= src and src + valid <= wend, "read outside W"
            covered.setdefault(r, []).append((src, src + valid))
    assert len(seen) == KBM * KCH, "chunk left unwritten"
    # every row of the matrix: its super-block's 210 bytes were read
    for r in range(min(KBM, w_rows - wrow)):
        start = wbase + (wrow + r) * row_bytes + SB_BYTES * sbg
        spans = sorted(covered.get(r, []))
        pos = start
        for a, b in spans:
            if a <= pos < b:
                pos = b
        assert pos >= start + SB_BYTES, f"row {r}: super-block not fully copied"
        # the decoder reads from the window's start plus (start & 15)
        assert (start & 15) + SB_BYTES <= KCH * 16


@pytest.mark.parametrize("k", [256, 1024, 2560, 4096, 14336])
@pytest.mark.parametrize("base_mod", [0, 16, 48, 112])
def test_q6k_window_walk(k, base_mod):
    rng = random.Random(k * 131 + base_mod)
    nsb = k // 256
    for w_rows in (1, 127, 128, 129, 385, 1000):
        tiles = range(0, w_rows, KBM)
        for wrow in tiles:
            for sbg in {0, nsb - 1, rng.randrange(nsb)}:
                check_slot(4096 + base_mod, k, w_rows, wrow, sbg)


def test_model_catches_a_wrong_carry():
    """A walk whose carry drops the row step revisits chunks and leaves others unwritten."""
    visited = []
    for lane in range(32):
        r, q = lane // KCH, lane % KCH
        for _ in range(KBM * KCH // 32):
            visited.append((r, q))
            r += 32 // KCH
            q += 32 % KCH
            if q >= KCH:
                q -= KCH  # the carry's row step is missing here
    assert len(set(visited)) < KBM * KCH
