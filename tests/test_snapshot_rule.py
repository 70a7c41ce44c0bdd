"""The compaction kernel's word-local snapshot rule against the oracle's CSR numbering.

An event at chunk c is some output group's predecessor (SparseGDN Sec. 2.5, Eqs. 16 and
20-21) iff the first even chunk m > c satisfies m <= the row's next event chunk and
m <= 2(G-1).  For odd c, m = c + 1 and the first condition always holds; for even c it
fails exactly when chunk c + 1 holds an event, which lies in the same 32-chunk mask word.
So the decision needs only the event's own word, which is how the GPU compaction takes it
(one block scan numbers events and snapshots together).  This file restates that bitwise
form and checks, on exhaustive and random masks, that numbering its events densely in CSR
order reproduces the oracle's snapshot slots, which follow the definition directly.
"""
import itertools

import numpy as np
import pytest

import oracle


def snap_bits(bits, w, G):
    """Events of mask word w (chunks 32w .. 32w + 31) that some group reads, as a bit mask."""
    top = 2 * (G - 1) - 32 * w - 2  # the largest allowed (c & ~1) - 32w
    if top < 0:
        lim = 0
    elif top >= 30:
        lim = 0xFFFFFFFF
    else:
        lim = (2 << ((top & ~1) + 1)) - 1
    return bits & (0xAAAAAAAA | (~(bits >> 1) & 0xFFFFFFFF)) & lim


def word_rule_slots(mask, ref):
    """Snapshot slots of the oracle's CSR events by the word-local rule, numbered densely."""
    B, P, C = mask.shape
    G = (C + 1) // 2
    rows = mask.reshape(B * P, C)
    slots, nxt = [], 0
    for j in range(B * P):
        i = int(ref["row_pair"][j])
        for e in range(int(ref["row_ptr"][j]), int(ref["row_ptr"][j + 1])):
            c = int(ref["ev_chunk"][e])
            w, p = divmod(c, 32)
            bits = 0
            for q in range(32):
                cc = 32 * w + q
                if cc < C and rows[i, cc]:
                    bits |= 1 << q
            if (snap_bits(bits, w, G) >> p) & 1:
                slots.append(nxt)
                nxt += 1
            else:
                slots.append(-1)
    return np.array(slots, dtype=np.int64), nxt


def check(mask):
    ref = oracle.events(mask)
    slots, n = word_rule_slots(mask, ref)
    assert n == ref["n_snap"]
    assert np.array_equal(slots, np.asarray(ref["snap_slot"], dtype=np.int64))


@pytest.mark.parametrize("C", range(1, 9))
def test_every_single_row_mask_up_to_8_chunks(C):
    for bits in itertools.product([0, 1], repeat=C):
        check(np.array(bits, np.uint8).reshape(1, 1, C))


@pytest.mark.parametrize("C", [31, 32, 33, 62, 63, 64, 65, 66, 95, 96, 97, 127, 128, 129, 200])
@pytest.mark.parametrize("p", [0.1, 0.5, 0.9, 1.0])
def test_random_masks_across_word_boundaries(C, p):
    rng = np.random.default_rng(1000 * C + int(100 * p))
    for B, P in ((1, 1), (2, 3), (3, 5)):
        check((rng.random((B, P, C)) < p).astype(np.uint8))


def test_alternating_and_paired_patterns():
    # even-odd pairs (only the odd event is read), lone even events (each read), and the last group
    for C in (64, 65, 96, 97):
        for pattern in ((1, 1, 0, 0), (1, 0), (0, 1), (1, 0, 0, 0), (1, 1, 1, 0)):
            row = np.array([pattern[c % len(pattern)] for c in range(C)], np.uint8)
            check(row.reshape(1, 1, C))
