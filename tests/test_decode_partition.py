"""The run partition of the decode-sized W4A16 product, checked on the host.

The product walks stages (64 input rows x 1024 columns) in column-block-major
order, b = cb * nch + ch, and CTA c owns the contiguous run
[floor(c B / ctas), floor((c + 1) B / ctas)).  Where a run leaves a column
block the CTA stores that block's sums in slot c + cb; the last of the CTAs
c_first .. c_last that touch a block (a ticket counter per block) adds their
slots in order.  The kernel's correctness rests on four facts about this
integer arithmetic, which these tests check over many shapes:

  * every stage belongs to exactly one run, and dq_cta_of(b) names its CTA;
  * a run meets a column block in at most one contiguous segment;
  * the slots c + cb are distinct and below 1024 + ncb (the workspace);
  * the CTAs that touch block cb are exactly c_first .. c_last, so the
    ticket target c_last - c_first + 1 is the number of segments.
"""
import random

import pytest

MAX_CTAS = 1024  # the grid bound the workspace is sized for


def cta_of(b, B, ctas):
    """The largest c with floor(c B / ctas) <= b (integer arithmetic as in the kernel)."""
    return ((b + 1) * ctas - 1) // B


def runs(B, ctas):
    return [(c * B // ctas, (c + 1) * B // ctas) for c in range(ctas)]


def check_partition(nch, ncb, ctas):
    B = nch * ncb
    ctas = min(ctas, MAX_CTAS, B)
    rs = runs(B, ctas)
    owner = [None] * B
    for c, (b0, b1) in enumerate(rs):
        assert b1 > b0, "every CTA gets at least one stage"
        for b in range(b0, b1):
            assert owner[b] is None
            owner[b] = c
    assert all(o is not None for o in owner)
    for b in range(B):
        assert cta_of(b, B, ctas) == owner[b]
    slots = set()
    for c, (b0, b1) in enumerate(rs):
        blocks = [b // nch for b in range(b0, b1)]
        # one contiguous segment per column block: the blocks of a run are non-decreasing
        assert blocks == sorted(blocks)
        for cb in set(blocks):
            slot = c + cb
            assert slot not in slots
            assert slot < MAX_CTAS + ncb
            slots.add(slot)
    for cb in range(ncb):
        touching = sorted({owner[b] for b in range(cb * nch, (cb + 1) * nch)})
        c_first, c_last = cta_of(cb * nch, B, ctas), cta_of((cb + 1) * nch - 1, B, ctas)
        assert touching == list(range(c_first, c_last + 1))


@pytest.mark.parametrize("nch,ncb,ctas", [
    (128, 28, 148),   # the large MLP layer on a 148-SM part
    (1, 8, 148),      # one 64-row chunk: one stage per CTA
    (16, 28, 148),    # runs of about 3 stages crossing column blocks
    (128, 2, 148),    # many segments per column block
    (172, 4, 148),    # the MLP-down layer's rows
    (3, 1, 148),      # fewer stages than CTAs
    (64, 1000, 1024), # a grid at the workspace bound
])
def test_decode_partition_shapes(nch, ncb, ctas):
    check_partition(nch, ncb, ctas)


def test_decode_partition_random():
    rng = random.Random(7)
    for _ in range(300):
        check_partition(rng.randint(1, 200), rng.randint(1, 60), rng.randint(1, 1100))
