"""Model check of the unit queue of the expert GEMM's small-batch variant
(down takes whole units dynamically; the producer hands each unit to the MMA
issuer, the scale-factor warps and the epilogue through a ring of tagged
shared-memory words and never waits for the readers).

The kernel relies on the pipeline's own barriers to keep the producer at most
NS + 3 units ahead of the slowest reader, so that a 16-entry ring is never
overwritten before every role has read an entry.  This test explores random
interleavings of the four roles under exactly those barriers and checks that
bound, for every ring depth NS the kernel uses and for units of 1 to 8 stages:

  producer  writes entry i, then per stage g of unit i waits until the MMA has
            committed stage g - NS (the stage's empty barrier) and issues it;
  scales    reads entry i, then per stage g waits for the same empty barrier
            and stores the stage's scales (its arrival on the full barrier);
  MMA       reads entry i, waits until the epilogue has taken the accumulator
            of unit i - 2 (two accumulator buffers), then per stage waits for
            the copies and the scales of the stage and commits it;
  epilogue  reads entry i, waits until the MMA committed every stage of unit
            i, and frees the accumulator.
"""
from __future__ import annotations

import random

import pytest

K_UQ = 16  # entries of the ring in the kernel


def _run(ns: int, stages: int, units: int, rng: random.Random) -> int:
    """One random interleaving; returns the largest producer lead over the
    slowest reader seen when writing an entry."""
    total = units * stages
    prod_unit = 0          # next entry the producer writes
    prod_stage = 0         # next stage the producer issues (global index)
    sf_unit, sf_read, sf_stage = 0, False, 0
    mma_unit, mma_read, mma_stage, committed = 0, False, 0, 0
    epi_unit, epi_read = 0, False
    acc_freed = 0          # units whose accumulator the epilogue has freed
    max_lead = 0
    term = False           # the ending entry (-1) is written

    def readers_taken() -> int:
        # entries every reader has read: each role has read entries < its
        # current unit, and its current unit's entry once it took it
        return min(sf_unit + sf_read, mma_unit + mma_read, epi_unit + epi_read)

    while epi_unit < units:
        moves = []
        # producer: write the entry of the next unit once the previous unit's
        # stages are issued, then issue stages
        if prod_unit <= units and not term and prod_stage == prod_unit * stages:
            moves.append("p_write")  # a unit's entry, or after the last one the ending entry
        elif prod_stage < min(total, prod_unit * stages):
            if prod_stage < ns or committed > prod_stage - ns:
                moves.append("p_issue")
        if not sf_read and sf_unit < units and sf_unit < prod_unit:
            moves.append("s_read")
        elif sf_read and sf_stage < (sf_unit + 1) * stages:
            if sf_stage < ns or committed > sf_stage - ns:
                moves.append("s_store")
        if not mma_read and mma_unit < units and mma_unit < prod_unit:
            moves.append("m_read")
        elif mma_read and mma_stage == mma_unit * stages and mma_unit >= 2 and acc_freed < mma_unit - 1:
            pass  # waiting for the accumulator of unit mma_unit - 2
        elif mma_read and mma_stage < (mma_unit + 1) * stages:
            if mma_stage < prod_stage and mma_stage < sf_stage:
                moves.append("m_commit")
        if not epi_read and epi_unit < prod_unit:
            moves.append("e_read")
        elif epi_read and committed >= (epi_unit + 1) * stages:
            moves.append("e_free")
        assert moves, "the model deadlocked"
        mv = rng.choice(moves)
        if mv == "p_write":
            lead = prod_unit - readers_taken()
            max_lead = max(max_lead, lead)
            # entry prod_unit overwrites entry prod_unit - K_UQ: all must have read it
            assert prod_unit - K_UQ < readers_taken(), (ns, stages, prod_unit, readers_taken())
            if prod_unit == units:
                term = True
            else:
                prod_unit += 1
        elif mv == "p_issue":
            prod_stage += 1
        elif mv == "s_read":
            sf_read = True
        elif mv == "s_store":
            sf_stage += 1
            if sf_stage == (sf_unit + 1) * stages:
                sf_unit, sf_read = sf_unit + 1, False
        elif mv == "m_read":
            mma_read = True
        elif mv == "m_commit":
            mma_stage += 1
            committed += 1
            if mma_stage == (mma_unit + 1) * stages:
                mma_unit, mma_read = mma_unit + 1, False
        elif mv == "e_read":
            epi_read = True
        elif mv == "e_free":
            acc_freed += 1
            epi_unit, epi_read = epi_unit + 1, False
    return max_lead


@pytest.mark.parametrize("ns", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("stages", [1, 2, 6, 8])
def test_unit_queue_is_never_overrun(ns, stages):
    rng = random.Random(1000 * ns + stages)
    lead = 0
    for _ in range(60):
        lead = max(lead, _run(ns, stages, units=40, rng=rng))
    # the kernel's bound: the producer is at most NS + 3 entries ahead
    assert lead <= ns + 3 < K_UQ


def test_model_reaches_the_bound_with_one_stage_units():
    """The bound matters: with one-stage units and six ring stages the
    producer does run NS + 2 = 8 units ahead of the slowest reader, so a ring
    of 8 entries or fewer would be overrun."""
    rng = random.Random(7)
    lead = max(_run(6, 1, units=40, rng=rng) for _ in range(200))
    assert lead == 6 + 2
