"""CPU model of the stack kernel's ring protocol: the rule that its stage
count be a multiple of the consumer warps.

In the decode-stack kernel one producer fills ring stages in box order and
consumer warp w takes boxes j = w, w + W, w + 2W, ... of every phase; box j of
a phase uses stage (q + j) % nst, q being the CTA's running box count.  A
consumer waits on a stage's full barrier by parity, which cannot tell the use
it wants from the one two uses back.  The model replays the waits: it marks a
wait that would return while the stage still holds an older use (an early
read) and checks that the ring sizes the host can choose (a multiple of W, as
round_ring_to_warps makes them) never give one, while other sizes do.
"""
import random

import pytest


def _parity_wait_passes(fills, u):
    """mbarrier parity wait for use u of a stage (its (u+1)-th fill): it
    passes when the count of completed fills has the parity of u + 1."""
    return fills % 2 == (u + 1) % 2


def _early_reads(nst, W, phases):
    """Count waits that a parity check would pass while the stage does not
    yet hold the awaited use.

    Worst-case interleaving: a warp may reach a wait at any time after its
    own previous box; the producer fills use u of a stage only after use
    u - 1 was released by the warp that consumed it.  So when use u's warp
    also consumed use u - 1, the stage holds at least u fills by the time it
    waits; when another warp owns use u - 1, the stage may still hold only
    u - 1 fills (use u - 1 not landed yet).  Between phases all warps meet at a
    barrier, so a phase's first use of a stage finds every earlier use done."""
    uses = [0] * nst        # uses of each stage before the current phase
    early = 0
    q = 0
    for nbox in phases:
        owners = {}
        for j in range(nbox):
            owners.setdefault((q + j) % nst, []).append(j % W)
        for s, ws in owners.items():
            for i, w in enumerate(ws):
                u = uses[s] + i
                fewest_fills = u if (i == 0 or ws[i - 1] == w) else u - 1
                if fewest_fills < u + 1 and _parity_wait_passes(fewest_fills, u):
                    early += 1
            uses[s] += len(ws)
        q += nbox
    return early


def round_ring_to_warps(nst, warps):
    return nst // warps * warps


@pytest.mark.parametrize("W", [8, 16])
def test_ring_multiple_of_warps_never_reads_early(W):
    rng = random.Random(W)
    for n in range(W, 33):
        nst = round_ring_to_warps(n, W)
        if nst < W:
            continue
        for _ in range(50):
            phases = [rng.randint(1, 200) for _ in range(12)]
            assert _early_reads(nst, W, phases) == 0, (nst, W, phases)


@pytest.mark.parametrize("W", [8, 16])
def test_ring_not_multiple_of_warps_reads_early(W):
    """The model is not vacuous: a ring that is not a multiple of W lets a
    warp wait on a stage another warp still has to consume."""
    rng = random.Random(100 + W)
    found = 0
    for nst in range(W + 1, 33):
        if nst % W == 0:
            continue
        phases = [rng.randint(nst + 1, 200) for _ in range(6)]
        found += _early_reads(nst, W, phases) > 0
    assert found > 0


def test_host_rounding_matches_rule():
    for W in (8, 16):
        for n in range(W, 64):
            r = round_ring_to_warps(n, W)
            assert r % W == 0 and r <= n and n - r < W

