"""A CPU model of the decode kernel's shared-memory ring protocol (no GPU).

The decode kernel's producer fills stage ``it % S`` for block ``it`` and
signals a "full" mbarrier; for each of the CTA's H KV heads, consumer warp
``it % W`` of that head waits on the barrier by phase parity, reads the stage
and arrives on its "empty" barrier (H arrivals complete a phase), which the
producer waits on (parity) before refilling.  A parity wait only tells two
consecutive phases apart, so a waiter must never be two phases ahead of its
barrier.  This model runs the protocol under random interleavings with the
mbarrier rules written out and checks that every consumer reads the block it
expects.  It pins the rule the kernel's static_assert encodes: the stage count
must be a multiple of the per-head warp count (6 stages over 4 warps breaks).
"""

import random

import pytest


class Barrier:
    """An mbarrier: arrival count, transaction bytes, phase."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0

    def phase_done(self, parity):
        # try_wait.parity(P) succeeds once the phase with parity P has completed,
        # i.e. while the current phase's parity differs from P.
        return (self.phase & 1) != parity

    def arrive(self, tx=0):
        assert self.pending > 0, "arrive on a phase with no pending arrival"
        self.pending -= 1
        self.tx += tx
        self._advance()

    def complete_tx(self, tx):
        self.tx -= tx
        assert self.tx >= 0
        self._advance()

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count


def run_protocol(nblk, stages, warps, seed, heads=1):
    rnd = random.Random(seed)
    full = [Barrier(1) for _ in range(stages)]
    empty = [Barrier(heads) for _ in range(stages)]
    holds = [None] * stages          # block whose bytes have landed in the stage
    in_flight = []                   # (stage, block) copies not yet landed
    produced = 0
    consumers = [(h, w) for h in range(heads) for w in range(warps)]
    next_block = {c: c[1] for c in consumers}
    for _ in range(10 ** 6):
        moves = []
        if produced < nblk:
            s = produced % stages
            if empty[s].phase_done(((produced // stages) & 1) ^ 1):
                moves.append(("produce",))
        if in_flight:
            moves.append(("land",))
        for c in consumers:
            it = next_block[c]
            if it < nblk and full[it % stages].phase_done((it // stages) & 1):
                moves.append(("consume", c))
        if not moves:
            break
        m = rnd.choice(moves)
        if m[0] == "produce":
            s = produced % stages
            full[s].arrive(tx=1)                      # arrive.expect_tx + TMA issue
            in_flight.append((s, produced))
            produced += 1
        elif m[0] == "land":
            s, it = in_flight.pop(rnd.randrange(len(in_flight)))
            holds[s] = it
            full[s].complete_tx(1)
        else:
            w = m[1]
            it = next_block[w]
            s = it % stages
            assert holds[s] == it, f"warp {w} read stage {s} holding block {holds[s]}, wanted {it}"
            empty[s].arrive()
            next_block[w] += warps
    assert produced == nblk and not in_flight
    assert all(next_block[c] >= nblk for c in consumers)


@pytest.mark.parametrize("stages,heads", [(8, 1), (16, 1), (8, 2), (16, 2)])
def test_kernel_stage_counts_are_safe(stages, heads):
    # The kernel uses 8 or 16 stages, 4 consumer warps per KV head, and one
    # (16-bit caches) or two (E4M3) KV heads per CTA.
    for nblk in (1, 2, 3, 5, 8, 13, 32, 64):
        for seed in range(100):
            run_protocol(nblk, stages, 4, seed, heads)


@pytest.mark.parametrize("heads", [1, 2])
def test_stage_count_not_a_multiple_of_warps_breaks(heads):
    with pytest.raises(AssertionError):
        for seed in range(300):
            run_protocol(8, 6, 4, seed, heads)
