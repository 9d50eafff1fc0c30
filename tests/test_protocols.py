"""Host models of the two wait protocols the kernels rely on, run under many
random interleavings (CPU only).

mbarrier semantics modelled (PTX mbarrier): a phase completes when its pending
arrival count and its transaction count are both zero; the count is then
re-armed and the phase number advances.  The transaction count may go
negative when bytes complete before the matching expect_tx.
`try_wait.parity(p)` succeeds while the current phase's parity differs from p,
which is why a waiter must never be more than one phase ahead.

1. The fused pipeline's ring (fused_tma.cu): one producer fills slot j % S
   with copy j after the consumers released that slot's previous fill; the
   consumers wait for copy j's fill, read it, release the slot.
2. The split-row exchange of the row kernel and the Lamport receive
   (fused.cu, lamport.cu): every CTA of a cluster, for each of its rows,
   arms its barrier b = row & 1 for C partials, pushes its partial into slot
   [b][rank] of every CTA (including itself; delivery takes any time) and
   waits for the phase (row >> 1) & 1 of barrier b.
"""
import random


class MBarrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, expect_tx=0):
        self.tx += expect_tx
        self.pending -= 1
        assert self.pending >= 0
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def try_wait_parity(self, parity):
        return (self.phase & 1) != parity


def run_ring(S, nt, rows, consumers, seed, wait_for_release=True):
    """One producer, `consumers` consumer warps (each must release a slot),
    copies in flight land in any order.  Checks that every consumer reads each
    copy's own data and that no fill overwrites a slot still being read."""
    rnd = random.Random(seed)
    total = rows * nt
    full = [MBarrier(1) for _ in range(S)]
    empty = [MBarrier(consumers) for _ in range(S)]
    slot_data = [None] * S
    readers_left = [0] * S            # consumers that have not released the slot's current fill
    issued = 0
    in_flight = []                    # copies issued, not landed: (slot, j)
    next_copy = [0] * consumers       # per consumer warp: next copy it reads
    steps = 0
    while min(next_copy) < total:
        steps += 1
        assert steps < 100000, "no progress"
        acts = []
        if issued < total:
            s = issued % S
            use = issued // S
            if use == 0 or not wait_for_release or empty[s].try_wait_parity((use - 1) & 1):
                acts.append(("issue",))
        if in_flight:
            acts.append(("land",))
        for c in range(consumers):
            j = next_copy[c]
            if j < total and full[j % S].try_wait_parity((j // S) & 1):
                acts.append(("read", c))
        act = rnd.choice(acts)
        if act[0] == "issue":
            s = issued % S
            assert readers_left[s] == 0, "slot refilled while consumers still read it"
            full[s].arrive(expect_tx=1)
            in_flight.append((s, issued))
            issued += 1
        elif act[0] == "land":
            s, j = in_flight.pop(rnd.randrange(len(in_flight)))
            slot_data[s] = j
            readers_left[s] = consumers
            full[s].complete_tx(1)
        else:
            c = act[1]
            j = next_copy[c]
            s = j % S
            assert slot_data[s] == j, f"consumer read copy {slot_data[s]} for copy {j}"
            readers_left[s] -= 1
            empty[s].arrive()
            next_copy[c] += 1


def run_exchange(C, rows, seed, wait_parity=lambda r: (r >> 1) & 1):
    """C CTAs exchange one value per row; deliveries are delayed arbitrarily.
    Checks that a CTA's wait completes only once all C values of that row
    sit in its slots, and that no later row overwrites them first."""
    rnd = random.Random(seed)
    bars = [[MBarrier(1) for _ in range(2)] for _ in range(C)]
    slots = [[[None] * C for _ in range(2)] for _ in range(C)]
    row = [0] * C                     # next row of each CTA
    state = ["send"] * C              # send -> wait -> (read) -> send
    in_flight = []                    # (target, b, sender, row)
    steps = 0
    while min(row) < rows or in_flight:
        steps += 1
        assert steps < 200000, "no progress"
        acts = [("deliver",)] if in_flight else []
        for k in range(C):
            if row[k] >= rows:
                continue
            b = row[k] & 1
            if state[k] == "send":
                acts.append(("send", k))
            elif bars[k][b].try_wait_parity(wait_parity(row[k])):
                acts.append(("read", k))
        act = rnd.choice(acts)
        if act[0] == "send":
            k = act[1]
            b = row[k] & 1
            bars[k][b].arrive(expect_tx=4 * C)
            for t in range(C):
                in_flight.append((t, b, k, row[k]))
            state[k] = "wait"
        elif act[0] == "deliver":
            t, b, k, r = in_flight.pop(rnd.randrange(len(in_flight)))
            assert slots[t][b][k] is None or slots[t][b][k] == r - 2, "a partial overwrote one not yet read"
            slots[t][b][k] = r
            bars[t][b].complete_tx(4)
        else:
            k = act[1]
            b = row[k] & 1
            assert slots[k][b] == [row[k]] * C, f"CTA {k} row {row[k]} saw {slots[k][b]}"
            row[k] += 1
            state[k] = "send"


def test_ring_protocol_under_random_interleavings():
    n = 0
    for S in (2, 3, 6, 9):
        for nt in (1, 3, 6, 9):
            for rows in (1, 2, 5):
                for consumers in (1, 3):
                    for seed in range(4):
                        run_ring(S, nt, rows, consumers, seed)
                        n += 1
    assert n == 4 * 4 * 3 * 2 * 4


def test_cluster_exchange_under_random_interleavings():
    for C in (2, 4, 8):
        for rows in (1, 2, 3, 7):
            for seed in range(25):
                run_exchange(C, rows, seed)


def _fails(fn, seeds):
    for seed in seeds:
        try:
            fn(seed)
        except AssertionError:
            return True
    return False


def test_models_reject_planted_mistakes():
    """Each model fails for a plausible protocol mistake: a producer that
    refills a slot without waiting for its release, and an exchange that waits
    on the row's parity instead of the barrier's use count."""
    assert _fails(lambda seed: run_ring(3, 3, 4, 2, seed, wait_for_release=False), range(50))
    assert _fails(lambda seed: run_exchange(4, 6, seed, wait_parity=lambda r: r & 1), range(50))


def test_parity_wait_is_ambiguous_two_phases_ahead():
    """Why each waiter stays within one phase: a parity wait cannot tell phase
    0 from phase 2.  After phase 0 completes, a wait meant for phase 2 (same
    parity) succeeds at once, while phase 1 is still open."""
    bar = MBarrier(1)
    bar.arrive(expect_tx=1)
    bar.complete_tx(1)                # phase 0 complete
    assert bar.phase == 1
    assert bar.try_wait_parity(0)     # a wait for phase 2 passes now, too early
    assert not bar.try_wait_parity(1)  # the wait for phase 1 correctly blocks
