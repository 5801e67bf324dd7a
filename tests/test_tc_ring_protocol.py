"""Host model of the tcgen05 decode-GEMM's ring protocol (kernels_tc.cu).

The kernel's correctness rests on mbarrier phase parity: a wait names a
phase only by its parity, so no waiter may fall two phases behind a
barrier.  This model runs the kernel's five roles -- weight producer, token
producer, UMMA thread, two decoder groups (a group's 8 warp arrivals are
one arrival here) -- against barriers with the hardware's parity semantics
(try_wait.parity(P) is true iff the current phase's parity differs from P),
with fills landing and UMMAs completing after random delays under random
scheduling.  It asserts, for every pair of ring sizes the kernel builds
(weight stages SW, token slots SX):
  - every role finishes (no deadlock);
  - a decoder reads a landed fill of its own unit, never a stale or
    in-flight one;
  - UMMAs read the unit's tokens and A buffer, unchanged until they
    complete, and the decoders never overwrite an A buffer under them;
  - the accumulator is read only after its piece's UMMAs completed and is
    not reset before both decoder groups read it.
A negative control runs the earlier scheme (one full barrier per slot and a
group waiting on the other group's fills), which the model must catch.
"""
import random


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0
        self._maybe_complete()

    def expect_tx(self, b):
        self.tx += b
        self.arrive()

    def complete_tx(self, b):
        self.tx -= b
        assert self.tx >= 0
        self._maybe_complete()

    def test(self, parity):
        return (self.phase & 1) != parity


def gp(i, S, per_group):
    if not per_group:
        return (i // S) & 1
    k = i // S
    return ((k >> 1) if (S & 1) else k) & 1


def run(SW, SX, n_units, KG, u0_off, seed, per_group=True, skip_wait=False, issuers=1):
    rnd = random.Random(seed)
    U = n_units
    # pieces: tiles of KG units, CTA range starts at offset u0_off inside a tile
    piece_of = [(u0_off + i) // KG for i in range(U)]
    last_of_piece = [i == U - 1 or piece_of[i + 1] != piece_of[i] for i in range(U)]
    first_of_piece = [i == 0 or piece_of[i - 1] != piece_of[i] for i in range(U)]
    nfull = 2 if per_group else 1
    full_w = [Bar(1) for _ in range(nfull * SW)]
    full_x = [Bar(1) for _ in range(nfull * SX)]
    empty_w = [Bar(1) for _ in range(SW)]
    empty_x = [Bar(1) for _ in range(SX)]
    a_full = [Bar(1) for _ in range((2 if issuers == 2 else 1) * SX)]
    acc_full, acc_empty = Bar(issuers), Bar(2)
    wstage = [None] * SW  # content: ('fly', i) or ('ok', i)
    xslot = [None] * SX
    abuf = [None] * SX
    abuf_busy = [0] * SX  # in-flight UMMAs reading it
    events = []  # (time, seq, fn)
    now = [0]
    seq = [0]
    piece_pending = {}
    epi_done = set()

    def sched(delay, fn):
        seq[0] += 1
        events.append((now[0] + delay, seq[0], fn))

    def fbar(arr, S, i):
        return arr[(2 * (i % S) + (i & 1)) if per_group else (i % S)]

    def WP():
        for i in range(U):
            s = i % SW
            if i >= SW:
                yield (empty_w[s], ((i // SW) - 1) & 1)
            assert wstage[s] is None or wstage[s][0] == 'read', ('WP overwrite', i, wstage[s])
            b = fbar(full_w, SW, i)
            b.expect_tx(1)
            wstage[s] = ('fly', i)

            def land(s=s, i=i, b=b):
                wstage[s] = ('ok', i)
                b.complete_tx(1)
            sched(rnd.randint(1, 40), land)

    def XP():
        for i in range(U):
            s = i % SX
            if i >= SX:
                yield (empty_x[s], ((i // SX) - 1) & 1)
            assert abuf_busy[s] == 0
            b = fbar(full_x, SX, i)
            b.expect_tx(1)
            xslot[s] = ('fly', i)

            def land(s=s, i=i, b=b):
                xslot[s] = ('ok', i)
                b.complete_tx(1)
            sched(rnd.randint(1, 25), land)

    def abar(i):
        return a_full[2 * (i % SX) + (i & 1)] if issuers == 2 else a_full[i % SX]

    def apar(i):
        return gp(i, SX, True) if issuers == 2 else (i // SX) & 1

    last_done = [0, 0]  # per issuer: its UMMAs complete in issue order

    def MMA(t):
        """UMMA issuer t: every unit (issuers == 1) or the units of parity t."""
        piece = -1
        for i in range(U):
            if first_of_piece[i]:
                piece += 1
                if piece > 0:
                    yield (acc_empty, (piece - 1) & 1)
                assert (piece - 1) in epi_done or piece == 0
            mine = issuers == 1 or (i & 1) == t
            if mine:
                sx = i % SX
                yield (abar(i), apar(i))
                assert xslot[sx] == ('ok', i), ('MMA x', i, xslot[sx])
                assert abuf[sx] == i, ('MMA A', i, abuf[sx])
                abuf_busy[sx] += 1
                piece_pending[piece] = piece_pending.get(piece, 0) + 1

                def done(sx=sx, i=i, p=piece):
                    assert xslot[sx] == ('ok', i) and abuf[sx] == i, ('UMMA operands changed', i)
                    abuf_busy[sx] -= 1
                    piece_pending[p] -= 1
                    empty_x[sx].arrive()
                # one issuer's UMMAs complete in issue order; the two
                # issuers' interleave in any order
                t_done = max(now[0] + rnd.randint(1, 30), last_done[t] + 1)
                last_done[t] = t_done
                seq[0] += 1
                events.append((t_done, seq[0], done))
            if last_of_piece[i]:
                # the commit arrives once this issuer's UMMAs so far completed
                t_done = max(now[0], last_done[t]) + 1
                seq[0] += 1
                events.append((t_done, seq[0], lambda: acc_full.arrive()))

    def DEC(grp):
        piece = 0
        for i in range(U):
            if (i & 1) == grp:
                s, sx = i % SW, i % SX
                yield (fbar(full_w, SW, i), gp(i, SW, per_group))
                assert wstage[s] == ('ok', i), ('DEC read', grp, i, wstage[s])
                wstage[s] = ('read', i)
                empty_w[s].arrive()
                yield ('delay', rnd.randint(1, 30))
                yield (fbar(full_x, SX, i), gp(i, SX, per_group))
                assert abuf_busy[sx] == 0, ('A overwrite under UMMA', i)
                assert xslot[sx] == ('ok', i), ('DEC x', i, xslot[sx])
                abuf[sx] = i
                abar(i).arrive()
            elif skip_wait:
                s, sx = i % SW, i % SX
                if SW & 1:
                    yield (full_w[s], (i // SW) & 1)
                if SX & 1:
                    yield (full_x[sx], (i // SX) & 1)
            if last_of_piece[i]:
                yield (acc_full, piece & 1)
                assert piece_pending.get(piece, 0) == 0, ('acc read early', piece)
                DEC.reads[piece] = DEC.reads.get(piece, 0) + 1
                if DEC.reads[piece] == 2:
                    epi_done.add(piece)
                acc_empty.arrive()
                piece += 1
    DEC.reads = {}

    actors = {'WP': WP(), 'XP': XP(), 'D0': DEC(0), 'D1': DEC(1)}
    for t in range(issuers):
        actors[f'MMA{t}'] = MMA(t)
    waiting = {k: None for k in actors}
    sleeping = {}
    done = set()
    steps = 0
    while len(done) < len(actors):
        steps += 1
        if steps > 2_000_000:
            raise RuntimeError('livelock')
        runnable = []
        for k, g in actors.items():
            if k in done or k in sleeping:
                continue
            w = waiting[k]
            if w is None or w[0].test(w[1]):
                runnable.append(k)
        if runnable and (not events or rnd.random() < 0.7):
            k = rnd.choice(runnable)
            try:
                w = next(actors[k])
                if w[0] == 'delay':
                    sleeping[k] = now[0] + w[1]
                    waiting[k] = None
                else:
                    waiting[k] = w
            except StopIteration:
                done.add(k)
            continue
        # advance time
        wake = [t for t in sleeping.values()]
        cand = [e[0] for e in events] + wake
        if not cand:
            blocked = {k: (waiting[k][1], waiting[k][0].phase) for k in actors if k not in done}
            raise RuntimeError(f'deadlock: {blocked}')
        t = min(cand)
        now[0] = t
        for k in [k for k, tt in sleeping.items() if tt <= t]:
            del sleeping[k]
        evs = sorted([e for e in events if e[0] <= t])
        for e in evs:
            events.remove(e)
            e[2]()
    return True


# ring sizes of tc_kernel<MP>: (SW, SX) for MP = 16, 32, 64, 128 (plain:
# 4 / 4, fused: 5 / 3), and neighbours (odd and even rings, tiny rings)
CONFIGS = [(8, 4), (7, 4), (6, 4), (4, 4), (5, 3), (3, 3), (4, 2), (2, 2), (5, 4), (7, 3)]


def _cases(seeds):
    for SW, SX in CONFIGS:
        for seed in range(seeds):
            rnd = random.Random(seed)
            n = rnd.randint(1, 60)
            KG = rnd.choice([1, 2, 3, 5, 40])
            yield SW, SX, n, KG, rnd.randint(0, KG - 1), seed


def test_ring_protocol_per_group_barriers():
    for SW, SX, n, KG, off, seed in _cases(40):
        assert run(SW, SX, n, KG, off, seed, per_group=True, skip_wait=False), (SW, SX, seed)


def test_ring_protocol_two_issuers():
    """Two UMMA issuers (even and odd units, one accumulator each), a_full
    per decoder group and slot, acc_full with two arrivals."""
    for SW, SX, n, KG, off, seed in _cases(40):
        assert run(SW, SX, n, KG, off, seed, per_group=True, skip_wait=False, issuers=2), (SW, SX, seed)


def test_model_catches_the_skip_wait_deadlock():
    failures = 0
    for SW, SX, n, KG, off, seed in _cases(10):
        if (SW & 1) == 0 and (SX & 1) == 0:
            continue
        try:
            run(SW, SX, n, KG, off, seed, per_group=False, skip_wait=True)
        except (AssertionError, RuntimeError):
            failures += 1
    assert failures > 0
