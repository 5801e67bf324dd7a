"""Host model of the tcgen05 decode-GEMM's ring protocol (kernels_tc.cu).

The kernel's correctness rests on mbarrier phase parity: a wait names a
phase only by its parity, so no waiter may fall two phases behind a
barrier.  This model runs the kernel's six roles -- weight producer, token
producer, two UMMA issuers, two decoder groups (a group's 8 warp arrivals
are one arrival here) -- against barriers with the hardware's parity
semantics (try_wait.parity(P) is true iff the current phase's parity differs
from P), with copies landing and UMMAs completing after random delays under
random scheduling.  Units are in the kernel's pair order: a pair of tiles
covers 2 KG units (k-group kg of tile j is unit 2 kg + j of the pair), an odd
tile count is padded by a phantom tile (its units copy and multiply
nothing), and a CTA's range [u0, u1) may start and end anywhere.  For every
combination of ring sizes the kernel builds (weight stages per group SWG,
token slots SX, A buffers per group NA) it asserts:
  - every role finishes (no deadlock);
  - a decoder reads a landed copy of its own unit, never a stale or
    in-flight one, and a weight stage is refilled only after its group read it;
  - UMMAs read their step's tokens and their unit's A buffer, both unchanged
    until they complete: the token producer never refills a slot and the
    decoders never overwrite an A buffer under them;
  - an accumulator is read only after its piece's UMMAs completed and is not
    reset before its decoder group read it.
A negative control gives the token slots' empty barrier one arrival (only
one issuer's commit) instead of two; the model must catch the refill under
the other issuer's UMMAs.
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


def run(SWG, SX, NA, u0, u1, KG, NB, seed, empty_x_count=2):
    """One CTA over units [u0, u1) of a product with KG groups and NB real
    tiles (pair order, phantom tile if NB is odd)."""
    rnd = random.Random(seed)
    NBP = NB + (NB & 1)
    assert 0 <= u0 < u1 <= KG * NBP

    def tile(u):
        return 2 * (u // (2 * KG)) + (u & 1)

    def kg_of(u):
        return (u % (2 * KG)) >> 1

    def phantom(u):
        return tile(u) >= NB

    def first_of_piece(u):
        return kg_of(u) == 0 or u - 2 < u0

    def last_of_piece(u):
        return kg_of(u) == KG - 1 or u + 2 >= u1

    full_w = [[Bar(1) for _ in range(SWG)] for _ in range(2)]
    empty_w = [[Bar(1) for _ in range(SWG)] for _ in range(2)]
    full_x = [Bar(1) for _ in range(SX)]
    empty_x = [Bar(empty_x_count) for _ in range(SX)]
    a_full = [[Bar(1) for _ in range(NA)] for _ in range(2)]
    a_empty = [[Bar(1) for _ in range(NA)] for _ in range(2)]
    acc_full = [Bar(1), Bar(1)]
    acc_empty = [Bar(1), Bar(1)]
    wstage = [[None] * SWG for _ in range(2)]  # ('fly', u) / ('ok', u) / ('read', u)
    xslot = [None] * SX                          # ('fly', step) / ('ok', step)
    xbusy = [0] * SX                             # UMMAs in flight reading the slot
    abuf = [[None] * NA for _ in range(2)]
    abusy = [[0] * NA for _ in range(2)]
    pending = [{}, {}]                           # per issuer: piece -> UMMAs in flight
    events = []
    now = [0]
    seq = [0]
    last_done = [0, 0]

    def sched_at(t, fn):
        seq[0] += 1
        events.append((t, seq[0], fn))

    s0, s1 = u0 >> 1, (u1 - 1) >> 1
    nsteps = s1 - s0 + 1

    def WP():
        issued = [0, 0]
        for u in range(u0, u1):
            j = u & 1
            k = issued[j]
            s = k % SWG
            if k >= SWG:
                yield (empty_w[j][s], ((k // SWG) - 1) & 1)
            assert wstage[j][s] is None or wstage[j][s][0] == 'read', ('WP overwrite', u, wstage[j][s])
            b = full_w[j][s]
            if phantom(u):
                wstage[j][s] = ('ok', u)
                b.arrive()
            else:
                b.expect_tx(1)
                wstage[j][s] = ('fly', u)

                def land(j=j, s=s, u=u, b=b):
                    wstage[j][s] = ('ok', u)
                    b.complete_tx(1)
                sched_at(now[0] + rnd.randint(1, 40), land)
            issued[j] += 1

    def XP():
        for t in range(nsteps):
            s = t % SX
            if t >= SX:
                yield (empty_x[s], ((t // SX) - 1) & 1)
            assert xbusy[s] == 0, ('token slot refilled under a UMMA', t)
            full_x[s].expect_tx(1)
            xslot[s] = ('fly', s0 + t)

            def land(s=s, st=s0 + t):
                xslot[s] = ('ok', st)
                full_x[s].complete_tx(1)
            sched_at(now[0] + rnd.randint(1, 25), land)

    def commit(j, fn):
        # a commit arrives once every UMMA this issuer issued before it completed
        sched_at(max(now[0], last_done[j]) + 1, fn)

    def MMA(j):
        pieces = 0
        uses = 0
        for t in range(nsteps):
            st = s0 + t
            u = 2 * st + j
            xs = t % SX
            yield (full_x[xs], (t // SX) & 1)
            if u0 <= u < u1:
                if first_of_piece(u) and pieces > 0:
                    yield (acc_empty[j], (pieces - 1) & 1)
                a = uses % NA
                yield (a_full[j][a], (uses // NA) & 1)
                assert xslot[xs] == ('ok', st), ('MMA tokens', u, xslot[xs])
                assert abuf[j][a] == u, ('MMA A', u, abuf[j][a])
                if not phantom(u):
                    xbusy[xs] += 1
                    abusy[j][a] += 1
                    pending[j][pieces] = pending[j].get(pieces, 0) + 1

                    def done(xs=xs, a=a, st=st, u=u, p=pieces):
                        assert xslot[xs] == ('ok', st) and abuf[j][a] == u, ('UMMA operands changed', u)
                        xbusy[xs] -= 1
                        abusy[j][a] -= 1
                        pending[j][p] -= 1
                    t_done = max(now[0] + rnd.randint(1, 30), last_done[j] + 1)
                    last_done[j] = t_done
                    sched_at(t_done, done)
                commit(j, lambda j=j, a=a: a_empty[j][a].arrive())
                uses += 1
                if last_of_piece(u):
                    commit(j, lambda j=j: acc_full[j].arrive())
                    pieces += 1
            commit(j, lambda xs=xs: empty_x[xs].arrive())

    def DEC(j):
        ws = 0
        wph = 0
        uses = 0
        pieces = 0
        u = u0 if (u0 & 1) == j else u0 + 1
        while u < u1:
            yield (full_w[j][ws], wph)
            assert wstage[j][ws] == ('ok', u), ('DEC read', j, u, wstage[j][ws])
            wstage[j][ws] = ('read', u)
            empty_w[j][ws].arrive()
            ws += 1
            if ws == SWG:
                ws, wph = 0, wph ^ 1
            yield ('delay', rnd.randint(1, 30))
            a = uses % NA
            if uses >= NA:
                yield (a_empty[j][a], ((uses // NA) - 1) & 1)
            assert abusy[j][a] == 0, ('A overwrite under UMMA', u)
            abuf[j][a] = u
            a_full[j][a].arrive()
            uses += 1
            if last_of_piece(u):
                yield (acc_full[j], pieces & 1)
                assert pending[j].get(pieces, 0) == 0, ('accumulator read early', j, pieces)
                yield ('delay', rnd.randint(1, 20))
                acc_empty[j].arrive()
                pieces += 1
            u += 2

    actors = {'WP': WP(), 'XP': XP(), 'D0': DEC(0), 'D1': DEC(1), 'M0': MMA(0), 'M1': MMA(1)}
    waiting = {k: None for k in actors}
    sleeping = {}
    done = set()
    steps = 0
    while len(done) < len(actors):
        steps += 1
        if steps > 2_000_000:
            raise RuntimeError('livelock')
        runnable = []
        for k in actors:
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
        cand = [e[0] for e in events] + list(sleeping.values())
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


# ring sizes of tc_kernel<MP> (SWG, SX, NA) for MP = 16, 32, 64, 128, and
# smaller or odd neighbours
CONFIGS = [(4, 4, 3), (4, 3, 3), (3, 4, 3), (3, 2, 2), (2, 2, 2), (2, 3, 2), (3, 1, 2), (2, 5, 4)]


def _cases(seeds):
    for SWG, SX, NA in CONFIGS:
        for seed in range(seeds):
            rnd = random.Random(1000 * SWG + 100 * SX + 10 * NA + seed)
            KG = rnd.choice([1, 2, 3, 5, 8, 40])
            NB = rnd.choice([1, 2, 3, 4, 5, 7])
            U = KG * (NB + (NB & 1))
            # ranges long enough to turn every ring over several times, and
            # a few short ones
            n = min(U, rnd.randint(1, 8)) if rnd.random() < 0.2 else rnd.randint(min(U, 16), min(U, 120))
            u0 = rnd.randint(0, U - n)
            u1 = u0 + n
            yield SWG, SX, NA, u0, u1, KG, NB, seed


def test_ring_protocol_pair_order():
    for case in _cases(40):
        assert run(*case), case


def test_ring_protocol_whole_product_from_unit_zero():
    """A CTA that holds a whole product (every pair, both tiles)."""
    for SWG, SX, NA in CONFIGS:
        for NB in (1, 2, 3, 6):
            for seed in range(4):
                KG = 3
                assert run(SWG, SX, NA, 0, KG * (NB + (NB & 1)), KG, NB, seed)


def test_model_catches_a_single_commit_token_slot():
    failures = 0
    for case in _cases(12):
        try:
            run(*case, empty_x_count=1)
        except (AssertionError, RuntimeError):
            failures += 1
    assert failures > 0
