"""A random-interleaving model of the barrier protocol of the forward kernel
(`fa_fwd_kernel` in exact_attention_93_gb300/csrc/fa_fwd.cu, dense bands).

Test infrastructure: nothing here runs on a GPU, and the kernel does not use
it.  Roles are generators that yield wherever the hardware may switch to
another role: the producer (Q per unit, K and V through a two-stage ring),
the MMA issuer (S_t = Q_t K^T and O_t += P_t V in the kernel's order: for
key tile j, P V of tile A, S_A(j+1), P V of tile B, S_B(j+1)), and the two
softmax warpgroups with their epilogues.  A seeded scheduler picks the next
step among the runnable roles, the tensor-core queue (executed in order) and
the copies in flight (landing in any order).  The model checks that every
parity wait is made within one phase of its barrier, and that the S buffers
(S, then P), the O accumulators, the Q sets, the K / V stages and the O
staging tiles hold what their readers expect and are not overwritten while
a reader still needs them.  The four warps of a softmax group are one role.
`skip` names waits to leave out.
"""
import random

from protocol_sched import Chooser


class ProtocolError(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phases = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending > self.count:
            raise ProtocolError(f"{self.name}: more arrivals than its count")
        if self.pending == self.count:
            self.pending = 0
            self.phases += 1


class Slot:
    """A buffer with what it holds, whether that has landed, and the
    products queued to read it (it may not be overwritten before they run)."""

    def __init__(self):
        self.content, self.landed, self.readers = None, False, 0


class FwdPipeline:
    """units: per unit, the key-tile ranges (lo, hi) of tiles A and B (an
    empty range has lo > hi); resident: several units per CTA (each with its
    own O staging); otherwise one unit, staged in its Q tiles."""

    def __init__(self, units, resident, seed, skip=frozenset(), slow=frozenset()):
        self.rng = random.Random(seed)
        self.chooser = Chooser(self.rng, slow)  # slow: see protocol_sched.Chooser
        self.units, self.res = list(units), resident
        self.nqs = 2 if resident else 1
        self.skip = set(skip)
        B = Barrier
        self.q_full = [B(f"q_full{i}", 1) for i in range(self.nqs)]
        self.q_empty = [B(f"q_empty{i}", 1) for i in range(self.nqs)]
        self.k_full = [B(f"k_full{i}", 1) for i in range(2)]
        self.k_empty = [B(f"k_empty{i}", 1) for i in range(2)]
        self.v_full = [B(f"v_full{i}", 1) for i in range(2)]
        self.v_empty = [B(f"v_empty{i}", 1) for i in range(2)]
        self.s_full = [B(f"s_full{t}", 1) for t in range(2)]
        self.p_full = [B(f"p_full{t}", 1) for t in range(2)]
        self.o_done = [B(f"o_done{t}", 1) for t in range(2)]
        self.drain = B("drain", 1)
        self.queue = []  # tensor-core queue, in order
        self.copies = []
        self.q = [[Slot(), Slot()] for _ in range(self.nqs)]  # Q set, tile
        self.k = [Slot(), Slot()]
        self.v = [Slot(), Slot()]
        self.S = [None, None]   # per tile: ['S', unit, j] or ['P', unit, j, consumed]
        self.O = [None, None]   # per tile: [unit, P V products added, read]
        self.stage = [None, None]  # per tile: [unit, store has read it]
        self.stored = []

    @staticmethod
    def tiles(u, t):
        lo, hi = u[t]
        return list(range(lo, hi + 1)) if lo <= hi else []

    def stream(self, u):
        """Key tiles loaded for a unit: the union of the two ranges."""
        ts = sorted(set(self.tiles(u, 0)) | set(self.tiles(u, 1)))
        if ts and ts != list(range(ts[0], ts[-1] + 1)):
            raise ValueError("the two tiles' key ranges must overlap or touch")
        return ts

    def wait(self, bar, k, name=None):
        if name is not None and name in self.skip:
            return
        while True:
            if (bar.phases & 1) != (k & 1):
                if bar.phases != k + 1:
                    raise ProtocolError(f"wait {bar.name} phase {k} passes at {bar.phases} phases")
                return
            if bar.phases >= k + 2:
                raise ProtocolError(f"wait {bar.name} phase {k} aliased ({bar.phases} phases)")
            self.chooser.blocked()
            yield

    def land(self, slot, content, bar, what):
        def copy():
            if slot.readers:
                raise ProtocolError(f"{what} lands while {slot.readers} products still read {slot.content}")
            slot.content, slot.landed = content, True
            bar.arrive()
        return copy

    # ------------------------------------------------------------ producer
    def producer(self):
        ring = 0
        for k, u in enumerate(self.units):
            qs, use = k % self.nqs, k // self.nqs
            if use > 0:
                yield from self.wait(self.q_empty[qs], use - 1, "prod.q_empty")
            for t in range(2):
                self.q[qs][t].landed = False
            # one transaction for the unit's Q tiles
            slots = [self.q[qs][t] for t in range(2)]

            def land_q(slots=slots, k=k, qs=qs):
                for sl in slots:
                    if sl.readers:
                        raise ProtocolError(f"Q of unit {k} lands while products read {sl.content}")
                    sl.content, sl.landed = k, True
                self.q_full[qs].arrive()
            self.copies.append(land_q)
            yield
            for _ in self.stream(u):
                st, use_st = ring & 1, ring >> 1
                if ring >= 2:
                    yield from self.wait(self.k_empty[st], use_st - 1, "prod.k_empty")
                self.copies.append(self.land(self.k[st], ring, self.k_full[st], f"K({ring})"))
                if ring >= 2:
                    yield from self.wait(self.v_empty[st], use_st - 1, "prod.v_empty")
                self.copies.append(self.land(self.v[st], ring, self.v_full[st], f"V({ring})"))
                ring += 1
                yield

    # ------------------------------------------------------------ MMA issuer
    def mma_issuer(self):
        kv, base = 0, [0, 0]
        for k, u in enumerate(self.units):
            qs, use = k % self.nqs, k // self.nqs
            stream = self.stream(u)
            left = [len(self.tiles(u, 0)) + len(self.tiles(u, 1))]
            yield from self.wait(self.q_full[qs], use, "mma.q_full")
            if not stream:
                if self.res:
                    self.queue.append(("commit", self.q_empty[qs]))
                continue

            def issue_s(t, j, g, qs=qs, k=k):
                st = g & 1
                qslot, kslot = self.q[qs][t], self.k[st]
                qslot.readers += 1
                kslot.readers += 1

                def product():
                    qslot.readers -= 1
                    kslot.readers -= 1
                    if not qslot.landed or qslot.content != k:
                        raise ProtocolError(f"S_{t}({j}) of unit {k} reads Q {qslot.content}")
                    if not kslot.landed or kslot.content != g:
                        raise ProtocolError(f"S_{t}({j}) reads K {kslot.content}, wants ring {g}")
                    old = self.S[t]
                    if old is not None and not (old[0] == "P" and old[3]):
                        raise ProtocolError(f"S_{t}({j}) overwrites {old}")
                    self.S[t] = ["S", k, j]
                self.queue.append(("mma", product))
                self.queue.append(("commit", self.s_full[t]))
                if self.res:
                    left[0] -= 1
                    if left[0] == 0:
                        self.queue.append(("commit", self.q_empty[qs]))

            jf, jl = stream[0], stream[-1]
            yield from self.wait(self.k_full[kv & 1], kv >> 1, "mma.k_full")
            for t in range(2):
                if jf in self.tiles(u, t):
                    issue_s(t, jf, kv)
            self.queue.append(("commit", self.k_empty[kv & 1]))
            for j in range(jf, jl + 1):
                g = kv + (j - jf)
                st = g & 1
                yield from self.wait(self.v_full[st], g >> 1, "mma.v_full")
                k_next = False
                for t in range(2):
                    lo, hi = u[t]
                    active = lo <= j <= hi
                    s_next = (j + 1 <= hi) if active else (j + 1 == lo and lo <= hi)
                    if active:
                        yield from self.wait(self.p_full[t], base[t] + j - lo, "mma.p_full")
                        vslot = self.v[st]
                        vslot.readers += 1

                        def pv(t=t, j=j, g=g, k=k, first=(j == lo), vslot=vslot):
                            vslot.readers -= 1
                            if not vslot.landed or vslot.content != g:
                                raise ProtocolError(f"P V_{t}({j}) reads V {vslot.content}")
                            s = self.S[t]
                            if s is None or s[:3] != ["P", k, j]:
                                raise ProtocolError(f"P V_{t}({j}) of unit {k} reads {s}")
                            s[3] = True
                            if first:
                                if self.O[t] is not None and not self.O[t][2]:
                                    raise ProtocolError(f"P V_{t}({j}) overwrites unread O {self.O[t]}")
                                self.O[t] = [k, 1, False]
                            else:
                                if self.O[t] is None or self.O[t][0] != k:
                                    raise ProtocolError(f"P V_{t}({j}) adds to O {self.O[t]}")
                                self.O[t][1] += 1
                        self.queue.append(("mma", pv))
                        self.queue.append(("commit", self.o_done[t]))
                    if s_next:
                        if not k_next:
                            yield from self.wait(self.k_full[(g + 1) & 1], (g + 1) >> 1, "mma.k_full")
                            k_next = True
                        issue_s(t, j + 1, g + 1)
                    yield
                self.queue.append(("commit", self.v_empty[st]))
                if k_next:
                    self.queue.append(("commit", self.k_empty[(g + 1) & 1]))
            kv += jl - jf + 1
            for t in range(2):
                base[t] += len(self.tiles(u, t))
        self.queue.append(("commit", self.drain))
        yield from self.wait(self.drain, 0)

    # ------------------------------------------------------------ softmax + epilogue
    def softmax(self, t):
        base = 0
        for k, u in enumerate(self.units):
            tiles = self.tiles(u, t)
            for jj, j in enumerate(tiles):
                yield from self.wait(self.s_full[t], base + jj, "sm.s_full")
                s = self.S[t]
                if s is None or s != ["S", k, j]:
                    raise ProtocolError(f"softmax {t} tile {j} of unit {k} reads {s}")
                yield
                if jj > 0 and self.rng.random() < 0.4:  # some row's maximum moved: rescale O
                    yield from self.wait(self.o_done[t], base + jj - 1, "sm.o_done")
                    if self.O[t] is None or self.O[t][:2] != [k, jj]:
                        raise ProtocolError(f"rescale of tile {t} before P V({j - 1}): O {self.O[t]}")
                    yield
                self.S[t] = ["P", k, j, False]
                self.p_full[t].arrive()
                yield
            # epilogue (a tile past the sequence's end, which sees no keys, has none)
            if not tiles:
                continue
            if tiles:
                yield from self.wait(self.o_done[t], base + len(tiles) - 1, "epi.o_done")
                if self.O[t] is None or self.O[t][:2] != [k, len(tiles)]:
                    raise ProtocolError(f"epilogue of tile {t}, unit {k} reads O {self.O[t]}")
            if self.res:
                cur = self.stage[t]
                if cur is not None and not cur[1]:
                    raise ProtocolError(f"epilogue of unit {k} stages over unit {cur[0]}")
            else:  # staged in its Q tile, no longer read
                qslot = self.q[0][t]
                if qslot.readers:
                    raise ProtocolError(f"epilogue stages over Q tile {t} still read")
            if tiles:
                self.O[t][2] = True
            self.stage[t] = [k, False]
            yield
            done = [False]

            def store(t=t, k=k, done=done):
                if self.stage[t] != [k, False]:
                    raise ProtocolError(f"store of tile {t}, unit {k} reads stage {self.stage[t]}")
                self.stage[t][1] = True
                self.stored.append((k, t))
                done[0] = True
            self.copies.append(store)
            while not done[0]:  # one thread waits for the store before the stage is reused
                yield
            base += len(tiles)

    # ------------------------------------------------------------ scheduler
    def run(self, max_steps=400000):
        roles = {"producer": self.producer(), "mma": self.mma_issuer(),
                 "softmax A": self.softmax(0), "softmax B": self.softmax(1)}
        steps = 0
        while roles or self.queue or self.copies:
            steps += 1
            if steps > max_steps:
                raise ProtocolError("no progress: " + ", ".join(roles))
            choices = list(roles) + (["queue"] if self.queue else []) + (["copy"] if self.copies else [])
            if not choices:
                raise ProtocolError("deadlock: nothing can run")
            c = self.chooser.pick(choices, steps)
            if c == "queue":
                kind, x = self.queue.pop(0)
                x() if kind == "mma" else x.arrive()
            elif c == "copy":
                self.copies.pop(self.rng.randrange(len(self.copies)))()
            else:
                self.chooser.enter(c, steps)
                try:
                    next(roles[c])
                except StopIteration:
                    del roles[c]
        want = sorted((k, t) for k, u in enumerate(self.units) for t in range(2) if self.tiles(u, t))
        if sorted(self.stored) != want:
            raise ProtocolError(f"tiles stored: {sorted(self.stored)}")


def band_range(q0, wl, wr, n, tile=128):
    """Key tiles a 128-row query tile at q0 sees (wl, wr < 0: unbounded)."""
    n_kv = (n + tile - 1) // tile
    first = 0 if wl < 0 else max(0, q0 - wl)
    last = min(n - 1, n - 1 if wr < 0 else q0 + tile - 1 + wr)
    return (first // tile, min(n_kv - 1, last // tile))


def units_for(n, wl, wr, heads):
    """The units of a launch in the kernel's order: pairs of query tiles,
    later pairs first when keys are bounded on the right only (causal)."""
    n_q = (n + 127) // 128
    pairs = (n_q + 1) // 2
    later_first = wl < 0 and wr >= 0
    out = []
    for _ in range(heads):
        for idx in range(pairs):
            pt = pairs - 1 - idx if later_first else idx
            u = []
            for t in range(2):
                qt = 2 * pt + t
                u.append((1, 0) if qt >= n_q else band_range(qt * 128, wl, wr, n))
            out.append(tuple(u))
    return out


# (N, window left, window right): causal, non-causal, bands and ragged sizes
BANDS = [(300, -1, 64), (300, 32, 16), (300, 0, 0), (300, 127, -1), (300, -1, -1),
         (1000, -1, 0), (1024, -1, 0), (17, -1, -1), (640, 200, 300), (129, -1, 0),
         (512, -1, -1), (2048, -1, 0), (700, 5, 400)]
