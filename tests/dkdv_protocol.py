"""A random-interleaving model of the barrier protocol of the dK/dV kernel
(`bwd_dkdv_pipe_kernel` in exact_attention_93_gb300/csrc/fa_bwd.cu).

Test infrastructure: nothing here runs on a GPU, and the kernel does not use
it.  Each role of the kernel is a generator that yields at every point where
the hardware may switch to another role; a seeded scheduler picks the next
step among the runnable roles, the two tensor-core issue queues (each
executed in order) and the asynchronous copies in flight (landing in any
order).  The model checks that

  - every parity wait is made within one phase of its barrier (a wait that
    would pass on a later phase, or one phase too early, is an error), and
  - every shared resource holds what its reader expects when it is read and
    is not overwritten while a reader still needs it: the TMEM buffers
    (S^T, then dQ^T; dP^T, then P^T / dS^T), the dV / dK accumulators, the
    Q / dO stages, the K / V buffers, the three dS^T tiles (also the staging
    of a resident CTA's dK, dV), and the two dQ stages of the bulk
    reductions at D = 64.

The eight elementwise warps are modelled as one role (they do the same
steps on the same tiles); the four buffer warps separately (each drains its
own TMEM lanes).  `skip` names waits to leave out, so that the tests can
show that each one is needed.
"""
import random

from protocol_sched import Chooser


class ProtocolError(Exception):
    pass


class Barrier:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phases = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending > self.count:
            raise ProtocolError(f"{self.name}: more arrivals than its count")
        if self.pending == self.count:
            self.pending = 0
            self.phases += 1


class DkdvPipeline:
    """units: tiles per unit (a one-unit CTA has one); buffers: S^T / dP^T
    buffers (3 at D = 64, 2 at D = 128); resident: several units per CTA
    (D = 64 only); atomic_dq: dQ^T products and their drain."""

    def __init__(self, units, buffers, resident, atomic_dq, d64, seed, skip=frozenset(),
                 independent_signal=False, slow=frozenset()):
        self.rng = random.Random(seed)
        # slow: see protocol_sched.Chooser (roles, or the queues "q_score",
        # "q_grad", "copy")
        self.chooser = Chooser(self.rng, slow)
        # independent_signal: epi_read signalled by its own role as soon as
        # the store has read its staging, instead of by thread 0 just before
        # the first wait on it (every arrival time the kernel can produce,
        # and more: the elementwise role stands for all eight warps, so with
        # the inline signal its own waits on epi_read are always satisfied)
        self.independent_signal = independent_signal
        self.units, self.nb, self.res, self.atomic, self.d64 = list(units), buffers, resident, atomic_dq, d64
        self.nqs = buffers + 1               # Q / dO stages
        self.nkv = 2 if resident else 1      # K / V buffers
        self.skip = set(skip)
        B = Barrier
        self.kv_full = [B(f"kv_full{i}", 1) for i in range(self.nkv)]
        self.kv_empty = [B(f"kv_empty{i}", 1) for i in range(self.nkv)]
        self.qdo_full = [B(f"qdo_full{i}", 1) for i in range(self.nqs)]
        self.qdo_empty = [B(f"qdo_empty{i}", 1) for i in range(self.nqs)]
        self.s_full = [B(f"s_full{i}", 1) for i in range(self.nb)]
        self.s_read = [B(f"s_read{i}", 1) for i in range(self.nb)]
        self.p_full = [B(f"p_full{i}", 1) for i in range(self.nb)]
        # four buffer warps and the commit of dV, dK(gi - buffers)
        self.buf_ready = [B(f"buf_ready{i}", 5) for i in range(self.nb)]
        self.tmem_free = [B(f"tmem_free{i}", 4) for i in range(self.nb)]
        self.dq_full = [B(f"dq_full{i}", 1) for i in range(3)]
        self.stage_full = [B(f"stage_full{i}", 2) for i in range(2)]
        self.stage_free = [B(f"stage_free{i}", 1) for i in range(2)]
        self.ds_last, self.acc_full, self.epi_read = B("ds_last", 1), B("acc_full", 1), B("epi_read", 1)
        self.last_issued = B("last_issued", 1)  # resident: a unit's last dV, dK issued
        self.drain = [B("drain0", 1), B("drain1", 1)]
        self.q_score, self.q_grad = [], []  # tensor-core issue queues, each in order
        self.copies = []                    # asynchronous copies in flight (any order)
        self.after_read = []                # (group, completion) of bulk stores / reductions
        self.groups = {"epilogue": [], "reduce": []}  # per issuing thread: [read, complete]
        self.spawned = []
        # resources
        self.S = [None] * self.nb     # ['S', gi, read] or ['dQ', j, drained]
        self.P = [None] * self.nb     # ['dP', gi] or ['PdS', gi, consumed]
        self.acc = None               # [unit, tiles added, read]
        self.stage = [None] * self.nqs  # (gi, landed)
        self.kv = [None] * self.nkv     # (unit, landed)
        self.dst = [None] * 3         # ['dS', j, consumed] or ['staging', unit, read]
        self.dq_stage = [None] * 2    # [j, read]
        self.total = sum(self.units)
        self.tile_unit = [k for k, n in enumerate(self.units) for _ in range(n)]
        self.drained_by = {}
        self.reduced, self.stored = [], []

    # ------------------------------------------------------------ helpers
    def wait(self, bar, k, name=None):
        """Wait for phase k of bar (the kernel passes parity k & 1)."""
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

    # ------------------------------------------------------------ producer
    def producer(self):
        gi = 0
        for k, n in enumerate(self.units):
            kvb = k % self.nkv
            if k >= self.nkv:
                yield from self.wait(self.kv_empty[kvb], (k - self.nkv) // self.nkv, "prod.kv_empty")
            self.kv[kvb] = (k, False)

            def land_kv(kvb=kvb, k=k):
                if self.kv[kvb] != (k, False):
                    raise ProtocolError(f"K/V of unit {k} lands over {self.kv[kvb]}")
                self.kv[kvb] = (k, True)
                self.kv_full[kvb].arrive()
            self.copies.append(land_kv)
            yield
            for _ in range(n):
                st = gi % self.nqs
                if gi >= self.nqs:
                    yield from self.wait(self.qdo_empty[st], (gi - self.nqs) // self.nqs, "prod.qdo_empty")
                if self.atomic and gi == self.nb:
                    # buffer 0's first phase complete before the tile that
                    # reuses it lands: the buffer warps' wait for that tile
                    # then implies it (later tiles' drains do)
                    yield from self.wait(self.buf_ready[0], 0, "prod.buf_ready")
                self.stage[st] = (gi, False)

                def land_q(st=st, gi=gi):
                    if self.stage[st] != (gi, False):
                        raise ProtocolError(f"Q / dO of tile {gi} lands over {self.stage[st]}")
                    self.stage[st] = (gi, True)
                    self.qdo_full[st].arrive()
                self.copies.append(land_q)
                gi += 1
                yield

    # ------------------------------------------------------------ score products
    def score_issuer(self):
        gi = 0
        for k, n in enumerate(self.units):
            kvb = k % self.nkv
            yield from self.wait(self.kv_full[kvb], k // self.nkv, "score.kv_full")
            for i in range(n):
                b, st = gi % self.nb, gi % self.nqs
                if self.res and i == 0 and k > 0:
                    yield from self.wait(self.last_issued, k - 1, "score.last_issued")
                yield from self.wait(self.buf_ready[b], gi // self.nb, "score.buf_ready")

                def products(b=b, st=st, gi=gi, kvb=kvb, k=k):
                    if self.kv[kvb] != (k, True):
                        raise ProtocolError(f"S({gi}) reads K / V {self.kv[kvb]}, wants unit {k}")
                    if self.stage[st] != (gi, True):
                        raise ProtocolError(f"S({gi}) reads Q stage {self.stage[st]}")
                    old = self.S[b]
                    if old is not None and not old[2]:
                        raise ProtocolError(f"S({gi}) overwrites {old[0]}({old[1]}) still in use")
                    oldp = self.P[b]
                    if oldp is not None and not (oldp[0] == "PdS" and oldp[2]):
                        raise ProtocolError(f"dP({gi}) overwrites {oldp}")
                    self.S[b] = ["S", gi, False]
                    self.P[b] = ["dP", gi]
                self.q_score.append(("mma", products))
                self.q_score.append(("commit", self.s_full[b]))
                gi += 1
                yield
        self.q_score.append(("commit", self.drain[0]))
        yield from self.wait(self.drain[0], 0)

    # ------------------------------------------------------------ gradient products
    def gradient_issuer(self):
        gi, kvb_prev, prev_last = 0, 0, False

        def issue_dq(j, kvb):
            def product(j=j, kvb=kvb):
                k = self.tile_unit[j]
                if self.kv[kvb] != (k, True):
                    raise ProtocolError(f"dQ({j}) reads K {self.kv[kvb]}, wants unit {k}")
                t = self.dst[j % 3]
                if t is None or t[:2] != ["dS", j]:
                    raise ProtocolError(f"dQ({j}) reads dS^T tile {t}")
                t[2] = True
                b = (j + 1) % self.nb
                old = self.S[b]
                if old is not None and not old[2]:
                    raise ProtocolError(f"dQ({j}) into buffer {b} holding {old}")
                self.S[b] = ["dQ", j, False]
            self.q_grad.append(("mma", product))
            self.q_grad.append(("commit", self.dq_full[j % 3]))

        for k, n in enumerate(self.units):
            kvb = k % self.nkv
            for i in range(n):
                b, st = gi % self.nb, gi % self.nqs
                if self.atomic and gi >= 1:
                    yield from self.wait(self.s_read[b], gi // self.nb, "grad.s_read")
                    issue_dq(gi - 1, kvb_prev)
                    if self.res and prev_last:
                        self.q_grad.append(("commit", self.kv_empty[kvb_prev]))
                yield from self.wait(self.p_full[b], gi // self.nb, "grad.p_full")

                def products(b=b, st=st, gi=gi, k=k, first=(i == 0)):
                    p = self.P[b]
                    if p is None or p[:2] != ["PdS", gi]:
                        raise ProtocolError(f"dV, dK({gi}) read {p}")
                    if self.stage[st] != (gi, True):
                        raise ProtocolError(f"dV, dK({gi}) read Q stage {self.stage[st]}")
                    p[2] = True
                    if first:
                        if self.acc is not None and not self.acc[2]:
                            raise ProtocolError(f"dV, dK({gi}) overwrite unread accumulators {self.acc}")
                        self.acc = [k, 1, False]
                    else:
                        if self.acc[0] != k:
                            raise ProtocolError(f"dV, dK({gi}) add to accumulators of unit {self.acc[0]}")
                        self.acc[1] += 1
                self.q_grad.append(("mma", products))
                self.q_grad.append(("commit", self.qdo_empty[st]))
                self.q_grad.append(("commit", self.buf_ready[b]))
                if self.res and i == n - 1:
                    self.last_issued.arrive()
                kvb_prev, prev_last = kvb, i == n - 1
                gi += 1
                yield
            self.q_grad.append(("commit", self.acc_full))
            if self.res and not self.atomic:
                self.q_grad.append(("commit", self.kv_empty[kvb]))
        if self.atomic and gi > 0:
            j = gi - 1
            yield from self.wait(self.ds_last, 0, "grad.ds_last")
            if j >= self.nb:
                yield from self.wait(self.tmem_free[(j + 1) % self.nb], (j - self.nb) // self.nb,
                                     "grad.tmem_free")
            issue_dq(j, kvb_prev)
        self.q_grad.append(("commit", self.drain[1]))
        yield from self.wait(self.drain[1], 0)

    # ------------------------------------------------------------ buffer / dQ warps
    def buffer_warp(self, w):
        quad = w - 8

        def drain_load(j, b):
            yield from self.wait(self.dq_full[j % 3], j // 3, "buf.dq_full")
            old = self.S[b]
            if old is None or old[:2] != ["dQ", j]:
                raise ProtocolError(f"drain of dQ({j}) by warp {w} finds {old}")
            self.drained_by.setdefault(j, set()).add(w)
            if len(self.drained_by[j]) == 4:
                old[2] = True
            self.tmem_free[b].arrive()

        def drain_add(j):
            if not self.d64:  # atomics straight from registers
                if quad == 0:
                    self.reduced.append(j)
                return
            sb = j & 1
            if quad < 2:  # stage the rows d < 64
                if j >= 2:
                    yield from self.wait(self.stage_free[sb], (j >> 1) - 1, "buf.stage_free")
                cur = self.dq_stage[sb]
                if cur is not None and cur[0] != j and not cur[1]:
                    raise ProtocolError(f"dQ stage {sb} for tile {j} holds unread tile {cur[0]}")
                self.dq_stage[sb] = [j, False]
                self.stage_full[sb].arrive()
            elif quad == 2:  # issue the bulk reduction
                yield from self.wait(self.stage_full[sb], j >> 1, "buf.stage_full")
                group = [False, False, sb, j]
                self.groups["reduce"].append(group)

                def read(group=group):
                    if self.dq_stage[group[2]][0] != group[3]:
                        raise ProtocolError(f"reduction of tile {group[3]} reads stage {self.dq_stage[group[2]]}")
                    group[0] = True
                    self.dq_stage[group[2]][1] = True

                def complete(group=group):
                    group[1] = True
                    self.reduced.append(group[3])
                self.copies.append(read)
                self.after_read.append((group, complete))
                while not all(g[0] for g in self.groups["reduce"][:-1]):  # all but the newest read
                    yield
                if j >= 1:
                    self.stage_free[(j - 1) & 1].arrive()

        # one loop, as in the kernel: the drains run buffers + 1 tiles behind
        for gi in range(self.total + (self.nb + 1 if self.atomic else 0)):
            b, j = gi % self.nb, gi - 1 - self.nb
            drain = self.atomic and 0 <= j < self.total
            if drain:
                yield from drain_load(j, b)
            if gi < self.total:
                yield from self.wait(self.qdo_full[gi % self.nqs], gi // self.nqs, "buf.qdo_full")
                # buffer b's previous phase (tile gi - buffers) complete before
                # this warp arrives for tile gi, else a fast warp's arrival
                # could complete it in a slow sibling's place; in atomic mode
                # the producer's wait (tile buffers) and the drains imply it
                if gi >= self.nb and not self.atomic:
                    yield from self.wait(self.buf_ready[b], (gi - self.nb) // self.nb, "buf.buf_ready")
                self.buf_ready[b].arrive()
                if gi < self.nb and w == 8:  # no dV, dK(gi - buffers) to commit
                    self.buf_ready[b].arrive()
            if drain:
                yield from drain_add(j)
            yield
        if self.atomic and self.d64 and quad == 2:
            while not all(g[1] for g in self.groups["reduce"]):
                yield

    # ------------------------------------------------------------ elementwise warps
    def signal_epi_read(self):
        """Thread 0 (one of the elementwise threads): the latest epilogue's
        store has read its staging before epi_read is signalled."""
        if self.epi_pending:
            while not all(g[0] for g in self.groups["epilogue"]):
                yield
            self.epi_read.arrive()
            self.epi_pending = False

    def elementwise(self):
        gi, epi_last = 0, -3
        self.epi_pending = False
        for k, n in enumerate(self.units):
            for _ in range(n):
                b, st, sd = gi % self.nb, gi % self.nqs, gi % 3
                yield from self.wait(self.s_full[b], gi // self.nb, "elem.s_full")
                yield from self.wait(self.qdo_full[st], gi // self.nqs, "elem.qdo_full")
                if self.S[b] is None or self.S[b][:2] != ["S", gi]:
                    raise ProtocolError(f"elementwise({gi}) reads S^T buffer {self.S[b]}")
                if self.P[b] is None or self.P[b][:2] != ["dP", gi]:
                    raise ProtocolError(f"elementwise({gi}) reads dP^T buffer {self.P[b]}")
                if self.stage[st] != (gi, True):
                    raise ProtocolError(f"elementwise({gi}) reads LSE / Di of stage {self.stage[st]}")
                self.S[b][2] = True
                if self.atomic:
                    self.s_read[b].arrive()
                yield
                self.P[b] = ["PdS", gi, False]
                self.p_full[b].arrive()
                if self.atomic:
                    yield from self.signal_epi_read()
                    if gi >= 3:
                        yield from self.wait(self.dq_full[sd], (gi - 3) // 3, "elem.dq_full")
                    if self.res and gi - epi_last <= 2:
                        yield from self.wait(self.epi_read, k - 1, "elem.epi_read")
                    cur = self.dst[sd]
                    if cur is not None and not cur[2]:
                        raise ProtocolError(f"dS^T({gi}) overwrites {cur}")
                    self.dst[sd] = ["dS", gi, False]
                gi += 1
                yield
            if self.atomic and k == len(self.units) - 1:
                self.ds_last.arrive()
            # epilogue: read dV, dK; resident CTAs stage them in dS^T tiles
            last = gi - 1
            yield from self.wait(self.acc_full, k, "epi.acc_full")
            yield from self.signal_epi_read()
            if self.res and k > 0:
                yield from self.wait(self.epi_read, k - 1, "epi.epi_read")
            if self.res and self.atomic:
                for j in range(max(0, last - 2), last):
                    yield from self.wait(self.dq_full[j % 3], j // 3, "epi.dq_full")
            if self.acc is None or self.acc[:2] != [k, n]:
                raise ProtocolError(f"epilogue of unit {k} reads accumulators {self.acc}")
            self.acc[2] = True
            yield
            if self.res:
                tiles = ((last + 1) % 3, (last + 2) % 3)
                for t in tiles:
                    cur = self.dst[t]
                    if cur is not None and not cur[2]:
                        raise ProtocolError(f"epilogue of unit {k} stages over {cur}")
                    self.dst[t] = ["staging", k, False]
                group = [False, False, k]
                self.groups["epilogue"].append(group)

                def read(group=group, tiles=tiles):
                    for t in tiles:
                        if self.dst[t][:2] != ["staging", group[2]]:
                            raise ProtocolError(f"store of unit {group[2]} reads {self.dst[t]}")
                        self.dst[t][2] = True
                    group[0] = True

                def complete(group=group):
                    group[1] = True
                    self.stored.append(group[2])
                self.copies.append(read)
                self.after_read.append((group, complete))
                if self.independent_signal:
                    def signaller():
                        while not all(g[0] for g in self.groups["epilogue"]):
                            yield
                        self.epi_read.arrive()
                    self.spawned.append(signaller())
                else:
                    self.epi_pending = True  # signalled before the next wait on epi_read
            else:
                self.stored.append(k)
            epi_last = last
            yield
        while not all(g[1] for g in self.groups["epilogue"]):
            yield

    # ------------------------------------------------------------ scheduler
    def run(self, max_steps=400000):
        roles = {"producer": self.producer(), "score": self.score_issuer(),
                 "gradient": self.gradient_issuer(), "elementwise": self.elementwise()}
        for w in range(8, 12):
            roles[f"buffer{w}"] = self.buffer_warp(w)
        steps = 0
        while roles or self.q_score or self.q_grad or self.copies or self.after_read:
            steps += 1
            while self.spawned:
                roles[f"issuer{steps}_{len(self.spawned)}"] = self.spawned.pop()
            if steps > max_steps:
                raise ProtocolError("no progress: " + ", ".join(roles))
            choices = list(roles)
            if self.q_score:
                choices.append("q_score")
            if self.q_grad:
                choices.append("q_grad")
            if self.copies:
                choices.append("copy")
            done_reading = [x for x in self.after_read if x[0][0]]
            if done_reading:
                choices.append("complete")
            if not choices:
                raise ProtocolError("deadlock: nothing can run")
            c = self.chooser.pick(choices, steps)
            if c in ("q_score", "q_grad"):
                kind, x = (self.q_score if c == "q_score" else self.q_grad).pop(0)
                if kind == "mma":
                    x()
                else:
                    x.arrive()
            elif c == "copy":
                self.copies.pop(self.rng.randrange(len(self.copies)))()
            elif c == "complete":
                entry = self.rng.choice(done_reading)
                self.after_read.remove(entry)
                entry[1]()
            else:
                self.chooser.enter(c, steps)
                try:
                    next(roles[c])
                except StopIteration:
                    del roles[c]
        if sorted(self.stored) != list(range(len(self.units))):
            raise ProtocolError(f"units stored: {sorted(self.stored)}")
        if self.atomic and sorted(self.reduced) != list(range(self.total)):
            raise ProtocolError(f"dQ tiles added: {sorted(self.reduced)} of {self.total}")


# Launch shapes: (buffers, resident, atomic_dq, d64).  Resident CTAs run at
# D = 64 only; D = 64 keeps three S^T / dP^T buffers, D = 128 two.
CONFIGS = [(3, True, True, True), (3, True, False, True), (3, False, True, True),
           (3, False, False, True), (2, False, True, False), (2, False, False, False)]

# Tiles per unit of a resident CTA's units (a one-unit CTA takes the first).
UNIT_PATTERNS = [[1], [2], [3], [4], [8], [1, 1, 1, 1, 1], [2, 1, 3, 1, 1, 2], [8, 8, 8],
                 [16, 14, 12, 2, 4, 6], [5, 1, 1, 7], [3, 3, 3, 3], [1, 2], [4, 1], [1] * 8]


def run_case(units, config, seed, skip=frozenset(), independent_signal=False, slow=frozenset()):
    buffers, resident, atomic_dq, d64 = config
    DkdvPipeline(units if resident else units[:1], buffers, resident, atomic_dq, d64, seed,
                 skip, independent_signal, slow).run()
