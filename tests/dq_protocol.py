"""A random-interleaving model of the barrier protocol of the deterministic
dQ kernel (`bwd_dq_pipe_kernel` in exact_attention_93_gb300/csrc/fa_bwd.cu).

Test infrastructure: nothing here runs on a GPU, and the kernel does not use
it.  One CTA owns one query tile and walks its 64-key tiles in order.  The
roles: the producer (Q, dO with their LSE / Di rows once; K, V through a
four-stage ring), the relay warp (K, V of a tile landed -> its buffer may
take S, dP), the score issuer (S = Q K^T and dP = dO V^T into one of three
TMEM buffers), the eight elementwise warps (dS over the dP columns) and the
gradient issuer (dQ += dS K, accumulated in TMEM in tile order), and the
epilogue (dQ staged over Q in shared memory, then stored).  A seeded
scheduler picks the next step among the runnable roles, the two tensor-core
queues (each in order) and the copies in flight.  The model checks every
parity wait and every buffer, as the dK/dV model does; `skip` names waits to
leave out.
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


class DqPipeline:
    BUFFERS, STAGES = 3, 4

    def __init__(self, n_tiles, seed, skip=frozenset(), slow=frozenset()):
        self.rng = random.Random(seed)
        self.chooser = Chooser(self.rng, slow)  # slow: see protocol_sched.Chooser
        self.n, self.skip = n_tiles, set(skip)
        B, nb, ns = Barrier, self.BUFFERS, self.STAGES
        self.q_full = B("q_full", 1)
        self.kv_full = [B(f"kv_full{i}", 1) for i in range(ns)]
        self.kv_empty = [B(f"kv_empty{i}", 1) for i in range(ns)]
        self.s_full = [B(f"s_full{i}", 1) for i in range(nb)]
        self.p_full = [B(f"p_full{i}", 1) for i in range(nb)]
        # the relay warp and the commit that retires dQ(it - buffers)
        self.buf_ready = [B(f"buf_ready{i}", 2) for i in range(nb)]
        self.all_done = B("all_done", 1)
        self.drain = [B("drain0", 1), B("drain1", 1)]
        self.q_score, self.q_grad, self.copies = [], [], []
        self.q_landed, self.q_readers, self.q_stage = False, 0, False  # Q / dO; Q reused for dQ
        self.kv = [None] * ns       # (tile, landed)
        self.kv_readers = [0] * ns  # products queued to read the stage
        self.buf = [None] * nb      # ['S', it] or ['dS', it, consumed]
        self.dq_tiles = 0           # dQ products executed, in order
        self.stored = False

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

    def producer(self):
        def land_q():
            self.q_landed = True
            self.q_full.arrive()
        self.copies.append(land_q)
        yield
        for it in range(self.n):
            st = it % self.STAGES
            if it >= self.STAGES:
                yield from self.wait(self.kv_empty[st], (it - self.STAGES) // self.STAGES, "prod.kv_empty")

            def land(st=st, it=it):
                if self.kv_readers[st]:
                    raise ProtocolError(f"K / V({it}) lands while products read tile {self.kv[st]}")
                self.kv[st] = (it, True)
                self.kv_full[st].arrive()
            self.copies.append(land)
            yield

    def relay(self):
        for it in range(self.n):
            yield from self.wait(self.kv_full[it % self.STAGES], it // self.STAGES, "relay.kv_full")
            self.buf_ready[it % self.BUFFERS].arrive()
            if it < self.BUFFERS:  # no dQ(it - buffers) to wait for
                self.buf_ready[it % self.BUFFERS].arrive()
            yield

    def score_issuer(self):
        yield from self.wait(self.q_full, 0, "score.q_full")
        for it in range(self.n):
            b, st = it % self.BUFFERS, it % self.STAGES
            yield from self.wait(self.buf_ready[b], it // self.BUFFERS, "score.buf_ready")
            self.kv_readers[st] += 1
            self.q_readers += 1

            def products(b=b, st=st, it=it):
                self.kv_readers[st] -= 1
                self.q_readers -= 1
                if self.kv[st] != (it, True):
                    raise ProtocolError(f"S, dP({it}) read K / V stage {self.kv[st]}")
                if not self.q_landed or self.q_stage:
                    raise ProtocolError(f"S, dP({it}) read Q / dO before they landed or after reuse")
                old = self.buf[b]
                if old is not None and not (old[0] == "dS" and old[2]):
                    raise ProtocolError(f"S, dP({it}) overwrite {old}")
                self.buf[b] = ["S", it]
            self.q_score.append(("mma", products))
            self.q_score.append(("commit", self.s_full[b]))
            yield
        self.q_score.append(("commit", self.drain[0]))
        yield from self.wait(self.drain[0], 0)

    def elementwise(self):
        yield from self.wait(self.q_full, 0, "elem.q_full")
        for it in range(self.n):
            b = it % self.BUFFERS
            yield from self.wait(self.s_full[b], it // self.BUFFERS, "elem.s_full")
            if self.buf[b] != ["S", it]:
                raise ProtocolError(f"elementwise({it}) reads {self.buf[b]}")
            yield
            self.buf[b] = ["dS", it, False]
            self.p_full[b].arrive()
            yield
        # epilogue: dQ read from TMEM, staged over Q, stored
        yield from self.wait(self.all_done, 0, "epi.all_done")
        if self.dq_tiles != self.n:
            raise ProtocolError(f"epilogue reads dQ after {self.dq_tiles} of {self.n} tiles")
        if self.q_readers:
            raise ProtocolError("epilogue stages dQ over Q while products still read it")
        self.q_stage = True
        yield
        self.stored = True

    def gradient_issuer(self):
        for it in range(self.n):
            b, st = it % self.BUFFERS, it % self.STAGES
            yield from self.wait(self.p_full[b], it // self.BUFFERS, "grad.p_full")
            self.kv_readers[st] += 1

            def product(b=b, st=st, it=it):
                self.kv_readers[st] -= 1
                if self.kv[st] != (it, True):
                    raise ProtocolError(f"dQ({it}) reads K stage {self.kv[st]}")
                if self.buf[b] is None or self.buf[b][:2] != ["dS", it]:
                    raise ProtocolError(f"dQ({it}) reads {self.buf[b]}")
                if self.dq_tiles != it:
                    raise ProtocolError(f"dQ({it}) after {self.dq_tiles} tiles")
                self.buf[b][2] = True
                self.dq_tiles += 1
            self.q_grad.append(("mma", product))
            self.q_grad.append(("commit", self.kv_empty[st]))
            self.q_grad.append(("commit", self.buf_ready[b]))
            yield
        self.q_grad.append(("commit", self.all_done))
        self.q_grad.append(("commit", self.drain[1]))
        yield from self.wait(self.drain[1], 0)

    def run(self, max_steps=200000):
        roles = {"producer": self.producer(), "relay": self.relay(), "score": self.score_issuer(),
                 "elementwise": self.elementwise(), "gradient": self.gradient_issuer()}
        steps = 0
        while roles or self.q_score or self.q_grad or self.copies:
            steps += 1
            if steps > max_steps:
                raise ProtocolError("no progress: " + ", ".join(roles))
            choices = list(roles) + [x for x, q in (("q_score", self.q_score), ("q_grad", self.q_grad),
                                                    ("copy", self.copies)) if q]
            if not choices:
                raise ProtocolError("deadlock: nothing can run")
            c = self.chooser.pick(choices, steps)
            if c in ("q_score", "q_grad"):
                kind, x = (self.q_score if c == "q_score" else self.q_grad).pop(0)
                x() if kind == "mma" else x.arrive()
            elif c == "copy":
                self.copies.pop(self.rng.randrange(len(self.copies)))()
            else:
                self.chooser.enter(c, steps)
                try:
                    next(roles[c])
                except StopIteration:
                    del roles[c]
        if not self.stored:
            raise ProtocolError("dQ not stored")


# 64-key tiles a query tile walks (0: a tile the block mask leaves without keys)
TILE_COUNTS = [0, 1, 2, 3, 4, 5, 7, 8, 13, 32]
