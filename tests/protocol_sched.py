"""The seeded step chooser shared by the barrier-protocol models
(tests/dkdv_protocol.py, tests/fwd_protocol.py, tests/dq_protocol.py).

Test infrastructure: nothing here runs on a GPU.  Each model's scheduler
asks `pick` for the next step among the runnable roles and queues, tells
`enter` which role it steps, and each model's wait calls `blocked` when the
barrier it waits on has not reached the awaited phase yet.
"""


class Chooser:
    """slow: roles (or queue names) picked rarely, so that interleavings in
    which one of them lags far behind the others come up often; "blocked":
    a role that finds a wait unsatisfied is, one time in ten, starved for
    the next 150 steps (a warp that falls behind just as its wait is about
    to pass, the case a uniform choice almost never produces)."""

    def __init__(self, rng, slow=frozenset()):
        self.rng = rng
        self.on_block = slow == "blocked"
        self.slow = set() if self.on_block else set(slow)
        self.current, self.steps, self.until = None, 0, 0

    def blocked(self):
        if self.on_block and not self.slow and self.rng.random() < 0.1:
            self.slow, self.until = {self.current}, self.steps + 150

    def enter(self, role, steps):
        self.current, self.steps = role, steps

    def pick(self, choices, steps):
        if self.on_block and self.slow and steps >= self.until:
            self.slow = set()
        if self.slow:
            return self.rng.choices(choices, [0.03 if c in self.slow else 1.0 for c in choices])[0]
        return self.rng.choice(choices)
