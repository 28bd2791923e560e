"""A discrete-event model of the mbarrier pipelines of the CUDA kernels, for checking
their synchronisation protocols on the host (compute-sanitizer's race checks are not
available here).

Each role of a kernel (a loader lane, an MMA-issuing lane, a softmax warp, ...) is a
Python generator that yields the operations it performs, in program order:

  ("wait", bar, k)        block until completion k (0-based) of `bar` has happened; the
                          hardware waits on a phase parity, so the model also checks that
                          the barrier is then at completion k or k + 1 (never two phases
                          off, which a parity wait cannot tell apart)
  ("arrive", bar)         one arrival
  ("expect", bar, nbytes) arrive with an expected transaction count (arrive.expect_tx)
  ("tma", bar, nbytes, write)   an asynchronous copy: `write()` runs when it lands, then
                          its bytes complete on `bar`
  ("mma", issuer, fn)     an MMA queued on the tensor pipe, which runs MMAs one at a time
                          in the order issued; `fn()` runs when the MMA executes
  ("commit", issuer, bar) arrive on `bar` once every MMA this issuer queued so far has run
  ("do", fn)              a synchronous action of the role (a register / TMEM access)

The scheduler runs one enabled event at a time, chosen at random: a role whose next
operation can proceed, a landing copy, or the MMA at the head of the queue.  A state in
which nothing can proceed while a role still waits is a deadlock.  Barrier misuse (an
arrival beyond the expected count, a transaction count below zero) raises at once;
resource checks (what a buffer holds when it is read or overwritten) are the kernel
models' own asserts inside the actions.
"""
import random
from collections import deque


class ProtocolError(AssertionError):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.completed = count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def arrive(self):
        if self.pending <= 0:
            raise ProtocolError(f"{self.name}: arrival beyond the expected count")
        self.pending -= 1
        self._maybe_complete()

    def expect(self, nbytes):
        if self.pending <= 0:
            raise ProtocolError(f"{self.name}: arrival beyond the expected count")
        self.tx += nbytes
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        if self.tx < 0:
            raise ProtocolError(f"{self.name}: more bytes completed than expected")
        self._maybe_complete()


class Deadlock(ProtocolError):
    pass


def run(roles, seed, end_idle=False, max_events=1_000_000):
    """Run the roles (name -> generator) to completion under one random schedule.
    end_idle: when the last role ends (the block exits), no copy, MMA or commit may still
    be in flight.  Returns the number of events."""
    rng = random.Random(seed)
    pending = {}            # role -> its next operation (not yet performed)
    first_look = {}         # role -> whether its current wait was checked for parity aliasing
    copies = []             # landing copies: (bar, nbytes, write)
    mma_queue = deque()     # (issuer, fn)
    issued = {}             # issuer -> MMAs queued so far
    done_mmas = {}          # issuer -> MMAs executed so far
    commits = []            # (issuer, target count, bar)
    gens = dict(roles)

    def advance(name):
        try:
            pending[name] = next(gens[name])
        except StopIteration:
            pending.pop(name, None)
            del gens[name]
        first_look[name] = False

    for name in list(gens):
        advance(name)

    def perform(name, op):
        kind = op[0]
        if kind == "arrive":
            op[1].arrive()
        elif kind == "expect":
            op[1].expect(op[2])
        elif kind == "tma":
            copies.append((op[1], op[2], op[3]))
        elif kind == "mma":
            issuer = op[1]
            mma_queue.append((issuer, op[2]))
            issued[issuer] = issued.get(issuer, 0) + 1
        elif kind == "commit":
            issuer, bar = op[1], op[2]
            target = issued.get(issuer, 0)
            if done_mmas.get(issuer, 0) >= target:
                bar.arrive()
            else:
                commits.append((issuer, target, bar))
        elif kind == "do":
            op[1]()
        else:
            raise ValueError(kind)

    def wait_ready(name, op):
        bar, k = op[1], op[2]
        if not first_look[name]:
            first_look[name] = True
            if bar.completed not in (k, k + 1):
                raise ProtocolError(f"{name}: waits for completion {k} of {bar.name} at completion "
                                    f"{bar.completed} (a parity wait would see the wrong phase)")
        if bar.completed > k + 1:
            raise ProtocolError(f"{name}: {bar.name} ran two phases past completion {k}")
        return bar.completed == k + 1

    for events in range(max_events):
        enabled = []
        for name, op in pending.items():
            if op[0] != "wait" or wait_ready(name, op):
                enabled.append(("role", name))
        enabled += [("copy", i) for i in range(len(copies))]
        if mma_queue:
            enabled.append(("mma", None))
        if not enabled:
            if pending:
                raise Deadlock("deadlock: " + ", ".join(
                    f"{n} waits {op[1].name}#{op[2]} (at {op[1].completed})" for n, op in pending.items()
                    if op[0] == "wait"))
            return events
        kind, which = enabled[rng.randrange(len(enabled))]
        if kind == "role":
            op = pending[which]
            if op[0] != "wait":
                perform(which, op)
            advance(which)
            if end_idle and not pending and (copies or mma_queue or commits):
                raise ProtocolError(f"the block exits with {len(copies)} copies, {len(mma_queue)} MMAs and "
                                    f"{len(commits)} commits in flight")
        elif kind == "copy":
            bar, nbytes, write = copies.pop(which)
            write()
            bar.complete_tx(nbytes)
        else:
            issuer, fn = mma_queue.popleft()
            fn()
            done_mmas[issuer] = done_mmas.get(issuer, 0) + 1
            still = []
            for c in commits:
                if c[0] == issuer and done_mmas[issuer] >= c[1]:
                    c[2].arrive()
                else:
                    still.append(c)
            commits[:] = still
    raise ProtocolError("no end within the event budget")
