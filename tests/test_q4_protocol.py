"""A model of the barrier protocol of the 4-bit decode projection kernel (gemm_q4.cu), run
under random schedules on the CPU.

Roles and barriers as the kernel uses them: one producer fills a ring of `S` shared-memory
stages (full / empty); eight converter warps unpack each stage's codes into a ring of `RA`
tensor-memory A slots (afull / aempty) and write the operand's group sums (xsf); two MMA
issuers take the stages of one parity each and fill a ring of `RG` accumulator slots
(accf / acce); four epilogue warps drain every stage in order.  An mbarrier wait only
compares the parity of the phase, so the model does the same: a waiter that runs two phases
ahead reads a stale phase as complete.  Every read is checked against the version of the data
it should see, and every schedule must finish (no deadlock).

The negative case is the arrangement the kernel used before: three issuers taking whole
stages in turn with more pipeline stages than accumulator slots, where an issuer can see a
slot two uses old as free; the model must catch it.
"""
import itertools
import random


class Bar:
    def __init__(self, count):
        self.count, self.arrived, self.done = count, 0, 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived, self.done = 0, self.done + 1

    def ready(self, parity):  # try_wait.parity: the phase with this parity has completed
        return (self.done & 1) != parity


def simulate(S, RA, RG, Tc, nsb, rng, n_issuers=2, NK=2, NC=8):
    nst = Tc * nsb
    full = [Bar(1) for _ in range(S)]
    empty = [Bar(1 + 4) for _ in range(S)]  # the stage's MMA commit, four epilogue warps
    xsf = [Bar(NC) for _ in range(S)]
    afull = [Bar(NC) for _ in range(RA)]
    aempty = [Bar(1) for _ in range(RA)]
    accf = [Bar(1) for _ in range(RG)]
    acce = [Bar(4) for _ in range(RG)]
    smem, xs, A, acc = [None] * S, [None] * S, [None] * RA, [None] * RG
    errors = []

    def check(what, have, want):
        if have != want:
            errors.append(what)

    def producer():
        for i in range(nst):
            st = i % S
            yield empty[st], ((i // S) & 1) ^ 1
            smem[st] = i
            full[st].arrive()

    def issuer(w):
        for i in range(w, nst, n_issuers):
            st, a = i % S, i % RA
            yield afull[a], (i // RA) & 1
            yield full[st], (i // S) & 1
            check("issuer reads the stage", smem[st], i)
            check("issuer reads A", A[a], i)
            for jj in range(NK):
                g = i * NK + jj
                sl = g % RG
                yield acce[sl], ((g // RG) & 1) ^ 1
                check("issuer finds the slot drained", acc[sl], ("drained", g - RG) if g >= RG else None)
                acc[sl] = g
                accf[sl].arrive()
            aempty[a].arrive()
            empty[st].arrive()

    def converter(w):
        for i in range(nst):
            st, a = i % S, i % RA
            yield full[st], (i // S) & 1
            yield aempty[a], ((i // RA) & 1) ^ 1
            check("converter reads the stage", smem[st], i)
            if w == 0:
                A[a] = i
            afull[a].arrive()
            if w == 0:
                xs[st] = i
            xsf[st].arrive()

    def epilogue(w):
        for i in range(nst):
            st = i % S
            yield full[st], (i // S) & 1
            yield xsf[st], (i // S) & 1
            check("epilogue reads scales", smem[st], i)
            check("epilogue reads group sums", xs[st], i)
            for jj in range(NK):
                g = i * NK + jj
                yield accf[g % RG], (g // RG) & 1
                check("epilogue reads the accumulator", acc[g % RG], g)
            for jj in range(NK):
                g = i * NK + jj
                before = acce[g % RG].done
                acce[g % RG].arrive()
                if acce[g % RG].done != before:
                    acc[g % RG] = ("drained", g)
            empty[st].arrive()

    roles = ([producer()] + [issuer(w) for w in range(n_issuers)] +
             [converter(w) for w in range(NC)] + [epilogue(w) for w in range(4)])
    waits = [None] * len(roles)
    alive = [True] * len(roles)
    for k, r in enumerate(roles):
        try:
            waits[k] = next(r)
        except StopIteration:
            alive[k] = False
    while any(alive):
        ready = [k for k in range(len(roles)) if alive[k] and waits[k][0].ready(waits[k][1])]
        if not ready:
            return "deadlock", errors
        k = rng.choice(ready)
        try:
            waits[k] = next(roles[k])
        except StopIteration:
            alive[k] = False
    return "done", errors


def test_kernel_protocol_has_no_deadlock_or_stale_read():
    rng = random.Random(5)
    # even pipeline depths (the kernel refuses odd ones); 8 slots for N <= 32, 4 for N = 64
    for RG, S in [(8, 8), (8, 6), (8, 4), (8, 2), (4, 8), (4, 4), (4, 2)]:
        for Tc, nsb in itertools.product([1, 2, 3], [1, 2, 3, 7, 16]):
            for _ in range(8):
                state, errors = simulate(S, 4, RG, Tc, nsb, rng)
                assert state == "done" and not errors, (RG, S, Tc, nsb, state, errors[:3])


def test_model_catches_out_of_order_issuers():
    rng = random.Random(5)
    failures = 0
    for Tc, nsb in itertools.product([1, 2], [7, 16]):
        for _ in range(20):
            state, errors = simulate(8, 4, 4, Tc, nsb, rng, n_issuers=3)
            failures += state != "done" or bool(errors)
    assert failures > 0
