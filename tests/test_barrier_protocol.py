"""CPU model of the score CTA's barrier protocol in the decode kernel.

The kernel's waits are mbarrier parity waits: a wait for phase k of a barrier that has completed
c phases returns when c & 1 != k & 1.  That is right only while c is k or k + 1; a waiter whose
barrier is a phase behind (c = k - 1) or two phases ahead (c = k + 2) is silently wrong.  This
model runs the page producer, the two MMA issuers and the softmax warps of one CTA as
coroutines under random schedules, with MMA completions delivered asynchronously. Every wait
asserts that c lies in {k, k + 1} whenever it is evaluated.

The protocol the kernel uses (with three page stages; the model also runs other counts):
- each item first occupies two stage positions with its query;
- page g goes to issuer g & 1 and S buffer g & 1;
- both issuers walk every stage position in order; the page's issuer commits, the other
  arrives (empty count 2);
- each issuer acknowledges each item's QReady (QAck, count 2), and the softmax waits for the
  previous item's acknowledgements before completing the next QReady.

Both rules are needed in general, which also shows the check has teeth. Without the
in-order walk the model finds aliasing at three stages. Without QAck it finds aliasing at five
stages; at three, the query stages' double release already orders QReady.
"""
import random

import pytest


class Aliasing(AssertionError):
    pass


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def simulate(items, seed, stages=3, qack=True, walk_all=True):
    STAGES = stages
    rnd = random.Random(seed)
    bars = {}
    for s in range(STAGES):
        bars[f"full{s}"] = Barrier(1)
        bars[f"empty{s}"] = Barrier(2 if walk_all else 1)
    for b in range(2):
        bars[f"sfull{b}"] = Barrier(1)
        bars[f"sempty{b}"] = Barrier(1)
    bars["qready"] = Barrier(1)
    bars["qack"] = Barrier(2)
    inflight = []  # asynchronous completions (TMA landings, MMA commits), in any order

    def ready(name, k):
        c = bars[name].done
        if c >= k + 2 or c < k:
            raise Aliasing(f"{name}: waiting for phase {k}, {c} completed")
        return (c & 1) != (k & 1)

    def producer():
        u = 0
        for T in items:
            for _ in range(2 + T):
                s = u % STAGES
                if u >= STAGES:
                    while not ready(f"empty{s}", u // STAGES - 1):
                        yield
                inflight.append(f"full{s}")
                u += 1
                yield

    def issuer(me):
        g = ic = u = 0
        for T in items:
            while not ready("qready", ic):
                yield
            ic += 1
            if qack:
                bars["qack"].arrive()
            if me == 0 or walk_all:
                bars[f"empty{u % STAGES}"].arrive()
                bars[f"empty{(u + 1) % STAGES}"].arrive()
            u += 2
            for _ in range(T):
                s = u % STAGES
                mine = (g & 1) == me
                if walk_all or mine:
                    while not ready(f"full{s}", u // STAGES):
                        yield
                if mine:
                    if g >= 2:
                        while not ready(f"sempty{me}", (g >> 1) - 1):
                            yield
                    inflight.append(f"empty{s}")
                    inflight.append(f"sfull{me}")
                elif walk_all:
                    bars[f"empty{s}"].arrive()
                g += 1
                u += 1
                yield

    def softmax():
        g = n = u = 0
        for T in items:
            if qack and n > 0:
                while not ready("qack", n - 1):
                    yield
            while not ready(f"full{u % STAGES}", u // STAGES):
                yield
            while not ready(f"full{(u + 1) % STAGES}", (u + 1) // STAGES):
                yield
            bars["qready"].arrive()
            u += 2
            for _ in range(T):
                while not ready(f"sfull{g & 1}", g >> 1):
                    yield
                bars[f"sempty{g & 1}"].arrive()
                g += 1
                u += 1
                yield
            n += 1

    roles = [producer(), issuer(0), issuer(1), softmax()]
    alive = list(range(len(roles)))
    for _ in range(2_000_000):
        if not alive:
            return
        if inflight and rnd.random() < 0.3:
            bars[inflight.pop(rnd.randrange(len(inflight)))].arrive()
            continue
        r = rnd.choice(alive)
        try:
            next(roles[r])
        except StopIteration:
            alive.remove(r)
    raise AssertionError("no progress")


def random_items(rnd):
    return [rnd.choice([1, 1, 1, 1, 2, 2, 3, 5, 8]) for _ in range(rnd.randint(1, 14))]


def count_aliasing(trials, **kw):
    bad = 0
    for t in range(trials):
        rnd = random.Random(7000 + t)
        try:
            simulate(random_items(rnd), seed=t, **kw)
        except Aliasing:
            bad += 1
    return bad


@pytest.mark.parametrize("stages", [2, 3, 4, 5])
def test_kernel_protocol_never_aliases(stages):
    assert count_aliasing(300, stages=stages) == 0


@pytest.mark.parametrize("kw", [dict(stages=3, walk_all=False), dict(stages=5, qack=False)])
def test_dropping_a_rule_is_caught(kw):
    assert count_aliasing(300, **kw) > 0
