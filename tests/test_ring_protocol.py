"""CPU model of the P-message path between the two CTAs of the decode kernel.

Roles, as in the kernel, for one CTA pair walking its pages g = 0, 1, ... (item boundaries
included):
- softmax (score CTA): per page, wait until ring slot g % R is free (PFree), write the message,
  then mark it staged (PStaged) -- at once on an item's last page, otherwise after the next
  page's scores have been read (the release then no longer waits for the message's stores);
- shipper (score CTA): wait for the oldest unpublished message, take the later staged ones of
  the same item (non-blocking tests, at most kMaxBatch), and publish each (PReady on the
  partner);
- P loader (accumulate CTA): per message, wait PReady, wait until P buffer g % PB is free
  (PBufFree), then start the copy (PFull completes asynchronously);
- releaser (accumulate CTA): per message, wait PFull, then free the ring slot (PFree on the
  partner) and give the buffer its first release (PBufFree);
- PV MMA warp (accumulate CTA): per message, wait PFull and run the MMAs. Their commit is the
  buffer's second release, except on an item's last page: there the epilogue uses the buffer as
  staging, and the MMA warp releases it once the epilogue reports done (CorrEvt), at the next
  item's first page;
- epilogue warps: serve each item's epilogue event (MmaEvt) and report done (CorrEvt).

As in the score-CTA model, every parity wait asserts that its barrier has completed neither
fewer phases than the one awaited nor two more, and every run must finish.
"""
import random

import pytest

MAX_BATCH = 4


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


def simulate(items, seed, ring=16, pbufs=4, max_steps=3_000_000, epilogue_release=True, deferred=True):
    rnd = random.Random(seed)
    bars = {}
    for j in range(ring):
        bars[f"pfree{j}"] = Barrier(1)
        bars[f"pready{j}"] = Barrier(1)
        bars[f"pstaged{j}"] = Barrier(1)
    for j in range(pbufs):
        bars[f"pfull{j}"] = Barrier(1)
        bars[f"pbuffree{j}"] = Barrier(2)
    bars["mmaevt"] = Barrier(2)   # the MMA warp's arrival and its commit
    bars["correvt"] = Barrier(1)  # the epilogue warps (one entity here)
    inflight = []                 # asynchronous completions: copies landing, MMA commits
    n_pages = sum(items)
    last_of = set()
    g = 0
    for T in items:
        g += T
        last_of.add(g - 1)
    item_end = []
    g = 0
    for T in items:
        item_end += [g + T] * T
        g += T

    def ready(name, k):
        c = bars[name].done
        if c >= k + 2 or c < k:
            raise Aliasing(f"{name}: waiting for phase {k}, {c} completed")
        return (c & 1) != (k & 1)

    def test(name, k):  # the shipper's non-blocking look at a later slot
        c = bars[name].done
        if c >= k + 2:
            raise Aliasing(f"{name}: testing phase {k}, {c} completed")
        return c > k and (c & 1) != (k & 1)

    def softmax():
        pending = None
        for g in range(n_pages):
            yield  # the page's scores are read
            if pending is not None:  # the previous message's deferred release
                bars[f"pstaged{pending}"].arrive()
                pending = None
            if g >= ring:
                while not ready(f"pfree{g % ring}", g // ring - 1):
                    yield
            yield  # the message's stores
            if g in last_of or not deferred:  # an item's last message goes at once
                bars[f"pstaged{g % ring}"].arrive()
            else:
                pending = g % ring

    def shipper():
        g = 0
        while g < n_pages:
            while not ready(f"pstaged{g % ring}", g // ring):
                yield
            n = 1
            while g + n < item_end[g] and n < MAX_BATCH and test(f"pstaged{(g + n) % ring}", (g + n) // ring):
                n += 1
            yield  # the cluster-scope fence
            for k in range(n):
                bars[f"pready{(g + k) % ring}"].arrive()
            g += n

    def loader():
        for g in range(n_pages):
            while not ready(f"pready{g % ring}", g // ring):
                yield
            if g >= pbufs:
                while not ready(f"pbuffree{g % pbufs}", g // pbufs - 1):
                    yield
            inflight.append(f"pfull{g % pbufs}")
            yield

    def releaser():
        for g in range(n_pages):
            while not ready(f"pfull{g % pbufs}", g // pbufs):
                yield
            bars[f"pfree{g % ring}"].arrive()
            bars[f"pbuffree{g % pbufs}"].arrive()
            yield

    def mma():
        cv = 0
        pending = None
        g = 0
        for T in items:
            for t in range(T):
                while not ready(f"pfull{g % pbufs}", g // pbufs):
                    yield
                if t == 0 and pending is not None:
                    while not ready("correvt", cv):
                        yield
                    cv += 1
                    if epilogue_release:  # the epilogue is done with its staging buffer
                        bars[f"pbuffree{pending}"].arrive()
                    pending = None
                if g not in last_of:
                    inflight.append(f"pbuffree{g % pbufs}")  # the MMA commit
                else:
                    bars["mmaevt"].arrive()
                    inflight.append("mmaevt")  # the commit after the item's last MMAs
                    pending = g % pbufs
                g += 1
                yield
        if pending is not None:
            while not ready("correvt", cv):
                yield

    def epilogue():
        for ev in range(len(items)):
            while not ready("mmaevt", ev):
                yield
            yield  # read out O through the staging buffer
            bars["correvt"].arrive()

    roles = [softmax(), shipper(), loader(), releaser(), mma(), epilogue()]
    alive = list(range(len(roles)))
    for _ in range(max_steps):
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
    return [rnd.choice([1, 1, 2, 3, 4, 7, 17, 40]) for _ in range(rnd.randint(1, 8))]


@pytest.mark.parametrize("ring,pbufs,deferred", [(16, 4, True), (8, 3, True), (4, 2, True), (16, 4, False)])
def test_ring_protocol_never_aliases(ring, pbufs, deferred):
    for t in range(100):
        rnd = random.Random(9100 + t)
        simulate(random_items(rnd), seed=t, ring=ring, pbufs=pbufs, deferred=deferred)


def test_dropping_the_epilogue_release_is_caught():
    """The model has teeth: without the MMA warp's release after the epilogue, an item's last
    P buffer gets one release instead of two, and the run cannot finish."""
    caught = 0
    for items in ([3, 1, 2, 5], [1, 1, 1, 1, 1, 1]):
        for seed in range(5):
            try:
                simulate(items, seed, max_steps=50_000, epilogue_release=False)
            except AssertionError:
                caught += 1
    assert caught == 10
