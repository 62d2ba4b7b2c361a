"""A model of the fused GEMM-epilogue kernel's persistent schedule with the
workspace exchange (host logic, CPU only).

A worker (a CTA, or a CTA pair) holds two items at once (two TMEM
accumulators): the main loop of its k-th item waits until the epilogue of
its (k-2)-th item has released the accumulator.  An item's epilogue
finishes once every item of its strip (T tiles) has published its row
statistics, and a worker's epilogues run in order.

Single-stage programs take their items, in strip-major order, as tickets
from a global counter: a running worker claims the next ticket once its
item two back has finished its strip exchange (modelled here, more
strictly, as a free accumulator), so workers that are not resident (their
SMs held by other work) hold no items, and while an item waits for its
strip the epilogue publishes the statistics of the worker's next item.  The
launch code keeps T <= 2 W; the model shows that every strip then finishes
with any number of running workers R for which T <= 2 R, and only then.

Chained programs keep a static order (worker w: items w, w + W, ...) in
which the epilogue publishes an item's statistics only when it reaches
that item: a worker holding two tiles of one strip would wait for itself,
and the model shows that T <= W (with every launched worker running) is
exactly the condition for every strip to finish.
"""
import pytest


def schedule_completes(workers: int, strips: int, tiles: int) -> bool:
    """The static order (chained programs): worker w takes items w, w + W,
    ...; its main loop runs ahead of its epilogue by at most two items (two
    accumulators); its epilogue handles its items in order and publishes an
    item's statistics only when it reaches that item, then waits until every
    tile of the strip has published."""
    items = strips * tiles
    queues = [list(range(w, items, workers)) for w in range(workers)]
    main_done = [False] * items
    published = [0] * strips
    k = [0] * workers                     # next item (queue index) to start its main loop
    e = [0] * workers                     # the item the epilogue is at
    pub = [0] * workers                   # the next item the epilogue will publish
    progress = True
    while progress:
        progress = False
        for w, q in enumerate(queues):
            while k[w] < len(q) and k[w] - e[w] < 2:       # a free accumulator
                main_done[q[k[w]]] = True
                k[w] += 1
                progress = True
            while e[w] < len(q):
                it = q[e[w]]
                if pub[w] == e[w]:
                    if not main_done[it]:
                        break
                    published[it // tiles] += 1
                    pub[w] += 1
                    progress = True
                if published[it // tiles] < tiles:
                    break                                   # waits for its strip-mates
                e[w] += 1
                progress = True
    return all(e[w] == len(q) for w, q in enumerate(queues))


def ticket_order(strips: int, tiles: int):
    """(strip, tile) of each ticket: strip-major, alternate strips walking
    the tiles backwards."""
    return [(u, tiles - 1 - to if u % 2 else to) for u in range(strips) for to in range(tiles)]


def tickets_complete(running: int, strips: int, tiles: int) -> bool:
    """Tickets claimed in order by `running` workers, each only with a free
    accumulator (at most two unfinished items); an item's statistics are
    published once its main loop has run (the epilogue publishes a worker's
    next item while the current one waits)."""
    order = ticket_order(strips, tiles)
    assert sorted(order) == [(s, t) for s in range(strips) for t in range(tiles)]
    remaining = [tiles] * strips
    held = [[] for _ in range(running)]   # items of each worker, oldest first
    nxt = 0
    progress = True
    while progress:
        progress = False
        for w in range(running):
            while len(held[w]) < 2 and nxt < len(order):     # claim with a free accumulator
                strip, _ = order[nxt]
                nxt += 1
                held[w].append(strip)
                remaining[strip] -= 1                      # main loop, then published
                progress = True
            while held[w] and remaining[held[w][0]] == 0:  # the oldest epilogue finishes
                held[w].pop(0)
                progress = True
    return nxt == len(order) and all(not h for h in held)


def host_accepts(workers: int, tiles: int) -> bool:
    """The launch rule of the static order: a strip's tiles do not outnumber
    the workers (a worker never holds two tiles of one strip)."""
    return tiles <= workers


@pytest.mark.parametrize("workers", [1, 2, 3, 5, 8, 13, 19, 32])
def test_rule_is_exact(workers):
    for strips in (1, 2, 3, 7):
        for tiles in range(1, 3 * workers + 3):
            # The launch never starts more workers than items.
            w = min(workers, strips * tiles)
            assert schedule_completes(w, strips, tiles) == host_accepts(w, tiles), (w, strips, tiles)


def test_gb300_shapes():
    # Chained programs (static order) on a 152-SM GB300: 64 tiles per strip
    # pair fit the 76 pairs; 100 tiles need the 152 one-CTA workers; 153 do
    # not fit.  A worker holding two tiles of one strip waits for itself: the
    # earlier launch rule (twice the workers) let such shapes through.
    assert host_accepts(76, 64) and schedule_completes(76, 4, 64)
    assert not host_accepts(76, 100) and not schedule_completes(76, 4, 100)
    assert host_accepts(152, 100) and schedule_completes(152, 4, 100)
    assert not host_accepts(152, 153) and not schedule_completes(152, 4, 153)
    # Single-stage programs take tickets and publish a worker's next tile
    # early: up to twice the workers (197 tiles of a 50,257-wide row on 152
    # one-CTA workers, up to 304 tiles: N <= 77,824).
    assert tickets_complete(152, 4, 197) and tickets_complete(152, 2, 304)
    assert not tickets_complete(152, 2, 305)


@pytest.mark.parametrize("running", [1, 2, 3, 5, 8, 13])
def test_tickets_need_only_running_workers(running):
    # Whatever the launched grid, the schedule completes exactly when a
    # strip's tiles fit in twice the running workers' accumulators.
    for strips in (1, 2, 3, 7):
        for tiles in range(1, 3 * running + 3):
            assert tickets_complete(running, strips, tiles) == (tiles <= 2 * running), (running, strips, tiles)


def test_static_assignment_needs_every_launched_worker():
    # A static round-robin assignment over a launched grid of 8 workers of
    # which 5 run leaves the absent workers' items unprocessed (their
    # strip-mates wait); tickets taken by the 5 running workers finish.
    launched, running, strips, tiles = 8, 5, 4, 6
    items = strips * tiles
    static_items_of_absent = [i for w in range(running, launched) for i in range(w, items, launched)]
    assert static_items_of_absent  # the absent workers own items
    assert tickets_complete(running, strips, tiles)
