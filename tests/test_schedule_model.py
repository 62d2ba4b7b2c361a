"""A model of the fused GEMM-epilogue kernel's persistent schedule with the
workspace exchange (host logic, CPU only).

W workers (CTAs, or CTA pairs) take the work items of a strip-major order
round-robin (worker w: items w, w + W, w + 2W, ...).  A worker holds two
items at once (two TMEM accumulators): the main loop of its k-th item waits
until the epilogue of its (k-2)-th item has released the accumulator.  An
item's epilogue finishes once every item of its strip (T tiles) has finished
its main loop, and a worker's epilogues run in order.  The launch code
refuses (or re-plans with more workers) any strip wider than 2 W tiles; the
model shows that this is exactly the condition for every strip to finish.
"""
import pytest


def schedule_completes(workers: int, strips: int, tiles: int) -> bool:
    items = strips * tiles
    queues = [list(range(w, items, workers)) for w in range(workers)]
    mma_done = [False] * items
    remaining = [tiles] * strips          # tiles of each strip whose main loop has not finished
    k = [0] * workers                     # next item (index into the queue) to start its main loop
    e = [0] * workers                     # next item whose epilogue must finish
    progress = True
    while progress:
        progress = False
        for w, q in enumerate(queues):
            while k[w] < len(q) and k[w] - e[w] < 2:       # a free accumulator
                it = q[k[w]]
                mma_done[it] = True
                remaining[it // tiles] -= 1
                k[w] += 1
                progress = True
            while e[w] < k[w] and remaining[q[e[w]] // tiles] == 0:  # strip complete
                e[w] += 1
                progress = True
    return all(e[w] == len(q) for w, q in enumerate(queues))


def host_accepts(workers: int, tiles: int) -> bool:
    """The launch rule: a strip's tiles fit in twice the resident workers."""
    return tiles <= 2 * workers


@pytest.mark.parametrize("workers", [1, 2, 3, 5, 8, 13, 19, 32])
def test_rule_is_exact(workers):
    for strips in (1, 2, 3, 7):
        for tiles in range(1, 3 * workers + 3):
            # The launch never starts more workers than items.
            w = min(workers, strips * tiles)
            assert schedule_completes(w, strips, tiles) == host_accepts(w, tiles), (w, strips, tiles)


def test_gb300_shapes():
    # CTA pairs on a 152-SM GB300 (76 pairs): the 16384-wide softmax head
    # (64 tiles per strip pair) fits; a 50,257-wide row (197 tiles) needs the
    # 1-CTA tiles (152 workers, up to 304 tiles, N <= 77,824).
    assert host_accepts(76, 64) and schedule_completes(76, 4, 64)
    assert not host_accepts(76, 197) and not schedule_completes(76, 4, 197)
    assert host_accepts(152, 197) and schedule_completes(152, 4, 197)
    assert not host_accepts(152, 305)
