"""A model of the tensor-core prefill kernel's work counter, run under random
interleavings of its CTAs.

The counter is one 64-bit word, (launch tag << 32 | count).  Per launch:
* every CTA reads the word at entry and, if it holds another tag (or a count
  past the list), swaps exactly the value it read for (tag, 0);
* CTA b takes item b without the counter; a CTA with an item then draws
  numbers until one comes back past the list.  A draw adds 1; if the word it
  added to was stale, it re-reads the word and swaps exactly what it read
  for (tag, 1), taking 0 (it never adds to a stale word again);
* the CTA whose draw returns the last number (T - 1) stores (tag, 0), so a
  replay with the same tag starts from zero;
* a CTA that gave up mid-way keeps drawing to the end of the list without
  running the items.

Each atomic step of a CTA is one step of a Python generator, and a seeded
scheduler interleaves them.  Checked: every launch that nobody abandons runs
each dynamic item exactly once, and every launch leaves the word at (tag, 0),
whatever the word held before (a previous launch's tag, a replay of the same
tag, a clobbered header).
"""

import random

M64 = (1 << 64) - 1


def _launch(word, tag, grid, total, rnd, give_up_p):
    def fresh(v):
        return (v >> 32) == tag and (v & 0xFFFFFFFF) < total

    def take():
        v = word[0]
        word[0] = (word[0] + 1) & M64
        yield
        for _ in range(4096):
            if fresh(v):
                return v & 0xFFFFFFFF
            cur = word[0]
            yield
            if fresh(cur):
                v = word[0]
                word[0] = (word[0] + 1) & M64
                yield
            else:
                won = word[0] == cur
                if won:
                    word[0] = (tag << 32) | 1
                yield
                if won:
                    return 0
        raise AssertionError("a draw gave up")

    ran = []

    def cta(b):
        seen = word[0]
        yield
        if not fresh(seen):
            if word[0] == seen:
                word[0] = tag << 32
            yield
        if b >= total:
            return
        gave_up = rnd.random() < give_up_p
        if not gave_up:
            ran.append(b)
        while True:
            n = yield from take()
            if n == total - 1:
                word[0] = tag << 32
                yield
            e = grid + n
            if e >= total:
                return
            if not gave_up:
                ran.append(e)

    gens = [cta(b) for b in range(grid)]
    live = list(range(grid))
    while live:
        i = rnd.choice(live)
        try:
            next(gens[i])
        except StopIteration:
            live.remove(i)
    return ran


def test_work_counter_model_under_random_interleavings():
    for seed in range(300):
        rnd = random.Random(seed)
        word = [rnd.choice([0, M64, rnd.getrandbits(64), (9 << 32) | 5])]
        tags = [rnd.randint(1, 6) for _ in range(6)]  # repeats model graph replays
        for k, tag in enumerate(tags):
            grid = rnd.randint(1, 40)
            total = rnd.choice([rnd.randint(1, 30), rnd.randint(grid, grid + 150)])
            if rnd.random() < 0.2:
                word[0] = rnd.getrandbits(64)  # a clobbered header between launches
            give_up_p = 0.3 if rnd.random() < 0.3 else 0.0
            ran = _launch(word, tag, grid, total, rnd, give_up_p)
            if give_up_p == 0.0:
                assert sorted(ran) == list(range(total)), (seed, k)
            assert word[0] == tag << 32, (seed, k, hex(word[0]))
