"""The slot pool's buffer map (host logic, no GPU).

The LRU kernel gives every access a buffer of the slot pool: a first-wave
access (index i < n_slots) the buffer of its LRU slot, a later one spare
buffer i - n_slots; at the end of a step every later-wave access that keeps its
slot swaps buffers with it.  This restates that rule next to the oracle's LRU
and checks, over random steps with many waves, the property the kernels rely
on: a hit always finds its expert in the buffer it is given, no fill
overwrites a buffer another access of the step reads, and after each step
every slot's buffer holds the expert the table names.
"""
import random

from oracle.lru import SlotTable


def _run(E, S, k, N, steps, rng):
    X = max(0, min(E, N * k) - S)
    T = SlotTable(E, S)
    buf = list(range(S)) + [S + 1 + j for j in range(X)]   # buffer S is the shared expert's
    content = {}
    for _ in range(steps):
        acc = T.step([rng.randrange(E) for _ in range(rng.randint(1, N) * k)])
        U = len(acc)
        assert U - S <= X
        nh = sum(1 for a in acc if a[2])
        ab = [buf[a[1]] if i < S else buf[S + (i - S)] for i, a in enumerate(acc)]
        assert S not in ab
        for i in range(nh):
            assert content.get(ab[i]) == acc[i][0]
        filled = ab[nh:]
        assert len(set(filled)) == len(filled) and not set(filled) & set(ab[:nh])
        for i in range(nh, U):
            content[ab[i]] = acc[i][0]
        for i in range(max(S, U - S), U):
            s, j = acc[i][1], S + (i - S)
            buf[s], buf[j] = buf[j], buf[s]
        for s in range(S):
            if T.expert_of[s] >= 0:
                assert content.get(buf[s]) == T.expert_of[s]
        assert sorted(buf) == list(range(S)) + [S + 1 + j for j in range(X)]


def test_buffer_map_keeps_data_with_the_table():
    rng = random.Random(7)
    for _ in range(200):
        E = rng.randint(2, 64)
        S = rng.randint(1, E)
        k = rng.randint(1, min(8, E))
        _run(E, S, k, rng.randint(1, 16), 30, rng)


def test_decode_35b_batch16_shape():
    # 128 experts, 47 slots, top-8, 16 tokens: two or three waves per step
    _run(128, 47, 8, 16, 60, random.Random(11))
