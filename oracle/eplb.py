"""Oracle for the expert placement/replication plan (test infrastructure only: imported by
tests/, never by the library).

Source: "Wide-EP ... MoE ... NVIDIA" explainer, section "Load imbalance: EPLB" -- the
per-expert load decides where experts go, and the most loaded experts get copies on
several GPUs.  The page prints no algorithm; the reading implemented here (and by the
library) is the plain greedy one:

1. Replication.  Every expert starts with one copy.  While free slots remain, the expert
   with the largest load per copy (load / copies; ties: lower id) that has fewer than G
   copies gets one more.
2. Placement.  Copies, each carrying load / copies, are taken in descending load (ties:
   lower expert id, then lower copy index); each goes to the least loaded GPU (ties:
   lower GPU id) that has a free slot and no copy of the same expert.  An extra copy no
   GPU can take is dropped.
3. The GPU loads are the sums of load / (copies placed) over each GPU's copies.

Loads per copy are exact fractions here, so every comparison is exact.
"""
from fractions import Fraction


def eplb_plan(load, G: int, S: int):
    E = len(load)
    assert E >= 1 and G >= 1 and S >= 1 and E <= G * S
    assert all(int(v) >= 0 for v in load)
    load = [int(v) for v in load]

    # 1. replication
    copies = [1] * E
    free = G * S - E
    while free > 0:
        candidates = [e for e in range(E) if copies[e] < G]
        if not candidates:
            break
        best = candidates[0]
        for e in candidates[1:]:
            if Fraction(load[e], copies[e]) > Fraction(load[best], copies[best]):
                best = e
        copies[best] += 1
        free -= 1

    # 2. placement
    order = [(e, c) for e in range(E) for c in range(copies[e])]
    order.sort(key=lambda ec: (-Fraction(load[ec[0]], copies[ec[0]]), ec[0], ec[1]))
    gpu_slots = [[] for _ in range(G)]
    gpu_sum = [Fraction(0)] * G
    for e, _c in order:
        eligible = [g for g in range(G) if len(gpu_slots[g]) < S and e not in gpu_slots[g]]
        if not eligible:
            continue
        g = min(eligible, key=lambda q: (gpu_sum[q], q))
        gpu_slots[g].append(e)
        gpu_sum[g] += Fraction(load[e], copies[e])

    # 3. final loads from the copies actually placed
    placed = [sum(row.count(e) for row in gpu_slots) for e in range(E)]
    gpu_load = [sum((Fraction(load[e], placed[e]) for e in row), Fraction(0)) for row in gpu_slots]
    slot_expert = [row + [-1] * (S - len(row)) for row in gpu_slots]
    return slot_expert, placed, gpu_load
