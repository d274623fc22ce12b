"""Oracle for the query-aware anchor-KV cache plan. Test infrastructure.

Source: "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por GPU", section
"Como funciona", first bullet (the engine knows the whole query plan in advance, so it can
predict accesses, prefetch, and evict without regret - unlike agent workloads whose
access gaps are unpredictable), and "Quail, il motore di inferenza che supera il
miliardo di token al minuto su una H100", the paragraph on KV regret (a general server
discards key/value state that it needs later and so processes tokens it did not need).

Model (the plainest reading; the pages give no algorithm):
  * a plan is a sequence of accesses to anchors; anchor a's KV holds size[a] tokens; the
    GPU keeps at most `capacity` tokens of anchor KV;
  * an access to a resident anchor is a hit; otherwise its KV is prefilled (size[a]
    tokens): the first prefill of an anchor is compulsory, every later one is regret;
  * after a miss the anchor is inserted unless the policy bypasses it (or it is larger
    than the capacity), evicting residents until it fits.
Policies:
  * LRU (what a general server does): evict the resident with the oldest last access;
    always insert.
  * BELADY (query-aware, furthest next use): among the residents and the incoming anchor,
    repeatedly drop the one whose next access is furthest in the future (never = infinite;
    ties: larger size first, then larger anchor id); if the incoming anchor is dropped it
    is bypassed and nothing else is evicted.
`min_regret` is the exact minimum over every eviction/bypass choice (exhaustive search,
tiny plans only).
"""
from __future__ import annotations

import math

LRU, BELADY = 0, 1


def _next_use(accesses):
    nxt = [math.inf] * len(accesses)
    seen = {}
    for i in range(len(accesses) - 1, -1, -1):
        a = accesses[i]
        nxt[i] = seen.get(a, math.inf)
        seen[a] = i
    return nxt


def simulate(accesses, size, capacity, policy):
    """Returns (hits list of 0/1, compulsory tokens, regret tokens, peak resident tokens)."""
    nxt = _next_use(accesses)
    resident = {}          # anchor -> (last access index, next access index)
    used = 0
    seen = set()
    hits, compulsory, regret, peak = [], 0, 0, 0
    for i, a in enumerate(accesses):
        if a in resident:
            hits.append(1)
            resident[a] = (i, nxt[i])
            continue
        hits.append(0)
        if a in seen:
            regret += size[a]
        else:
            compulsory += size[a]
            seen.add(a)
        if size[a] > capacity:
            continue       # streamed: never resident
        if policy == LRU:
            while used + size[a] > capacity:
                victim = min(resident, key=lambda b: resident[b][0])
                used -= size[victim]
                del resident[victim]
            resident[a] = (i, nxt[i])
            used += size[a]
        else:
            cand = dict(resident)
            cand[a] = (i, nxt[i])
            free = capacity - used
            drop = []
            while free < size[a] and a not in drop:
                far = max(cand, key=lambda b: (cand[b][1], size[b], b))
                drop.append(far)
                del cand[far]
                if far != a:
                    free += size[far]
            if a in drop:
                continue   # bypass: nothing is evicted
            for b in drop:
                used -= size[b]
                del resident[b]
            resident[a] = (i, nxt[i])
            used += size[a]
        peak = max(peak, used)
    return hits, compulsory, regret, peak


def min_regret(accesses, size, capacity):
    """Exact minimum regret over all eviction and bypass choices (exhaustive; tiny plans)."""
    best = [math.inf]

    def rec(i, resident, seen, regret):
        if regret >= best[0]:
            return
        if i == len(accesses):
            best[0] = regret
            return
        a = accesses[i]
        if a in resident:
            rec(i + 1, resident, seen, regret)
            return
        r2 = regret + (size[a] if a in seen else 0)
        s2 = seen | {a}
        rec(i + 1, resident, s2, r2)            # bypass
        if size[a] > capacity:
            return
        res = sorted(resident)
        for mask in range(1 << len(res)):       # every set of victims that makes room
            keep = [b for k, b in enumerate(res) if not (mask >> k) & 1]
            if sum(size[b] for b in keep) + size[a] <= capacity:
                rec(i + 1, frozenset(keep) | {a}, s2, r2)

    rec(0, frozenset(), frozenset(), 0)
    return best[0]
