"""EPLB replica planner, oracle side -- TEST INFRASTRUCTURE ONLY.

Follows "xDeepServe on CloudMatrix384", section "专家负载均衡":
  P069-P075  greedy selection of redundant experts: the hot expert of time
             slice t is argmax_e token_count[e][t]; the layer's tail load is
             L = sum_t token_count[h_t][t]; each round, for every candidate
             (an expert that is the hot one of some slice) simulate splitting
             its tokens evenly over one more copy, keep the candidate with the
             smallest simulated L, and apply that split;
  P076       placement: sort the selected replicas by total load, heaviest
             first, and put each on the least-loaded rank that still has a
             free redundant slot, adding the replica's share to that rank;
  P078-P079  forward-time map physical(i, e) = R_e[i mod |R_e|].

Readings where the page is silent:
  - ties: lower expert id / lower rank id win;
  - a replica's share is total_load[e] / (number of instances of e), and a
    rank's starting load is the sum of the shares of its primary experts;
  - a rank that already hosts an instance of e is skipped while another rank
    with a free slot exists (the page replicates hot experts onto other NPUs);
  - R_e is listed in ascending physical id (matches the page's [4, 256]
    example, where logical expert 1 with primary slot 2 and redundant slot 1
    rotates 1, 2).
Physical layout: rank r owns slots r*epr .. r*epr+epr-1; its first E_log/R
slots hold logical experts r*(E_log/R) + m, the rest are redundant.
"""
from __future__ import annotations

import numpy as np


def select_replicas(token_count: np.ndarray, budget: int) -> tuple[list[int], np.ndarray]:
    """token_count: [n_slices, E_log].  Returns (replicas in selection order, copies[E_log])."""
    tc = np.asarray(token_count, dtype=np.float64)
    n_slices, E = tc.shape
    copies = np.ones(E, dtype=np.int64)
    sim = tc.copy()
    replicas: list[int] = []
    for _ in range(budget):
        cands = sorted({int(np.argmax(sim[t])) for t in range(n_slices)})
        best, best_tail = None, float("inf")
        for c in cands:
            trial = sim.copy()
            trial[:, c] = tc[:, c] / float(copies[c] + 1)
            tail = 0.0
            for t in range(n_slices):
                tail += float(np.max(trial[t]))
            if tail < best_tail:
                best, best_tail = c, tail
        if best is None:
            break
        replicas.append(best)
        copies[best] += 1
        sim[:, best] = tc[:, best] / float(copies[best])
    return replicas, copies


def place_replicas(token_count: np.ndarray, replicas: list[int], copies: np.ndarray,
                   E_phys: int, R: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Returns (rep_table [E_log, max_copies] padded with -1, n_copies [E_log],
    phys_to_logical [E_phys])."""
    tc = np.asarray(token_count, dtype=np.float64)
    E = tc.shape[1]
    total = [float(sum(tc[t, e] for t in range(tc.shape[0]))) for e in range(E)]
    ppr = E // R
    epr = E_phys // R
    rpr = epr - ppr
    phys_to_logical = np.full(E_phys, -1, dtype=np.int32)
    hosts = [set() for _ in range(R)]
    load = [0.0] * R
    for r in range(R):
        for m in range(ppr):
            e = r * ppr + m
            phys_to_logical[r * epr + m] = e
            hosts[r].add(e)
            load[r] += total[e] / float(copies[e])
    free = [rpr] * R
    ordered = sorted(replicas, key=lambda e: (-total[e], e))
    for e in ordered:
        elig = [r for r in range(R) if free[r] > 0 and e not in hosts[r]]
        if not elig:
            elig = [r for r in range(R) if free[r] > 0]
        tgt = min(elig, key=lambda r: (load[r], r))
        slot = tgt * epr + ppr + (rpr - free[tgt])
        free[tgt] -= 1
        phys_to_logical[slot] = e
        hosts[tgt].add(e)
        load[tgt] += total[e] / float(copies[e])
    n_copies = np.zeros(E, dtype=np.int32)
    lists: list[list[int]] = [[] for _ in range(E)]
    for p in range(E_phys):
        e = int(phys_to_logical[p])
        if e >= 0:
            lists[e].append(p)
    maxc = max(len(l) for l in lists)
    rep = np.full((E, maxc), -1, dtype=np.int32)
    for e in range(E):
        n_copies[e] = len(lists[e])
        rep[e, :len(lists[e])] = sorted(lists[e])
    return rep, n_copies, phys_to_logical


def plan(token_count: np.ndarray, E_phys: int, R: int):
    """Selection + placement.  token_count: [n_slices, E_log] (or [E_log])."""
    tc = np.atleast_2d(np.asarray(token_count, dtype=np.float64))
    E = tc.shape[1]
    if E % R or E_phys % R or E_phys < E:
        raise ValueError("eplb: E_log and E_phys must be multiples of R, E_phys >= E_log")
    replicas, copies = select_replicas(tc, E_phys - E)
    return place_replicas(tc, replicas, copies, E_phys, R)


def physical(i: int, e: int, rep_table: np.ndarray, n_copies: np.ndarray) -> int:
    """physical(i, e) = R_e[i mod |R_e|]."""
    return int(rep_table[e, i % int(n_copies[e])])
