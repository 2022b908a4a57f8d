"""Host simulation of the decode kernel's ticket protocol under adversarial routings.

Forward progress of the persistent expert kernels rests on the task order, not on grid
barriers ("Persistent execution for Flash-Next GGUF on SM70", section "First implementation
boundary"): every gate/up task precedes every down task, a down task waits only for the
gate/up tasks of its own expert, and an un-route task only for the down tasks of its stripe.
This test rebuilds the kernel's ticket order from a plan (gate/up tasks of 8-row passes,
down tasks of G stripes per ticket with the last grid-many tickets single stripes, trailing
un-route tasks), checks its invariants, and runs it on simulated CTAs that claim tickets in
order, take random times per chunk and block on their dependencies exactly where the kernel
does.  Every routing must finish with every task done; a deadlock would leave CTAs blocked.
"""
import heapq
import random

import numpy as np
import pytest

ROWS = 8  # routed rows per pass


def plan_passes(ids, E, rows=ROWS):
    counts = np.bincount(np.asarray(ids).reshape(-1), minlength=E)
    touched = [e for e in range(E) if counts[e] > 0]
    return [(e, (int(counts[e]) + rows - 1) // rows) for e in touched]


def ticket_order(passes, S_gu, S_dn, G, grid, T):
    """The kernel's tickets: ('gu', u, p, s) ..., ('dn', u, p, s0, g) ..., ('ur', block, stripe)."""
    gu, dn = [], []
    for u, (_, npass) in enumerate(passes):
        for p in range(npass):
            gu += [("gu", u, p, s) for s in range(S_gu)]
            dn += [("dn", u, p, s) for s in range(S_dn)]
    G = min(G, S_dn)
    ngroup = (len(dn) - min(len(dn), grid)) // G
    tickets = list(gu)
    for j in range(ngroup):
        first = dn[j * G]
        tickets.append(("dn", first[1], first[2], first[3], G))
    for entry in dn[ngroup * G:]:
        tickets.append(entry + (1,))
    blocks = (T + 7) // 8
    tickets += [("ur", c // S_dn, c % S_dn) for c in range(S_dn * blocks)]
    return tickets, ngroup


def check_order(tickets, passes, S_gu, S_dn):
    # a down ticket's stripes belong to one expert pass; every dependency has a lower ticket
    pos_gu = {}
    for i, t in enumerate(tickets):
        if t[0] == "gu":
            pos_gu.setdefault(t[1], []).append(i)
        elif t[0] == "dn":
            u, p, s0, g = t[1:]
            assert s0 % g == 0 and s0 + g <= S_dn, t
            before = pos_gu.get(u, [])  # the expert's gate/up tickets already in the order
            assert len(before) == passes[u][1] * S_gu, t
    covered = {}
    for t in tickets:
        if t[0] == "dn":
            for s in range(t[3], t[3] + t[4]):
                covered[(t[1], t[2], s)] = covered.get((t[1], t[2], s), 0) + 1
    assert all(v == 1 for v in covered.values())
    assert len(covered) == sum(n for _, n in passes) * S_dn


def simulate(tickets, passes, S_gu, S_dn, grid, chunks_gu, chunks_dn, rng):
    """Event simulation: CTA b starts with ticket b, then claims the next free ticket when its
    task's chunks are issued; a task runs once its dependency is met (a blocked CTA holds its
    ticket and blocks).  Returns (all done, finish time)."""
    n = len(tickets)
    ready = [0] * len(passes)           # gate/up tasks published per touched expert
    need = [npass * S_gu for _, npass in passes]
    dn_done = [0] * S_dn                # down stripes published per stripe
    dn_need = sum(npass for _, npass in passes)
    nxt = grid
    done = 0
    blocked = []                        # (cta, ticket) waiting on a counter
    events = []                         # (time, cta, ticket finished)
    t_now = 0.0

    def dep_met(t):
        if t[0] == "dn":
            return ready[t[1]] >= need[t[1]]
        if t[0] == "ur":
            return dn_done[t[2]] >= dn_need
        return True

    def start(cta, i, now):
        t = tickets[i]
        if t[0] == "gu":
            dur = sum(rng.uniform(0.5, 1.5) for _ in range(chunks_gu))
        elif t[0] == "dn":
            dur = sum(rng.uniform(0.5, 1.5) for _ in range(chunks_dn * t[4]))
        else:
            dur = rng.uniform(0.5, 1.5)
        heapq.heappush(events, (now + dur, cta, i))

    for b in range(min(grid, n)):
        if dep_met(tickets[b]):
            start(b, b, 0.0)
        else:
            blocked.append((b, b))
    while events:
        t_now, cta, i = heapq.heappop(events)
        t = tickets[i]
        done += 1
        if t[0] == "gu":
            ready[t[1]] += 1
        elif t[0] == "dn":
            for s in range(t[3], t[3] + t[4]):
                dn_done[s] += 1
        # blocked CTAs whose counter is now met resume
        still = []
        for bc, bi in blocked:
            if dep_met(tickets[bi]):
                start(bc, bi, t_now)
            else:
                still.append((bc, bi))
        blocked = still
        if nxt < n:
            j, nxt = nxt, nxt + 1
            if dep_met(tickets[j]):
                start(cta, j, t_now)
            else:
                blocked.append((cta, j))
    return done == n and not blocked, t_now


def routings(T, E, k, rng):
    yield "random", np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    yield "all_same", np.tile(np.arange(k), (T, 1))                       # every token on the same k experts
    yield "disjoint", np.stack([(np.arange(k) + t * k) % E for t in range(T)])
    hot = np.stack([np.concatenate(([0], rng.choice(np.arange(1, E), k - 1, replace=False))) for _ in range(T)])
    yield "one_hot_expert", hot                                           # expert 0 in every token: T rows
    pz = 1.0 / np.arange(1, E + 1) ** 1.1
    pz /= pz.sum()
    yield "zipf", np.stack([rng.choice(E, k, replace=False, p=pz) for _ in range(T)])  # a few hot experts


@pytest.mark.parametrize("T,E,k,grid,G", [(4, 512, 10, 152, 2), (32, 512, 10, 152, 4), (256, 512, 10, 152, 4),
                                          (8, 8, 8, 152, 2), (64, 16, 16, 20, 4), (1, 512, 10, 152, 2),
                                          (128, 64, 8, 7, 4)])
def test_ticket_order_invariants_and_forward_progress(T, E, k, grid, G):
    rng = np.random.default_rng(T * 1000 + E + k)
    S_gu, S_dn = 8, 16
    for name, ids in routings(T, E, k, rng):
        assert ids.shape == (T, k) and all(len(set(r)) == k for r in ids.tolist()), name
        passes = plan_passes(ids, E)
        tickets, _ = ticket_order(passes, S_gu, S_dn, G, grid, T)
        check_order(tickets, passes, S_gu, S_dn)
        for seed in range(3):
            ok, _ = simulate(tickets, passes, S_gu, S_dn, grid, 8, 2, random.Random(seed))
            assert ok, (name, seed)


def test_simulation_detects_a_broken_order():
    # the model must fail where the protocol would: a down ticket placed before the gate/up
    # tickets of its expert, with fewer CTAs than blocked down tasks, never finishes
    T, E, k, grid = 16, 16, 4, 2
    ids = np.tile(np.arange(k), (T, 1))
    passes = plan_passes(ids, E)
    tickets, _ = ticket_order(passes, 2, 4, 2, grid, T)
    gu = [t for t in tickets if t[0] == "gu"]
    dn = [t for t in tickets if t[0] == "dn"]
    ur = [t for t in tickets if t[0] == "ur"]
    with pytest.raises(AssertionError):
        check_order(dn + gu + ur, passes, 2, 4)
    ok, _ = simulate(dn + gu + ur, passes, 2, 4, grid, 8, 2, random.Random(0))
    assert not ok


@pytest.mark.parametrize("T,E,k,grid", [(2048, 64, 8, 152), (512, 16, 4, 152), (4096, 512, 10, 152), (1024, 32, 8, 5)])
def test_wide_kernel_ticket_order_forward_progress(T, E, k, grid):
    # the wide kernel's order: passes of up to 192 routed rows, every gate/up task (touched,
    # pass, stripe) before every down task, one stripe per down ticket, no un-route tasks; a
    # down task waits for every gate/up stripe of all passes of its expert
    rng = np.random.default_rng(T + E + k)
    S_gu, S_dn = 8, 16
    for name, ids in routings(T, E, k, rng):
        passes = plan_passes(ids, E, rows=192)
        tickets, ngroup = ticket_order(passes, S_gu, S_dn, 1, grid, 0)
        assert ngroup == sum(n for _, n in passes) * S_dn - min(sum(n for _, n in passes) * S_dn, grid)
        assert not any(t[0] == "ur" for t in tickets)
        check_order(tickets, passes, S_gu, S_dn)
        ok, _ = simulate(tickets, passes, S_gu, S_dn, grid, 16, 4, random.Random(1))
        assert ok, name
