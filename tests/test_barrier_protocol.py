"""Host model of the mbarrier protocols of the three tensor-core kernels.

Each role (TMA producer, MMA issuer, elementwise / softmax warpgroups) is written as the
sequence of barrier operations its loop performs, in the order of the kernel source.  Arrivals
that the hardware makes asynchronously (a TMA copy completing, a ``tcgen05.commit`` firing when
the MMAs before it finish) become pending events that a random scheduler delivers later; commit
arrivals of one issuer keep their order, as MMAs complete in issue order.

A wait is ``mbarrier.try_wait.parity``: it passes when the barrier's current phase parity
differs from the parity asked for.  The model flags
  * a wait that passes while the barrier is not exactly one phase past the one the role wants
    (a missed or an early phase: the parity test cannot tell them apart),
  * an arrival, where the model names the phase it is meant for, that lands in another phase
    (on a barrier that several roles arrive at, one role running ahead could complete an
    earlier phase in place of another), and
  * a schedule in which no role can move while some have not finished (deadlock), and
  * in models that track a buffer's contents (a TMEM region several products take turns in):
    a product issued into the buffer while some reader has not released its previous contents,
    or a read that finds other contents than the role expects.
Random schedules explore the interleavings that the kernels' timing normally hides; the dQ
kernel's dS barrier was a single barrier per warpgroup until this model (and a variant that
moved the K/V waits) showed that the warpgroups can complete two of its phases before the MMA
warp waits for the first; it is now one barrier per block parity.
"""
from __future__ import annotations

import random

import pytest

# ----------------------------------------------------------------------------- engine

W, A, C = "wait", "arrive", "commit"  # C: asynchronous arrive (TMA completion or tcgen05.commit)
# Buffer contents: WR (buffer, label, readers) when a product into the buffer is issued (the
# earliest moment it may write), RD (buffer, label) when a role reads it, RL (buffer) when that
# role is done with it.
WR, RD, RL = "write", "read", "release"


class Hazard(AssertionError):
    pass


def run(progs: dict, counts: dict, rng: random.Random) -> None:
    done = {b: 0 for b in counts}      # completed phases
    pend = {b: 0 for b in counts}      # arrivals in the current phase
    pc = {r: 0 for r in progs}
    asyncq = {r: [] for r in progs}    # in-order asynchronous arrivals issued by each role
    bufs = {}                          # buffer -> [label, readers not yet released]

    def arrive(b, ph=None):
        if ph is not None and done[b] != ph:
            raise Hazard(f"arrival for phase {ph} of {b} landed in phase {done[b]}")
        pend[b] += 1
        if pend[b] == counts[b]:
            pend[b] = 0
            done[b] += 1

    while True:
        moves = []
        for r, prog in progs.items():
            if pc[r] < len(prog):
                op, b, *k = prog[pc[r]]
                if op != W or (done[b] & 1) != (k[0] & 1):
                    moves.append(("step", r))
            if asyncq[r]:
                moves.append(("async", r))
        if not moves:
            stuck = {r: progs[r][pc[r]] for r in progs if pc[r] < len(progs[r])}
            if stuck:
                raise Hazard(f"deadlock: {stuck}")
            return
        kind, r = rng.choice(moves)
        if kind == "async":
            arrive(*asyncq[r].pop(0))
            continue
        op, b, *k = progs[r][pc[r]]
        pc[r] += 1
        if op == WR:
            if bufs.get(b, [None, 0])[1] > 0:
                raise Hazard(f"{r}: {k[0]} issued into {b} while {bufs[b][0]} is unread")
            bufs[b] = [k[0], k[1]]
        elif op == RD:
            if bufs.get(b, [None])[0] != k[0]:
                raise Hazard(f"{r}: read {k[0]} from {b}, which holds {bufs.get(b, [None])[0]}")
        elif op == RL:
            bufs[b][1] -= 1
        elif op == W:
            if done[b] != k[0] + 1:
                raise Hazard(f"{r}: wait for phase {k[0]} of {b} passed with {done[b]} completed")
        elif op == A:
            arrive(b, *k)
        else:
            asyncq[r].append((b, *k))


# ----------------------------------------------------------------------------- dQ kernel

def dq_protocol(n, ks=3, vs=2, e_per_parity=True, kv_waits_first=False, groups=4):
    """fa_bwd_dq_tc_kernel: producer (V then K per block), MMA issuer, `groups` elementwise
    warpgroups that all arrive on one dS barrier per block parity (each warpgroup is one actor
    here: its warps' arrivals come after the same waits)."""
    prod, mma = [], []
    for j in range(n):
        if j >= vs:
            prod.append((W, ("vempty", j % vs), j // vs - 1))
        prod.append((C, ("vfull", j % vs)))
        if j >= ks:
            prod.append((W, ("kempty", j % ks), j // ks - 1))
        prod.append((C, ("kfull", j % ks)))
    wk = lambda j: (W, ("kfull", j % ks), j // ks)  # noqa: E731
    wv = lambda j: (W, ("vfull", j % vs), j // vs)  # noqa: E731
    ebar = (lambda j: (("e", j & 1), j >> 1)) if e_per_parity else (lambda j: (("e", 0), j))

    def dp(j):
        return [(C, ("dp", j & 1)), (C, ("vempty", j % vs))]

    def s(j):
        return ([(W, "sfree", j - 1)] if j > 0 else []) + [(C, "s")]

    mma += [wk(0), wv(0)] + s(0) + dp(0)
    if n > 1:
        mma += [wv(1)] + dp(1) + [wk(1)] + s(1)
    for it in range(n):
        if kv_waits_first and it + 2 < n:
            mma += [wv(it + 2), wk(it + 2)]
        b, k = ebar(it)
        mma.append((W, b, k))
        mma.append((C, ("kempty", it % ks)))
        if it + 2 < n:
            if not kv_waits_first:
                mma.append(wv(it + 2))
            mma += dp(it + 2)
            if not kv_waits_first:
                mma += [(W, "sfree", it + 1), wk(it + 2), (C, "s")]
            else:
                mma += s(it + 2)
    progs = {"producer": prod, "mma": mma}
    for h in range(groups):
        g = []
        for j in range(n):
            b, _ = ebar(j)
            g += [(W, "s", j), (A, "sfree"), (W, ("dp", j & 1), j >> 1), (A, b)]
        progs[f"wg{h}"] = g
    counts = {"s": 1, "sfree": groups, ("dp", 0): 1, ("dp", 1): 1}
    counts |= {(x, i): 1 for x in ("vfull", "vempty") for i in range(vs)}
    counts |= {(x, i): 1 for x in ("kfull", "kempty") for i in range(ks)}
    counts |= {("e", b): groups for b in (0, 1)}
    return progs, counts


def dq_persistent_protocol(tiles, ks=3, vs=2, groups=4, use_of=lambda o: (o - 1) >> 1,
                           qfree_commits=True):
    """The persistent dQ kernel over a sequence of work tiles (key-block counts, 0 for a tile
    without keys): the producer loads each tile's Q/dO once the previous tile's S and dP products
    ran (qfree), streams K/V through the rings with block indices counted over the whole
    sequence, then requests the next tile (cluster launch control; the response arrives
    asynchronously) and publishes its index in a two-slot queue; the MMA warp and the elementwise
    groups read every index and release its slot; the accumulator barrier completes once per
    tile with keys."""
    prod, mma = [], []
    wk = lambda j: (W, ("kfull", j % ks), j // ks)  # noqa: E731
    wv = lambda j: (W, ("vfull", j % vs), j // vs)  # noqa: E731

    def dp(j):
        return [wv(j), (C, ("dp", j & 1)), (C, ("vempty", j % vs))]

    def s(j):
        return ([(W, "sfree", j - 1)] if j > 0 else []) + [wk(j), (C, "s")]

    # ordinal o >= 1 is use (o - 1) >> 1 of queue slot o & 1 (and of response slot o & 1)
    def take(ti):  # consumers: read the index of ordinal ti + 1, release its slot
        o = ti + 1
        return [(W, ("tfull", o & 1), use_of(o)), (A, ("tempty", o & 1))]

    g = at = 0
    for ti, n in enumerate(tiles):
        if n > 0:
            if at > 0:
                prod.append((W, "qfree", at - 1))
            prod.append((C, "res"))
            for it in range(n):
                j = g + it
                if j >= vs:
                    prod.append((W, ("vempty", j % vs), j // vs - 1))
                prod.append((C, ("vfull", j % vs)))
                if j >= ks:
                    prod.append((W, ("kempty", j % ks), j // ks - 1))
                prod.append((C, ("kfull", j % ks)))
            g += n
            at += 1
        o = ti + 1
        # the next tile is requested after this tile's loads; the response lands asynchronously
        prod += [(C, "clc"), (W, "clc", ti)]
        if use_of(o) > 0:
            prod.append((W, ("tempty", o & 1), use_of(o) - 1))
        prod.append((A, ("tfull", o & 1)))
    g = at = 0
    for ti, n in enumerate(tiles):
        if n > 0:
            mma.append((W, "res", at))
            mma += s(g) + dp(g)
            if n > 1:
                mma += dp(g + 1) + s(g + 1)
            if n <= 2 and qfree_commits:
                mma.append((C, "qfree"))
            for it in range(n):
                j = g + it
                mma += [(W, ("e", j & 1), j >> 1), (C, ("kempty", j % ks))]
                if it + 2 < n:
                    mma += dp(j + 2) + s(j + 2)
                    if it + 3 == n and qfree_commits:
                        mma.append((C, "qfree"))
            mma.append((C, "acc"))
            g += n
            at += 1
        mma += take(ti)
    progs = {"producer": prod, "mma": mma}
    for h in range(groups):
        prog, g, at = [], 0, 0
        for ti, n in enumerate(tiles):
            for it in range(n):
                j = g + it
                prog += [(W, "s", j), (A, "sfree"), (W, ("dp", j & 1), j >> 1), (A, ("e", j & 1))]
            prog += take(ti)
            if n > 0:
                prog.append((W, "acc", at))
                g += n
                at += 1
        progs[f"wg{h}"] = prog
    counts = {"s": 1, "sfree": groups, ("dp", 0): 1, ("dp", 1): 1, "acc": 1, "res": 1, "qfree": 1}
    counts |= {(x, i): 1 for x in ("vfull", "vempty") for i in range(vs)}
    counts |= {(x, i): 1 for x in ("kfull", "kempty") for i in range(ks)}
    counts |= {("e", b): groups for b in (0, 1)}
    counts |= {("tfull", b): 1 for b in (0, 1)}
    counts["clc"] = 1
    counts |= {("tempty", b): groups + 1 for b in (0, 1)}
    return progs, counts


# ----------------------------------------------------------------------------- dK/dV kernel

def dkv_protocol(n, qs=3, gs=2, groups=2, chunks=2):
    """fa_bwd_dkv_tc_kernel: producer (Q then dO per block), MMA issuer, `groups` elementwise
    warpgroups that each signal their columns in `chunks` chunks, chunk x on barrier x, which
    every warpgroup arrives on."""
    prod, mma = [], []
    for j in range(n):
        if j >= qs:
            prod.append((W, ("qempty", j % qs), j // qs - 1))
        prod.append((C, ("qfull", j % qs)))
        if j >= gs:
            prod.append((W, ("gempty", j % gs), j // gs - 1))
        prod.append((C, ("gfull", j % gs)))
    wq = lambda j: (W, ("qfull", j % qs), j // qs)  # noqa: E731
    wg = lambda j: (W, ("gfull", j % gs), j // gs)  # noqa: E731
    mma += [wq(0), (C, "s"), wg(0), (C, "dp")]
    for it in range(n):
        mma += [(W, ("p", x), it) for x in range(chunks)] + [(C, ("gempty", it % gs))]
        if it + 1 < n:
            mma += [wq(it + 1), (C, "s")]
        mma += [(W, ("e", x), it) for x in range(chunks)] + [(C, ("qempty", it % qs))]
        if it + 1 < n:
            mma += [wg(it + 1), (C, "dp")]
    progs = {"producer": prod, "mma": mma}
    for h in range(groups):
        progs[f"wg{h}"] = [x for j in range(n)
                           for x in ([(W, "s", j)] + [(A, ("p", c)) for c in range(chunks)] +
                                     [(W, "dp", j)] + [(A, ("e", c)) for c in range(chunks)])]
    counts = {"s": 1, "dp": 1}
    counts |= {(x, c): groups for x in ("p", "e") for c in range(chunks)}
    counts |= {(x, i): 1 for x in ("qfull", "qempty") for i in range(qs)}
    counts |= {(x, i): 1 for x in ("gfull", "gempty") for i in range(gs)}
    return progs, counts


# ----------------------------------------------------------------------------- forward kernel

def fwd_protocol(j0, j1, stages=2, split=True):
    """fa_fwd_tc_kernel: producer (K then V per block), MMA issuer, one softmax group per tile.
    split: P signalled in two halves (d = 64, e4m3), else at once (bf16, d = 128)."""
    halves = (0, 1) if split else (1,)
    jmax = max(j0, j1)
    jt = (j0, j1)
    prod = [(C, "q")]
    for j in range(jmax):
        if j >= stages:
            prod.append((W, ("kempty", j % stages), j // stages - 1))
        prod.append((C, ("kfull", j % stages)))
        if j >= stages:
            prod.append((W, ("vempty", j % stages), j // stages - 1))
        prod.append((C, ("vfull", j % stages)))
    wk = lambda j: (W, ("kfull", j % stages), j // stages)  # noqa: E731
    mma = [(W, "q", 0), wk(0)]
    for t in (0, 1):
        if jt[t] > 0:
            mma.append((C, ("sfull", t)))
    mma.append((C, ("kempty", 0)))
    for j in range(jmax):
        mma.append((W, ("vfull", j % stages), j // stages))
        k_next = False
        for t in (0, 1):
            if j < jt[t]:  # the P V product in halves, each after its half of P
                mma += [(W, ("pfull", t, x), j) for x in halves]
                if j + 1 == jt[t]:
                    mma.append((C, ("ofinal", t)))
                else:
                    if not k_next:
                        mma.append(wk(j + 1))
                    k_next = True
                    mma.append((C, ("sfull", t)))
        if k_next:
            mma.append((C, ("kempty", (j + 1) % stages)))
        mma.append((C, ("vempty", j % stages)))
    progs = {"producer": prod, "mma": mma}
    for t in (0, 1):
        g = []
        for j in range(jt[t]):
            g += [(W, ("sfull", t), j)] + [(A, ("pfull", t, x)) for x in halves]
        if jt[t] > 0:
            g.append((W, ("ofinal", t), 0))
        progs[f"softmax{t}"] = g
    counts = {"q": 1}
    counts |= {(x, i): 1 for x in ("kfull", "kempty", "vfull", "vempty") for i in range(stages)}
    counts |= {(x, t): 1 for x in ("sfull", "ofinal") for t in (0, 1)}
    counts |= {("pfull", t, x): 1 for t in (0, 1) for x in (0, 1)}
    return progs, counts


def fwd_persistent_protocol(tiles, stages=2, split=True):
    """The persistent forward over a sequence of query-tile pairs, each given as (J0, J1), the key
    blocks its two query tiles visit (0 for an empty slot or a tile that sees no key).  K/V blocks
    are counted over the whole sequence for the rings; each query-tile slot counts its own S
    products for its S and P barriers and its finished pairs for its O barrier; the producer loads
    a pair's Q tiles once the previous pair's S products have run (qfree); tile indices go through
    the two-slot queue as in the backward.  Releases of the K / V ring stages name their
    phase."""
    halves = (0, 1) if split else (1,)
    wk = lambda j: (W, ("kfull", j % stages), j // stages)  # noqa: E731

    def take(ti):
        o = ti + 1
        return [(W, ("tfull", o & 1), (o - 1) >> 1), (A, ("tempty", o & 1))]

    prod, mma = [], []
    gk = at = 0
    for ti, (j0, j1) in enumerate(tiles):
        jmax = max(j0, j1)
        if jmax > 0:
            if at > 0:
                prod.append((W, "qfree", at - 1))
            prod.append((C, "q"))
            for j in range(gk, gk + jmax):
                if j >= stages:
                    prod.append((W, ("kempty", j % stages), j // stages - 1))
                prod.append((C, ("kfull", j % stages)))
                if j >= stages:
                    prod.append((W, ("vempty", j % stages), j // stages - 1))
                prod.append((C, ("vfull", j % stages)))
            gk += jmax
            at += 1
        o = ti + 1
        prod += [(C, "clc"), (W, "clc", ti)]
        if (o - 1) >> 1 > 0:
            prod.append((W, ("tempty", o & 1), ((o - 1) >> 1) - 1))
        prod.append((A, ("tfull", o & 1)))
    gk = at = 0
    cs = [0, 0]
    for ti, (j0, j1) in enumerate(tiles):
        jt = (j0, j1)
        jmax = max(jt)
        if jmax > 0:
            mma += [(W, "q", at), wk(gk)]
            for t in (0, 1):
                if jt[t] > 0:
                    mma.append((C, ("sfull", t)))
            mma.append((C, ("kempty", gk % stages), gk // stages))
            if jmax == 1:
                mma.append((C, "qfree"))
            for j in range(jmax):
                gj = gk + j
                mma.append((W, ("vfull", gj % stages), gj // stages))
                k_next = False
                for t in (0, 1):
                    if j < jt[t]:
                        mma += [(W, ("pfull", t, x), cs[t] + j) for x in halves]
                        if j + 1 == jt[t]:
                            mma.append((C, ("ofinal", t)))
                        else:
                            if not k_next:
                                mma.append(wk(gj + 1))
                            k_next = True
                            mma.append((C, ("sfull", t)))
                if k_next:
                    mma.append((C, ("kempty", (gj + 1) % stages), (gj + 1) // stages))
                if j + 2 == jmax:
                    mma.append((C, "qfree"))
                mma.append((C, ("vempty", gj % stages), gj // stages))
            cs = [cs[0] + j0, cs[1] + j1]
            gk += jmax
            at += 1
        mma += take(ti)
    progs = {"producer": prod, "mma": mma}
    for t in (0, 1):
        g, c, co = [], 0, 0
        for ti, jts in enumerate(tiles):
            for j in range(jts[t]):
                g += [(W, ("sfull", t), c + j)] + [(A, ("pfull", t, x)) for x in halves]
            g += take(ti)
            if jts[t] > 0:
                g.append((W, ("ofinal", t), co))
                c += jts[t]
                co += 1
        progs[f"softmax{t}"] = g
    counts = {"q": 1, "qfree": 1, "clc": 1}
    counts |= {(x, i): 1 for x in ("kfull", "kempty", "vfull", "vempty") for i in range(stages)}
    counts |= {(x, t): 1 for x in ("sfull", "ofinal") for t in (0, 1)}
    counts |= {("pfull", t, x): 1 for t in (0, 1) for x in (0, 1)}
    counts |= {("tfull", b): 1 for b in (0, 1)}
    counts |= {("tempty", b): 3 for b in (0, 1)}  # both softmax groups and the MMA warp
    return progs, counts


def dkv_persistent_protocol(tiles, qs=3, gs=2, s_waits_p=True):
    """The persistent dK/dV kernel over a sequence of key-block tiles (streamed query blocks per
    tile): K/V resident per tile and reloaded once its S^T and dP^T products have run (kvfree);
    Q/dO rings and per-block barriers counted over the whole sequence.  The TMEM buffers X (S^T,
    then P^T over it) and Y (dP^T, then dS^T) are tracked: S^T(j+1) may only be issued once
    both groups have turned S^T(j) into P^T (s_waits_p=False issues it before that wait)."""
    def take(ti):
        o = ti + 1
        return [(W, ("tfull", o & 1), (o - 1) >> 1), (A, ("tempty", o & 1))]

    wq = lambda j: (W, ("qfull", j % qs), j // qs)  # noqa: E731
    wg = lambda j: (W, ("gfull", j % gs), j // gs)  # noqa: E731
    prod, mma = [], []
    g = at = 0
    for ti, n in enumerate(tiles):
        if n > 0:
            if at > 0:
                prod.append((W, "kvfree", at - 1))
            prod.append((C, "res"))
            for j in range(g, g + n):
                if j >= qs:
                    prod.append((W, ("qempty", j % qs), j // qs - 1))
                prod.append((C, ("qfull", j % qs)))
                if j >= gs:
                    prod.append((W, ("gempty", j % gs), j // gs - 1))
                prod.append((C, ("gfull", j % gs)))
            g += n
            at += 1
        o = ti + 1
        prod += [(C, "clc"), (W, "clc", ti)]
        if (o - 1) >> 1 > 0:
            prod.append((W, ("tempty", o & 1), ((o - 1) >> 1) - 1))
        prod.append((A, ("tfull", o & 1)))
    g = at = 0
    for ti, n in enumerate(tiles):
        if n > 0:
            mma += [(W, "res", at), wq(g), (WR, "X", ("S", g), 2), (C, "s"), wg(g),
                    (WR, "Y", ("dP", g), 2), (C, "dp")]
            if n == 1:
                mma.append((C, "kvfree"))
            for it in range(n):
                j = g + it
                s_next = [wq(j + 1), (WR, "X", ("S", j + 1), 2), (C, "s")] if it + 1 < n else []
                if not s_waits_p:
                    mma += s_next
                mma += [(W, ("p", 0), j), (W, ("p", 1), j), (C, ("gempty", j % gs))]
                if s_waits_p:
                    mma += s_next
                mma += [(W, ("e", 0), j), (W, ("e", 1), j), (C, ("qempty", j % qs))]
                if it + 1 < n:
                    mma += [wg(j + 1), (WR, "Y", ("dP", j + 1), 2), (C, "dp")]
                    if it + 2 == n:
                        mma.append((C, "kvfree"))
            mma.append((C, "acc"))
            g += n
            at += 1
        mma += take(ti)
    progs = {"producer": prod, "mma": mma}
    for h in (0, 1):
        prog, g, at = [], 0, 0
        for ti, n in enumerate(tiles):
            for j in range(g, g + n):
                # each group loads its columns, writes its half-results back, then signals
                prog += [(W, "s", j), (RD, "X", ("S", j)), (A, ("p", 0)), (RL, "X"), (A, ("p", 1)),
                         (W, "dp", j), (RD, "Y", ("dP", j)), (A, ("e", 0)), (RL, "Y"),
                         (A, ("e", 1))]
            prog += take(ti)
            if n > 0:
                prog.append((W, "acc", at))
                g += n
                at += 1
        progs[f"wg{h}"] = prog
    counts = {"s": 1, "dp": 1, "acc": 1, "res": 1, "kvfree": 1, "clc": 1}
    counts |= {(x, c): 2 for x in ("p", "e") for c in (0, 1)}
    counts |= {(x, i): 1 for x in ("qfull", "qempty") for i in range(qs)}
    counts |= {(x, i): 1 for x in ("gfull", "gempty") for i in range(gs)}
    counts |= {("tfull", b): 1 for b in (0, 1)}
    counts |= {("tempty", b): 3 for b in (0, 1)}  # both elementwise groups and the MMA warp
    return progs, counts


# ----------------------------------------------------------------------------- decode kernel

def decode_protocol(J, stages=3):
    """fa_decode_split_kernel: producer (Q, then K and V per block), MMA issuer with two S
    buffers, one softmax group; block jj's softmax waits for the P V product of block jj-1."""
    prod = [(C, "q")]
    for j in range(J):
        if j >= stages:
            prod.append((W, ("kempty", j % stages), j // stages - 1))
        prod.append((C, ("kfull", j % stages)))
        if j >= stages:
            prod.append((W, ("vempty", j % stages), j // stages - 1))
        prod.append((C, ("vfull", j % stages)))
    mma = []
    if J > 0:
        mma += [(W, "q", 0), (W, ("kfull", 0), 0), (C, ("sfull", 0)), (C, ("kempty", 0))]
    for j in range(J):
        if j + 1 < J:
            s1 = (j + 1) % stages
            mma += [(W, ("kfull", s1), (j + 1) // stages), (C, ("sfull", (j + 1) & 1)),
                    (C, ("kempty", s1))]
        mma += [(W, "pfull", j), (W, ("vfull", j % stages), j // stages), (C, "pv"),
                (C, ("vempty", j % stages))]
    soft = []
    for j in range(J):
        soft.append((W, ("sfull", j & 1), j >> 1))
        if j > 0:
            soft.append((W, "pv", j - 1))
        soft.append((A, "pfull"))
    if J > 0:
        soft.append((W, "pv", J - 1))
    progs = {"producer": prod, "mma": mma, "softmax": soft}
    counts = {"q": 1, "pfull": 1, "pv": 1, ("sfull", 0): 1, ("sfull", 1): 1}
    counts |= {(x, i): 1 for x in ("kfull", "kempty", "vfull", "vempty") for i in range(stages)}
    return progs, counts


# ----------------------------------------------------------------------------- tests

SCHEDULES = 300


def explore(make, seeds=SCHEDULES):
    for seed in range(seeds):
        progs, counts = make()
        run(progs, counts, random.Random(seed))


@pytest.mark.parametrize("groups", [2, 4])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7])
def test_dq_protocol(n, groups):
    explore(lambda: dq_protocol(n, groups=groups))


@pytest.mark.parametrize("tiles", [[1], [3], [1, 1, 1], [2, 5], [0, 3, 0, 0, 1], [4, 1, 2, 3, 1],
                                   [1, 2, 1, 2, 1, 2, 1]])
def test_dq_persistent_protocol(tiles):
    explore(lambda: dq_persistent_protocol(tiles))


def test_persistent_model_catches_a_missing_qfree_commit():
    """Without the MMA warp's commit after a tile's last S and dP products, the producer never
    loads the next tile's Q and dO: the model must report the deadlock."""
    with pytest.raises(Hazard, match="deadlock"):
        explore(lambda: dq_persistent_protocol([3, 3], qfree_commits=False), seeds=5)


def test_persistent_model_catches_a_slot_phase_off_by_one():
    """Ordinal o is use (o - 1) >> 1 of its slot: counting it as use o >> 1 makes the first use
    of slot 0 wait for a parity that a fresh barrier already shows as complete, so a consumer
    could read a tile index before it is written."""
    with pytest.raises(Hazard):
        explore(lambda: dq_persistent_protocol([1, 1, 1, 1], use_of=lambda o: o >> 1))


@pytest.mark.parametrize("groups,chunks", [(2, 2), (4, 1)])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7])
def test_dkv_protocol(n, groups, chunks):
    explore(lambda: dkv_protocol(n, groups=groups, chunks=chunks))


@pytest.mark.parametrize("stages,split", [(2, False), (4, True)])  # bf16 d = 128; d = 64, e4m3
@pytest.mark.parametrize("j0,j1", [(1, 1), (1, 2), (2, 3), (3, 3), (4, 5), (0, 1), (6, 7)])
def test_fwd_protocol(j0, j1, stages, split):
    explore(lambda: fwd_protocol(j0, j1, stages, split))


@pytest.mark.parametrize("stages,split", [(2, False), (4, True)])
@pytest.mark.parametrize("tiles", [[(1, 1)], [(3, 4)], [(1, 2), (2, 3), (1, 0)], [(0, 0), (2, 2), (0, 1)],
                                   [(4, 5), (1, 1), (3, 3), (2, 0)], [(1, 1)] * 6,
                                   [(6, 7), (2, 3), (5, 5)]])
def test_fwd_persistent_protocol(tiles, stages, split):
    explore(lambda: fwd_persistent_protocol(tiles, stages, split), seeds=150)



@pytest.mark.parametrize("tiles", [[1], [3], [2, 1, 2], [0, 4, 0, 1], [5, 2, 3, 1], [1] * 6])
def test_dkv_persistent_protocol(tiles):
    explore(lambda: dkv_persistent_protocol(tiles))


def test_dkv_model_catches_s_over_an_unread_buffer():
    """S^T of the next block issued before both groups have read S^T and written P^T: the
    product may overwrite the buffer they still read."""
    with pytest.raises(Hazard, match="unread"):
        explore(lambda: dkv_persistent_protocol([4, 3], s_waits_p=False))


@pytest.mark.parametrize("stages", [3, 6])  # d = 128 and d = 64
@pytest.mark.parametrize("J", [0, 1, 2, 3, 5, 8])
def test_decode_protocol(J, stages):
    explore(lambda: decode_protocol(J, stages))


def test_model_catches_a_barrier_two_phases_ahead():
    """The dQ protocol with a single dS barrier (instead of one per block parity) lets the
    elementwise warps complete block j+1 before the MMA warp waits for block j: the model must
    find that schedule."""
    with pytest.raises(Hazard):
        explore(lambda: dq_protocol(6, e_per_parity=False))


def test_model_catches_a_deadlock():
    """A producer that waits for the release of the stage it is about to fill deadlocks."""
    progs = {"producer": [(W, "empty", 0), (C, "full")], "consumer": [(W, "full", 0), (C, "empty")]}
    with pytest.raises(Hazard, match="deadlock"):
        run(progs, {"empty": 1, "full": 1}, random.Random(0))


def test_model_catches_an_arrival_in_the_wrong_phase():
    """Two roles release a barrier of count 2 once per phase; one that releases two phases
    without waiting completes the first phase in place of the other role."""
    progs = {"fast": [(A, "bar", 0), (A, "bar", 1), (A, "go")],
             "slow": [(W, "go", 0), (A, "bar", 0), (A, "bar", 1)]}
    with pytest.raises(Hazard, match="landed in phase"):
        run(progs, {"bar": 2, "go": 1}, random.Random(0))
