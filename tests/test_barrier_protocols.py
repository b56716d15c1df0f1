"""The mbarrier protocols of the two attention kernels (csrc/attn_fwd.cu,
csrc/attn_bwd.cu), checked on the CPU by exploring interleavings.

Each role of a kernel (the TMA producer, the MMA issuer, the softmax or
compute warpgroups, in the forward the prep warps of the Q prologue, and in
the backward the dQ reducer and the row warp) is
written here as its sequence of barrier operations and shared-memory / TMEM
accesses, in the kernel's order.  Asynchronous work is modelled by agents
that the scheduler may delay arbitrarily:

  - a TMA load writes its tile and then completes its barrier, at any time;
  - a tcgen05.mma runs at any time after its issue; MMAs into the same
    accumulator run in issue order, other MMAs in any order (the PTX rule:
    only MMAs into the same accumulator are implicitly pipelined);
  - a tcgen05.commit arrives once every MMA issued before it has run.

Barriers follow the hardware's parity rule: a wait for phase k (parity
k & 1) passes while the number of completed phases c has the other parity.
Vector clocks carry happens-before through the barriers (arrivals join the
phase's clock, a passing wait joins it into the waiter's).

Three properties are asserted over many random schedules, with random role
speeds so that any role can fall far behind:

  - no waiter ever finds its barrier two or more phases past the one it
    waits for (the parity would then name the wrong phase: a wait that never
    returns, or one that returns too early);
  - every role finishes (no deadlock);
  - every pair of conflicting accesses to a tile or a TMEM region (a write
    and any other access) is ordered by happens-before, and nothing reads a
    region before it was written (no data race).

The models must follow the kernels: a change to a kernel's barriers or
buffers changes this file.  For the backward, `fixed=False` restores the
protocol before warpgroup 1 waited for the reducer before staging its dQ
half; the checker must find that deadlock.
"""
import random

import pytest


class Overrun(AssertionError):
    pass


class Race(AssertionError):
    pass


def _join(a, b):
    out = dict(a)
    for k, v in b.items():
        if out.get(k, 0) < v:
            out[k] = v
    return out


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending = 0
        self.acc = {}
        self.phase_vc = []   # clock of each completed phase

    @property
    def completed(self):
        return len(self.phase_vc)

    def arrive(self, vc):
        self.acc = _join(self.acc, vc)
        self.pending += 1
        if self.pending == self.count:
            self.phase_vc.append(self.acc)
            self.pending, self.acc = 0, {}


# --------------------------------------------------------------------------
# bwd_main_kernel (persistent).  Buffers: IT0/IT1 (the work-item slots),
# K0/K1, V (the item's K/V tile: K written raw by TMA and rotated in place,
# compute warpgroup cw taking the dims of half K<cw>), Q0/Q1 (the q~ slots, which also receive warpgroup 1's
# staged dQ half), DO, DS0/DS1 (each warpgroup's half of the dS^T tile),
# STAGE (warpgroup 0's dQ staging tile), ROW0/ROW1 (the -LSE2 / -D rows of a
# slot); TMEM A (S^T, then P^T and dS^T packed into it: A<cw>P and A<cw>S are
# the P^T and dS^T columns of warpgroup cw's half), B<cw> (dP^T, then dQ),
# DV, DK.  `items` lists each item's Q-tile count and whether its last Q tile
# runs past the sample's end (the row warp then zeroes that tile's q~ and dO
# rows past the end before the MMAs read them).
# --------------------------------------------------------------------------

def _bwd_roles(items, fixed, head_dim=128, tail_bars=True, tail_slots=2):
    """head_dim 64 has no reducer: dQ leaves by atomics, q_free takes the
    MMA's arrival alone and staging is a no-op.  Ragged item n uses the tail
    barriers q_tail / do_tail / tail_fixed n % tail_slots.  fixed=False
    restores the staging protocol before warpgroup 1 waited for the reducer;
    tail_bars=False has the row warp wait for a ragged tile on its slots'
    q_full / do_full, skipping their earlier phases; tail_slots=1 shares one
    set of tail barriers among all ragged items (checks of the checker)."""
    T = tail_slots
    a_all = ["A0P", "A0S", "A1P", "A1S"]
    n_items = len(items)

    def take(k):
        yield ("wait", f"item_full{k & 1}", k >> 1)
        yield ("read", [f"IT{k & 1}"])
        yield ("arrive", f"item_empty{k & 1}")

    def producer():
        gq = n_tail = 0
        for k in range(n_items + 1):
            if k >= 2:
                yield ("wait", f"item_empty{k & 1}", (k >> 1) - 1)
            yield ("write", [f"IT{k & 1}"])
            yield ("arrive", f"item_full{k & 1}")
            if k == n_items:
                break
            n_q, ragged = items[k]

            def load_q(i):
                g = gq + i
                s = g & 1
                if g >= 2:
                    yield ("wait", f"q_free{s}", (g >> 1) - 1)
                if ragged and i == n_q - 1 and tail_bars:
                    yield ("arrive", f"q_full{s}")
                    yield ("tma", f"q_tail{n_tail % T}", [f"Q{s}"])
                else:
                    yield ("tma", f"q_full{s}", [f"Q{s}"])

            def load_do(i):
                g = gq + i
                if g >= 1:
                    yield ("wait", "do_free", g - 1)
                if ragged and i == n_q - 1 and tail_bars:
                    yield ("arrive", "do_full")
                    yield ("tma", f"do_tail{n_tail % T}", ["DO"])
                else:
                    yield ("tma", "do_full", ["DO"])

            yield from load_q(0)
            if k >= 1:
                yield ("wait", "kv_empty", k - 1)
            yield ("tma", "kv_full", ["K0", "K1", "V"])
            yield from load_do(0)
            for i in range(1, n_q):
                yield from load_q(i)
                yield from load_do(i)
                if i >= 2:
                    yield ("arrive", "q_issued")
            gq += n_q
            n_tail += ragged
        # teardown: the kernel's drain of its own last copies (each must name
        # the phase of that copy: a stale one would stall the drain)
        if n_items:
            yield ("wait", "kv_full", n_items - 1)
            for g in range(max(0, gq - 2), gq):
                yield ("wait", f"q_full{g & 1}", g >> 1)
            yield ("wait", "do_full", gq - 1)
        if tail_bars:
            for t in range(max(0, n_tail - T), n_tail):
                yield ("wait", f"q_tail{t % T}", t // T)
                yield ("wait", f"do_tail{t % T}", t // T)

    def mma():
        gq = n_tail = 0
        for k in range(n_items + 1):
            yield from take(k)
            if k == n_items:
                break
            n_q, ragged = items[k]

            def q_in(i):
                g = gq + i
                if ragged and i == n_q - 1:
                    yield ("wait", f"tail_fixed{n_tail % T}", n_tail // T)
                else:
                    yield ("wait", f"q_full{g & 1}", g >> 1)

            def do_in(i):
                if not (ragged and i == n_q - 1):
                    yield ("wait", "do_full", gq + i)

            yield ("wait", "kv_ready", k)
            yield from q_in(0)
            if gq > 0:
                yield ("wait", "a_free", gq - 1)
            yield ("mma", ["K0", "K1", f"Q{gq & 1}"], a_all, "A")   # S^T_0
            yield ("commit", "s_full")
            yield from do_in(0)
            if gq > 0:
                yield ("wait", "dq_free", gq - 1)
            yield ("mma", ["V", "DO"], ["B0", "B1"], "B")             # dP^T_0
            yield ("commit", "dp_full")
            for i in range(n_q):
                g = gq + i
                s, s1 = g & 1, (g + 1) & 1
                # dV += P^T dO and dK += dS^T q~ reduce over the queries: the
                # half of compute warpgroup cw goes as soon as its operand is in
                for cw in range(2):
                    yield ("wait", f"p_ready{cw}", g)
                    yield ("mma", [f"A{cw}P", "DO"], ["DV"], "DV")
                yield ("commit", "do_free")
                for cw in range(2):
                    yield ("wait", f"ds_ready{cw}", g)
                    yield ("mma", [f"A{cw}S", f"Q{s}"], ["DK"], "DK")
                yield ("commit", "a_free")
                yield ("commit", f"q_free{s}")
                yield ("mma", ["K0", "K1", "DS0", "DS1"], ["B0", "B1"], "B")  # dQ_i
                yield ("commit", "dq_full")
                if i + 1 == n_q:
                    break
                yield from q_in(i + 1)
                yield ("wait", "a_free", g)
                yield ("mma", ["K0", "K1", f"Q{s1}"], a_all, "A")   # S^T_{i+1}
                yield ("commit", "s_full")
                yield from do_in(i + 1)
                yield ("wait", "dq_free", g)
                yield ("mma", ["V", "DO"], ["B0", "B1"], "B")         # dP^T_{i+1}
                yield ("commit", "dp_full")
            yield ("commit", "kv_empty")
            yield ("commit", "acc_full")
            gq += n_q
            n_tail += ragged
        yield ("commit", "fin")
        yield ("wait", "fin", 0)

    def reducer():
        gq = qi_base = 0
        for k in range(n_items + 1):
            yield from take(k)
            if k == n_items:
                break
            n_q = items[k][0]
            for i in range(n_q):
                g = gq + i
                yield ("wait", "stage_full1", g)
                yield ("read", [f"Q{g & 1}"])        # the TMA reduce of the q~-slot half
                yield ("arrive", f"q_free{g & 1}")
                if i + 2 < n_q:
                    yield ("wait", "q_issued", qi_base + i)
                yield ("wait", "stage_full0", g)
                yield ("read", ["STAGE"])
                yield ("arrive", "stage_free")
            gq += n_q
            qi_base += max(0, n_q - 2)

    def row_warp():
        gq = n_tail = 0
        for k in range(n_items + 1):
            yield from take(k)
            if k == n_items:
                break
            n_q, ragged = items[k]
            for i in range(n_q):
                g = gq + i
                s = g & 1
                if g >= 2:
                    yield ("wait", f"q_free{s}", (g >> 1) - 1)
                yield ("write", [f"ROW{s}"])
                yield ("arrive", f"q_ready{s}")
                if ragged and i == n_q - 1:
                    if tail_bars:
                        yield ("wait", f"q_tail{n_tail % T}", n_tail // T)
                        yield ("wait", f"do_tail{n_tail % T}", n_tail // T)
                    else:
                        yield ("wait", f"q_full{s}", g >> 1)
                        yield ("wait", "do_full", g)
                    yield ("write", [f"Q{s}", "DO"])        # rows past the sample's end
                    yield ("arrive", f"tail_fixed{n_tail % T}")
                    n_tail += 1
            gq += n_q

    def compute(cw):
        def dq_load(t):
            yield ("wait", "dq_full", t)
            yield ("read", [f"B{cw}"])
            yield ("arrive", "dq_free")

        def dq_stage(t):
            if head_dim != 128:
                return
            if cw == 0 and t >= 1:
                yield ("wait", "stage_free", t - 1)
            if fixed and cw == 1 and t >= 1:
                yield ("wait", f"q_free{(t - 1) & 1}", (t - 1) >> 1)
            yield ("write", ["STAGE" if cw == 0 else f"Q{t & 1}"])
            yield ("arrive", f"stage_full{cw}")

        def body():
            gq = 0
            for k in range(n_items + 1):
                yield from take(k)
                if k == n_items:
                    break
                n_q = items[k][0]
                yield ("wait", "kv_full", k)
                yield ("read", [f"K{cw}"])
                yield ("write", [f"K{cw}"])                          # the K prologue: its half of the dims
                yield ("arrive", "kv_ready")
                for i in range(n_q):
                    g = gq + i
                    s = g & 1
                    if i > 0:
                        yield from dq_load(g - 1)
                        if cw == 1:
                            yield from dq_stage(g - 1)
                    yield ("wait", f"q_ready{s}", g >> 1)
                    yield ("wait", "s_full", g)
                    yield ("read", [f"A{cw}P", f"A{cw}S", f"ROW{s}"])   # S^T and -LSE2
                    yield ("write", [f"A{cw}P"])                       # P^T
                    yield ("arrive", f"p_ready{cw}")
                    yield ("wait", "dp_full", g)
                    yield ("read", [f"B{cw}", f"ROW{s}"])              # dP^T and -D
                    yield ("write", [f"A{cw}S", f"DS{cw}"])            # dS^T
                    yield ("arrive", f"ds_ready{cw}")
                    if i > 0 and cw == 0:
                        yield from dq_stage(g - 1)
                yield from dq_load(gq + n_q - 1)
                yield from dq_stage(gq + n_q - 1)
                yield ("wait", "acc_full", k)
                yield ("read", ["DV", "DK"])                           # epilogue
                gq += n_q
        return body()

    roles = {"producer": producer(), "mma": mma(), "row": row_warp(), "wg0": compute(0), "wg1": compute(1)}
    if head_dim == 128:
        roles["reducer"] = reducer()
    return roles


def _bwd_barriers(head_dim=128, tail_slots=2):
    nf = 2 if head_dim == 128 else 1
    readers = 5 if head_dim == 128 else 4        # MMA, row warp, two compute warpgroups (+ reducer)
    counts = {"kv_full": 1, "kv_ready": 2, "kv_empty": 1, "acc_full": 1, "fin": 1,
              "item_full0": 1, "item_full1": 1, "item_empty0": readers, "item_empty1": readers,
              "q_full0": 1, "q_full1": 1, "q_ready0": 1, "q_ready1": 1,
              "q_free0": nf, "q_free1": nf, "do_full": 1, "do_free": 1, "s_full": 1, "p_ready0": 1, "p_ready1": 1,
              "dp_full": 1, "ds_ready0": 1, "ds_ready1": 1, "a_free": 1, "dq_full": 1, "dq_free": 2, "stage_full0": 1,
              "stage_full1": 1, "stage_free": 1, "q_issued": 1}
    for t in range(tail_slots):
        counts.update({f"q_tail{t}": 1, f"do_tail{t}": 1, f"tail_fixed{t}": 1})
    return {n: Barrier(n, c) for n, c in counts.items()}


# --------------------------------------------------------------------------
# attn_fwd_kernel (persistent).  Buffers: IT0/IT1 (the work-item slots), Q0/Q1
# (the two Q tiles, written raw by TMA and rotated in place by their softmax
# warpgroups), K<s>, V<s> (the rings, running on across items), TMEM S<a> (S, then
# P packed over it) and O<a> for Q tile a.  `items` lists each item's K/V
# tile count and whether its last V tile has rows past the sample's end (the
# prep warps then zero them before PV reads the tile).
# --------------------------------------------------------------------------

def _fwd_roles(items, rng, k_stages=3, v_stages=2, pv_drain=True, item_ring=True, v_tail=True, tail_slots=2):
    """The item ring, the Q prologue, the K ring (k_stages), the V ring
    (v_stages), the ping-pong MMA order QK_0(j), PV_1(j-1), QK_1(j), PV_0(j),
    and the two softmax warpgroups, whose O rescale waits for the tile's
    previous PV only when the running max grew (data-dependent: drawn at
    random here).  pv_drain=False drops the MMA issuer's wait for PV_a before
    QK_a overwrites S_a; item_ring=False drops the producer's wait for the
    readers of an item slot; v_tail=False has the prep warps wait for a
    ragged item's last V tile on its slot's v_full, skipping that slot's
    earlier phases; ragged item n uses v_tail / v_fixed n % tail_slots, and
    tail_slots=1 shares one of each among all ragged items (checks of the
    checker)."""
    n_items = len(items)
    T = tail_slots

    def take(k):
        yield ("wait", f"item_full{k & 1}", k >> 1)
        yield ("read", [f"IT{k & 1}"])
        yield ("arrive", f"item_empty{k & 1}")

    def producer():
        kc = vc = n_tail = 0
        for k in range(n_items + 1):           # the last slot carries "no more work"
            if k >= 2 and item_ring:
                yield ("wait", f"item_empty{k & 1}", (k >> 1) - 1)
            yield ("write", [f"IT{k & 1}"])
            yield ("arrive", f"item_full{k & 1}")
            if k == n_items:
                break
            n = items[k][0]

            def load_q(a):
                if k >= 1:
                    yield ("wait", f"q_empty{a}", k - 1)
                yield ("tma", f"q_full{a}", [f"Q{a}"])

            def load_k(j):
                g = kc + j
                s = g % k_stages
                if g >= k_stages:
                    yield ("wait", f"k_free{s}", g // k_stages - 1)
                yield ("tma", f"k_full{s}", [f"K{s}"])

            def load_v(j):
                g = vc + j
                s = g % v_stages
                if g >= v_stages:
                    yield ("wait", f"v_free{s}", g // v_stages - 1)
                if items[k][1] and j == n - 1 and v_tail:
                    yield ("arrive", f"v_full{s}")          # the slot's phase, without the data
                    yield ("tma", f"v_tail{n_tail % T}", [f"V{s}"])
                else:
                    yield ("tma", f"v_full{s}", [f"V{s}"])

            yield from load_q(0)
            yield from load_k(0)
            yield from load_q(1)
            for j in range(1, n + 1):
                if j < n:
                    yield from load_k(j)
                yield from load_v(j - 1)
            kc += n
            vc += n
            n_tail += items[k][1]
        # teardown: the drain of the producer's own last copies
        if n_items:
            for a in range(2):
                yield ("wait", f"q_full{a}", n_items - 1)
            for g in range(max(0, kc - k_stages), kc):
                yield ("wait", f"k_full{g % k_stages}", g // k_stages)
            for g in range(max(0, vc - v_stages), vc):
                yield ("wait", f"v_full{g % v_stages}", g // v_stages)
        if v_tail:
            for t in range(max(0, n_tail - T), n_tail):
                yield ("wait", f"v_tail{t % T}", t // T)

    def qk(a, g):
        return ("mma", [f"Q{a}", f"K{g % k_stages}"], [f"S{a}"], f"S{a}")

    def pv(a, g):
        return ("mma", [f"S{a}", f"V{g % v_stages}"], [f"O{a}"], f"O{a}")

    def mma():
        gs = n_ragged = 0
        for k in range(n_items + 1):
            yield from take(k)
            if k == n_items:
                break
            n, ragged = items[k]
            yield ("wait", "q_ready0", k)
            yield ("wait", f"k_full{gs % k_stages}", gs // k_stages)
            if gs > 0 and pv_drain:
                yield ("wait", "pv_done0", gs - 1)
            yield qk(0, gs)
            yield ("commit", "s_full0")
            if n == 1:
                yield ("commit", "q_empty0")
            for j in range(n):
                g = gs + j
                if j > 0:
                    yield ("wait", "p_full1", g - 1)
                    yield pv(1, g - 1)
                    yield ("commit", "pv_done1")
                    yield ("commit", f"v_free{(g - 1) % v_stages}")
                    if pv_drain:
                        yield ("wait", "pv_done1", g - 1)
                else:
                    yield ("wait", "q_ready1", k)
                    if gs > 0 and pv_drain:
                        yield ("wait", "pv_done1", gs - 1)
                yield qk(1, g)
                yield ("commit", "s_full1")
                yield ("commit", f"k_free{g % k_stages}")
                if j == n - 1:
                    yield ("commit", "q_empty1")
                yield ("wait", "p_full0", g)
                if ragged and j == n - 1:
                    yield ("wait", f"v_fixed{n_ragged % T}", n_ragged // T)
                else:
                    yield ("wait", f"v_full{g % v_stages}", g // v_stages)
                yield pv(0, g)
                yield ("commit", "pv_done0")
                if j + 1 < n:
                    yield ("wait", f"k_full{(g + 1) % k_stages}", (g + 1) // k_stages)
                    if pv_drain:
                        yield ("wait", "pv_done0", g)
                    yield qk(0, g + 1)
                    yield ("commit", "s_full0")
                    if j + 2 == n:
                        yield ("commit", "q_empty0")
            yield ("wait", "p_full1", gs + n - 1)
            yield pv(1, gs + n - 1)
            yield ("commit", "pv_done1")
            yield ("commit", f"v_free{(gs + n - 1) % v_stages}")
            gs += n
            n_ragged += ragged
        yield ("commit", "final")
        yield ("wait", "final", 0)

    def prep():
        vc = n_ragged = 0
        for k in range(n_items + 1):
            yield from take(k)
            if k == n_items:
                break
            n, ragged = items[k]
            if ragged:
                g = vc + n - 1
                if v_tail:
                    yield ("wait", f"v_tail{n_ragged % T}", n_ragged // T)
                else:
                    yield ("wait", f"v_full{g % v_stages}", g // v_stages)
                yield ("write", [f"V{g % v_stages}"])       # rows past the sample's end
                yield ("arrive", f"v_fixed{n_ragged % T}")
                n_ragged += 1
            vc += n

    def softmax(a):
        def prologue(k):
            yield from take(k)
            if k < n_items:
                yield ("wait", f"q_full{a}", k)
                yield ("read", [f"Q{a}"])
                yield ("write", [f"Q{a}"])              # the Q prologue: rotation in place
                yield ("arrive", f"q_ready{a}")

        gs = 0
        yield from prologue(0)
        for k in range(n_items):
            n = items[k][0]
            for j in range(n):
                g = gs + j
                yield ("wait", f"s_full{a}", g)
                yield ("read", [f"S{a}"])
                yield ("write", [f"S{a}"])                  # P over S
                if j > 0 and rng.random() < 0.3:
                    yield ("wait", f"pv_done{a}", g - 1)    # O rescale
                    yield ("read", [f"O{a}"])
                    yield ("write", [f"O{a}"])
                yield ("arrive", f"p_full{a}")
            yield from prologue(k + 1)                      # the next item's, before this epilogue
            yield ("wait", f"pv_done{a}", gs + n - 1)
            yield ("read", [f"O{a}"])                       # epilogue
            gs += n

    return {"producer": producer(), "mma": mma(), "prep": prep(), "sm0": softmax(0), "sm1": softmax(1)}


def _fwd_barriers(k_stages=3, v_stages=2, tail_slots=2):
    names = ["final", "s_full0", "s_full1", "p_full0", "p_full1", "pv_done0", "pv_done1",
             "item_full0", "item_full1", "q_full0", "q_full1", "q_ready0", "q_ready1", "q_empty0", "q_empty1"]
    names += [f"k_full{s}" for s in range(k_stages)] + [f"k_free{s}" for s in range(k_stages)]
    names += [f"v_full{s}" for s in range(v_stages)] + [f"v_free{s}" for s in range(v_stages)]
    names += [f"v_tail{t}" for t in range(tail_slots)] + [f"v_fixed{t}" for t in range(tail_slots)]
    bars = {n: Barrier(n, 1) for n in names}
    for s in range(2):
        bars[f"item_empty{s}"] = Barrier(f"item_empty{s}", 4)   # MMA, prep, two softmax warpgroups
    return bars


# --------------------------------------------------------------------------
# the explorer
# --------------------------------------------------------------------------

def run_schedule(n, seed, fixed=True, kernel="bwd", head_dim=128, pv_drain=True, item_ring=True,
                 v_tail=True, tail_bars=True, tail_slots=2, max_steps=400000):
    """One random interleaving of `kernel`'s protocol over the work items
    n = [(Q tiles, ragged), ...] (backward) or [(K/V tiles, ragged), ...]
    (forward).  Returns None when every role finished, or a string
    describing the deadlock; raises Overrun on a phase overrun and Race on a
    data race."""
    rng = random.Random(seed)
    if kernel == "bwd":
        bars, roles = _bwd_barriers(head_dim, tail_slots), _bwd_roles(n, fixed, head_dim, tail_bars, tail_slots)
    else:
        bars, roles = _fwd_barriers(tail_slots=tail_slots), _fwd_roles(n, random.Random(seed + 7919), pv_drain=pv_drain,
                                                                       item_ring=item_ring, v_tail=v_tail,
                                                                       tail_slots=tail_slots)
    nxt = {r: next(g) for r, g in roles.items()}
    vc = {r: {r: 1} for r in roles}
    weight = {r: rng.choice([0.02, 0.2, 1.0, 1.0, 5.0]) for r in roles}  # some roles run far behind
    buffers = {}
    tma = []        # (barrier, tiles written, clock)
    mmaq = []       # the MMA unit's items in issue order
    ids = iter(range(1, 1 << 30))

    def access(epoch, cur, names, kind, who):
        for b in names:
            st = buffers.setdefault(b, {"w": None, "r": []})
            hb = lambda ep: cur.get(ep[0], 0) >= ep[1]   # noqa: E731
            if kind == "read":
                if st["w"] is None:
                    raise Race(f"{who} reads {b} before anything wrote it")
                if not hb(st["w"]):
                    raise Race(f"{who} reads {b} unordered with the write by {st['w'][2]}")
                st["r"].append(epoch + (who,))
            else:
                if st["w"] is not None and not hb(st["w"]):
                    raise Race(f"{who} writes {b} unordered with the write by {st['w'][2]}")
                for r in st["r"]:
                    if not hb(r):
                        raise Race(f"{who} writes {b} unordered with the read by {r[2]}")
                st["w"], st["r"] = epoch + (who,), []

    def ready(role):
        op = nxt[role]
        if op is None:
            return False
        if op[0] == "wait":
            c = bars[op[1]].completed
            if c >= op[2] + 2:
                raise Overrun(f"{role} waits for phase {op[2]} of {op[1]}, which has completed {c} phases")
            if c < op[2]:
                # the parity would name an earlier phase: the wait would pass at once
                raise Overrun(f"{role} waits for phase {op[2]} of {op[1]}, which has completed only {c} phases")
            return (c & 1) != (op[2] & 1)
        return True

    def mma_ready():
        out = []
        for idx, it in enumerate(mmaq):
            if it["done"]:
                continue
            earlier = [e for e in mmaq[:idx] if not e["done"]]
            if it["kind"] == "commit":
                if not earlier:
                    out.append(idx)
            elif not any(e["kind"] == "op" and e["acc"] == it["acc"] for e in earlier):
                out.append(idx)
        return out

    for _ in range(max_steps):
        cands = [r for r in roles if ready(r)]
        mr = mma_ready()
        pool = cands + (["<tma unit>"] if tma else []) + (["<mma unit>"] if mr else [])
        if not pool:
            break
        w = [weight[r] for r in cands] + [1.0] * (len(pool) - len(cands))
        pick = rng.choices(pool, weights=w)[0]
        if pick == "<tma unit>":
            bar, tiles, cvc = tma.pop(rng.randrange(len(tma)))
            tid = f"tma{next(ids)}"
            cvc = _join(cvc, {tid: 1})
            access((tid, 1), cvc, tiles, "write", f"TMA into {bar}")
            bars[bar].arrive(cvc)
            continue
        if pick == "<mma unit>":
            it = mmaq[rng.choice(mr)]
            it["done"] = True
            if it["kind"] == "commit":
                cvc = it["vc"]
                for e in mmaq:
                    if e["kind"] == "op" and e["seq"] < it["seq"]:
                        cvc = _join(cvc, e["exec_vc"])
                bars[it["bar"]].arrive(cvc)
            else:
                oid = f"mma{next(ids)}"
                cvc = _join(it["vc"], {oid: 1})
                for e in mmaq:
                    if e["kind"] == "op" and e["acc"] == it["acc"] and e["seq"] < it["seq"]:
                        cvc = _join(cvc, e["exec_vc"])
                access((oid, 1), cvc, it["reads"], "read", f"MMA into {it['acc']}")
                access((oid, 1), cvc, it["writes"], "write", f"MMA into {it['acc']}")
                it["exec_vc"] = cvc
            continue
        op = nxt[pick]
        kind = op[0]
        if kind == "wait":
            vc[pick] = _join(vc[pick], bars[op[1]].phase_vc[op[2]])
        elif kind == "arrive":
            bars[op[1]].arrive(vc[pick])
            vc[pick][pick] += 1
        elif kind == "tma":
            tma.append((op[1], op[2], dict(vc[pick])))
            vc[pick][pick] += 1
        elif kind == "mma":
            mmaq.append({"kind": "op", "reads": op[1], "writes": op[2], "acc": op[3], "vc": dict(vc[pick]),
                         "done": False, "seq": len(mmaq)})
            vc[pick][pick] += 1
        elif kind == "commit":
            mmaq.append({"kind": "commit", "bar": op[1], "vc": dict(vc[pick]), "done": False, "seq": len(mmaq)})
            vc[pick][pick] += 1
        else:
            access((pick, vc[pick][pick]), vc[pick], op[1], kind, pick)
        nxt[pick] = next(roles[pick], None)
    stuck = {r: op for r, op in nxt.items() if op is not None}
    if stuck:
        return "deadlock: " + ", ".join(f"{r} at {op}" for r, op in stuck.items())
    return None


BWD_ITEM_LISTS = [
    [(1, True)], [(2, False)], [(3, True), (3, True)], [(5, False), (1, True), (2, True)],
    [(1, False), (1, True), (1, False), (2, True)], [(8, True), (4, False)],
    [(2, True), (3, False), (1, True), (4, True), (2, False)],
    [(2, True), (1, True), (1, True)], [(1, True), (1, False), (1, True), (1, True), (1, True)],
]


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("items", BWD_ITEM_LISTS)
def test_bwd_protocol_is_race_and_deadlock_free(items, head_dim):
    for seed in range(200):
        assert run_schedule(items, seed, head_dim=head_dim) is None, (items, head_dim, seed)


FWD_ITEM_LISTS = [
    [(1, True)], [(2, False)], [(3, True), (3, True)], [(4, False), (1, True), (2, True)],
    [(1, False), (1, True), (1, False), (1, True)], [(5, True), (2, False), (7, True)],
    [(2, True), (3, False), (1, True), (4, True), (2, False)],
    [(2, True), (1, True), (1, True)], [(1, True), (1, True), (1, True), (1, True), (1, True)],
]


@pytest.mark.parametrize("items", FWD_ITEM_LISTS)
def test_fwd_protocol_is_race_and_deadlock_free(items):
    for seed in range(200):
        assert run_schedule(items, seed, kernel="fwd") is None, (items, seed)


def test_checker_finds_the_unthrottled_staging_deadlock():
    """Without warpgroup 1's wait for the reducer, some schedule lets it stage
    two dQ halves ahead: stage_full[1] then overruns the reducer's wait."""
    for seed in range(2000):
        try:
            out = run_schedule([(6, False)], seed, fixed=False)
        except Overrun as e:
            assert "stage_full1" in str(e)
            return
        except Race:
            return
        if out is not None:
            return
    pytest.fail("the old staging protocol passed every schedule")


def test_checker_finds_a_missing_tmem_drain():
    """Without the MMA issuer's wait for PV_a before QK_a rewrites S_a, the
    two MMAs (different accumulators, so not ordered) race on S_a."""
    for seed in range(500):
        try:
            run_schedule([(4, False), (2, True)], seed, kernel="fwd", pv_drain=False)
        except Race as e:
            assert "S0" in str(e) or "S1" in str(e)
            return
    pytest.fail("the checker missed the S/P race")


def test_checker_finds_an_unguarded_item_slot():
    """Without the producer's wait for every reader of an item slot, some
    schedule rewrites a slot that a slow role has not read yet."""
    for seed in range(2000):
        try:
            out = run_schedule([(1, False)] * 5, seed, kernel="fwd", item_ring=False)
        except (Race, Overrun) as e:
            assert "IT" in str(e) or "item_full" in str(e)
            return
        assert out is None
    pytest.fail("the checker missed the item-slot race")


def test_checker_finds_a_skipped_phase_wait():
    """A ragged item's last V tile waited for on its slot's v_full skips that
    slot's earlier phases: the parity can then name a phase that has not
    completed (the wait would pass before the tile lands)."""
    for seed in range(2000):
        try:
            run_schedule([(3, True), (3, True), (2, True)], seed, kernel="fwd", v_tail=False)
        except (Overrun, Race) as e:
            assert "v_full" in str(e) or "V" in str(e)
            return
    pytest.fail("the checker missed the skipped-phase wait")


def test_checker_finds_a_skipped_phase_wait_in_the_backward():
    """The row warp waiting for a ragged item's last q~ / dO tile on the
    slots' own barriers skips their earlier phases, as in the forward."""
    for seed in range(2000):
        try:
            run_schedule([(3, True), (2, True), (3, True)], seed, tail_bars=False)
        except (Overrun, Race):
            return
    pytest.fail("the checker missed the skipped-phase wait")


@pytest.mark.parametrize("kernel", ["fwd", "bwd"])
def test_checker_finds_a_shared_tail_barrier(kernel):
    """One set of tail barriers for every ragged item: two short ragged items
    in a row can complete two phases of a tail barrier before its waiter
    looked (the second tail needs only the other ring slot)."""
    for seed in range(2000):
        try:
            run_schedule([(2, True), (1, True), (1, True)], seed, kernel=kernel, tail_slots=1)
        except (Overrun, Race):
            return
    pytest.fail("the checker missed the shared tail barrier")


def test_checker_finds_a_stale_drain_phase():
    """A teardown drain naming the phase of the last plain dO load, when tail
    loads completed later phases of do_full, overruns (the kernel's drain
    would stall until its time limit)."""
    roles = _bwd_roles([(3, True), (2, True)], True)
    prod = list(roles["producer"])
    waits = [op for op in prod if op[0] == "wait" and op[1] == "do_full"]
    assert waits[-1][2] == 4           # the last dO load (a tail) completed phase 4
