"""The mbarrier protocols of the two attention kernels (csrc/attn_fwd.cu,
csrc/attn_bwd.cu), checked on the CPU by exploring interleavings.

Each role of a kernel (the TMA producer, the MMA issuer, the softmax or
compute warpgroups, and in the backward the dQ reducer and the row warp) is
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
# bwd_main_kernel.  Buffers: K, V, Q0/Q1 (the q~ slots, which also receive
# warpgroup 1's staged dQ half), DO, DS0/DS1 (each warpgroup's half of the
# dS^T tile), STAGE (warpgroup 0's dQ staging tile), ROW0/ROW1 (the -LSE2 / -D
# rows of a slot); TMEM A (S^T, then P^T and dS^T packed into it: A<cw>P and
# A<cw>S are the P^T and dS^T columns of warpgroup cw's half), B<cw> (dP^T,
# then dQ), DV, DK.
# --------------------------------------------------------------------------

def _bwd_roles(n_q, fixed, head_dim=128):
    """head_dim 64 has no reducer: dQ leaves by atomics, q_free takes the
    MMA's arrival alone and staging is a no-op."""
    a_all = ["A0P", "A0S", "A1P", "A1S"]

    def producer():
        yield ("tma", "kv_full", ["K", "V"])
        for i in range(n_q):
            s = i & 1
            if i >= 2:
                yield ("wait", f"q_free{s}", (i >> 1) - 1)
            yield ("tma", f"q_full{s}", [f"Q{s}"])
            if i >= 1:
                yield ("wait", "do_free", i - 1)
            yield ("tma", "do_full", ["DO"])
            if i >= 2:
                yield ("arrive", "q_issued")

    def mma():
        yield ("wait", "kv_full", 0)
        yield ("wait", "q_full0", 0)
        yield ("mma", ["K", "Q0"], a_all, "A")                 # S^T_0
        yield ("commit", "s_full")
        yield ("wait", "do_full", 0)
        yield ("mma", ["V", "DO"], ["B0", "B1"], "B")          # dP^T_0
        yield ("commit", "dp_full")
        for i in range(n_q):
            s, s1 = i & 1, (i + 1) & 1
            yield ("wait", "p_ready", i)
            yield ("mma", ["A0P", "A1P", "DO"], ["DV"], "DV")  # dV += P^T dO
            yield ("commit", "do_free")
            yield ("wait", "ds_ready", i)
            yield ("mma", ["A0S", "A1S", f"Q{s}"], ["DK"], "DK")  # dK += dS^T q~
            yield ("commit", "a_free")
            yield ("commit", f"q_free{s}")
            yield ("mma", ["K", "DS0", "DS1"], ["B0", "B1"], "B")  # dQ_i
            yield ("commit", "dq_full")
            if i + 1 == n_q:
                break
            yield ("wait", f"q_full{s1}", (i + 1) >> 1)
            yield ("wait", "a_free", i)
            yield ("mma", ["K", f"Q{s1}"], a_all, "A")         # S^T_{i+1}
            yield ("commit", "s_full")
            yield ("wait", "do_full", i + 1)
            yield ("wait", "dq_free", i)
            yield ("mma", ["V", "DO"], ["B0", "B1"], "B")      # dP^T_{i+1}
            yield ("commit", "dp_full")
        yield ("commit", "fin")

    def reducer():
        for i in range(n_q):
            yield ("wait", "stage_full1", i)
            yield ("read", [f"Q{i & 1}"])        # the TMA reduce of the q~-slot half
            yield ("arrive", f"q_free{i & 1}")
            if i + 2 < n_q:
                yield ("wait", "q_issued", i)
            yield ("wait", "stage_full0", i)
            yield ("read", ["STAGE"])
            yield ("arrive", "stage_free")

    def row_warp():
        for i in range(n_q):
            s = i & 1
            if i >= 2:
                yield ("wait", f"q_free{s}", (i >> 1) - 1)
            yield ("write", [f"ROW{s}"])
            yield ("arrive", f"q_ready{s}")

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
            for i in range(n_q):
                s = i & 1
                if i > 0:
                    yield from dq_load(i - 1)
                    if cw == 1:
                        yield from dq_stage(i - 1)
                yield ("wait", f"q_ready{s}", i >> 1)
                yield ("wait", "s_full", i)
                yield ("read", [f"A{cw}P", f"A{cw}S", f"ROW{s}"])   # S^T and -LSE2
                yield ("write", [f"A{cw}P"])                       # P^T
                yield ("arrive", "p_ready")
                yield ("wait", "dp_full", i)
                yield ("read", [f"B{cw}", f"ROW{s}"])              # dP^T and -D
                yield ("write", [f"A{cw}S", f"DS{cw}"])            # dS^T
                yield ("arrive", "ds_ready")
                if i > 0 and cw == 0:
                    yield from dq_stage(i - 1)
            yield from dq_load(n_q - 1)
            yield from dq_stage(n_q - 1)
            yield ("wait", "fin", 0)
            yield ("read", ["DV", "DK"])                           # epilogue
        return body()

    roles = {"producer": producer(), "mma": mma(), "row": row_warp(), "wg0": compute(0), "wg1": compute(1)}
    if head_dim == 128:
        roles["reducer"] = reducer()
    return roles


def _bwd_barriers(head_dim=128):
    nf = 2 if head_dim == 128 else 1
    counts = {"kv_full": 1, "fin": 1, "q_full0": 1, "q_full1": 1, "q_ready0": 1, "q_ready1": 1,
              "q_free0": nf, "q_free1": nf, "do_full": 1, "do_free": 1, "s_full": 1, "p_ready": 2,
              "dp_full": 1, "ds_ready": 2, "a_free": 1, "dq_full": 1, "dq_free": 2, "stage_full0": 1,
              "stage_full1": 1, "stage_free": 1, "q_issued": 1}
    return {n: Barrier(n, c) for n, c in counts.items()}


# --------------------------------------------------------------------------
# attn_fwd_kernel.  Buffers: Q0/Q1 (the two Q tiles), K<s>, V<s> (the rings),
# TMEM S<a> (S, then P packed over it) and O<a> for Q tile a.
# --------------------------------------------------------------------------

def _fwd_roles(n_kv, rng, k_stages=3, v_stages=2, pv_drain=True):
    """The K ring (k_stages), the V ring (v_stages), the ping-pong MMA order
    QK_0(j), PV_1(j-1), QK_1(j), PV_0(j), and the two softmax warpgroups, whose
    O rescale waits for the tile's previous PV only when the running max
    grew (data-dependent: drawn at random here).  pv_drain=False drops the
    MMA issuer's wait for PV_a before QK_a overwrites S_a (a check of the
    checker)."""

    def producer():
        yield ("tma", "q_full", ["Q0", "Q1"])
        for j in range(n_kv + 1):
            if j < n_kv:
                s = j % k_stages
                if j >= k_stages:
                    yield ("wait", f"k_free{s}", j // k_stages - 1)
                yield ("tma", f"k_full{s}", [f"K{s}"])
            jv = j - 1
            if jv >= 0:
                s = jv % v_stages
                if jv >= v_stages:
                    yield ("wait", f"v_free{s}", jv // v_stages - 1)
                yield ("tma", f"v_full{s}", [f"V{s}"])

    def qk(a, j):
        return ("mma", [f"Q{a}", f"K{j % k_stages}"], [f"S{a}"], f"S{a}")

    def pv(a, j):
        return ("mma", [f"S{a}", f"V{j % v_stages}"], [f"O{a}"], f"O{a}")

    def mma():
        yield ("wait", "q_full", 0)
        yield ("wait", "k_full0", 0)
        yield qk(0, 0)
        yield ("commit", "s_full0")
        for j in range(n_kv):
            if j > 0:
                yield ("wait", "p_full1", j - 1)
                yield pv(1, j - 1)
                yield ("commit", "pv_done1")
                yield ("commit", f"v_free{(j - 1) % v_stages}")
                if pv_drain:
                    yield ("wait", "pv_done1", j - 1)
            yield qk(1, j)
            yield ("commit", "s_full1")
            yield ("commit", f"k_free{j % k_stages}")
            yield ("wait", "p_full0", j)
            yield ("wait", f"v_full{j % v_stages}", j // v_stages)
            yield pv(0, j)
            yield ("commit", "pv_done0")
            if j + 1 < n_kv:
                yield ("wait", f"k_full{(j + 1) % k_stages}", (j + 1) // k_stages)
                if pv_drain:
                    yield ("wait", "pv_done0", j)
                yield qk(0, j + 1)
                yield ("commit", "s_full0")
        yield ("wait", "p_full1", n_kv - 1)
        yield pv(1, n_kv - 1)
        yield ("commit", "pv_done1")
        yield ("commit", f"v_free{(n_kv - 1) % v_stages}")
        yield ("commit", "final")
        yield ("wait", "final", 0)

    def softmax(a):
        for j in range(n_kv):
            yield ("wait", f"s_full{a}", j)
            yield ("read", [f"S{a}"])
            yield ("write", [f"S{a}"])                      # P over S
            if j > 0 and rng.random() < 0.3:
                yield ("wait", f"pv_done{a}", j - 1)        # O rescale
                yield ("read", [f"O{a}"])
                yield ("write", [f"O{a}"])
            yield ("arrive", f"p_full{a}")
        yield ("wait", f"pv_done{a}", n_kv - 1)
        yield ("read", [f"O{a}"])                           # epilogue

    return {"producer": producer(), "mma": mma(), "sm0": softmax(0), "sm1": softmax(1)}


def _fwd_barriers(k_stages=3, v_stages=2):
    names = ["q_full", "final", "s_full0", "s_full1", "p_full0", "p_full1", "pv_done0", "pv_done1"]
    names += [f"k_full{s}" for s in range(k_stages)] + [f"k_free{s}" for s in range(k_stages)]
    names += [f"v_full{s}" for s in range(v_stages)] + [f"v_free{s}" for s in range(v_stages)]
    return {n: Barrier(n, 1) for n in names}


# --------------------------------------------------------------------------
# the explorer
# --------------------------------------------------------------------------

def run_schedule(n, seed, fixed=True, kernel="bwd", head_dim=128, pv_drain=True, max_steps=400000):
    """One random interleaving of `kernel`'s protocol over n Q tiles
    (backward) or n K/V tiles (forward).  Returns None when every role
    finished, or a string describing the deadlock; raises Overrun on a phase
    overrun and Race on a data race."""
    rng = random.Random(seed)
    if kernel == "bwd":
        bars, roles = _bwd_barriers(head_dim), _bwd_roles(n, fixed, head_dim)
    else:
        bars, roles = _fwd_barriers(), _fwd_roles(n, random.Random(seed + 7919), pv_drain=pv_drain)
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


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("n_q", [1, 2, 3, 4, 5, 8])
def test_bwd_protocol_is_race_and_deadlock_free(n_q, head_dim):
    for seed in range(200):
        assert run_schedule(n_q, seed, head_dim=head_dim) is None, (n_q, head_dim, seed)


@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 7])
def test_fwd_protocol_is_race_and_deadlock_free(n_kv):
    for seed in range(200):
        assert run_schedule(n_kv, seed, kernel="fwd") is None, (n_kv, seed)


def test_checker_finds_the_unthrottled_staging_deadlock():
    """Without warpgroup 1's wait for the reducer, some schedule lets it stage
    two dQ halves ahead: stage_full[1] then overruns the reducer's wait."""
    for seed in range(2000):
        try:
            out = run_schedule(6, seed, fixed=False)
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
            run_schedule(4, seed, kernel="fwd", pv_drain=False)
        except Race as e:
            assert "S0" in str(e) or "S1" in str(e)
            return
    pytest.fail("the checker missed the S/P race")
