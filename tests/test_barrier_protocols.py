"""The mbarrier protocols of the two attention kernels (csrc/attn_fwd.cu,
csrc/attn_bwd.cu), checked on the CPU by exploring interleavings.

Each role of a kernel (the TMA producer, the MMA issuer, the softmax or
compute warpgroups, and in the backward the dQ reducer and the row warp) is
written here as its sequence of barrier operations, in the kernel's order.
Asynchronous work is modelled by agents that the scheduler may delay
arbitrarily: each TMA load completes its barrier on its own, and
tcgen05.commit arrivals land in issue order.  The barriers follow the
hardware's parity rule: a wait for phase k (parity k & 1) passes while the
number of completed phases c has the other parity.

Two properties are asserted over many random schedules (with random role
speeds, so that any role can fall far behind):

  - no waiter ever finds its barrier two or more phases past the one it
    waits for (the parity would then name the wrong phase: a wait that never
    returns, or one that returns too early);
  - every role finishes (no deadlock).

The models must follow the kernels: a change to a kernel's barriers changes
this file.  For the backward, `fixed=False` restores the protocol before
warpgroup 1 waited for the reducer before staging its dQ half; the checker
must find that deadlock.
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending = 0
        self.completed = 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.completed += 1


class Overrun(AssertionError):
    pass


def _bwd_roles(n_q, fixed, head_dim=128):
    """head_dim 64 has no reducer: dQ leaves by atomics, q_free takes the
    MMA's arrival alone and staging is a no-op.  Generators yielding ('wait', bar, phase), ('arrive', bar),
    ('commit', bar) or ('tma', bar)."""

    def producer():
        yield ("tma", "kv_full")
        for i in range(n_q):
            s = i & 1
            if i >= 2:
                yield ("wait", f"q_free{s}", (i >> 1) - 1)
            yield ("tma", f"q_full{s}")
            if i >= 1:
                yield ("wait", "do_free", i - 1)
            yield ("tma", "do_full")
            if i >= 2:
                yield ("arrive", "q_issued")

    def mma():
        yield ("wait", "kv_full", 0)
        yield ("wait", "q_full0", 0)
        yield ("commit", "s_full")
        yield ("wait", "do_full", 0)
        yield ("commit", "dp_full")
        for i in range(n_q):
            s, s1 = i & 1, (i + 1) & 1
            yield ("wait", "p_ready", i)
            yield ("commit", "do_free")          # dV_i
            yield ("wait", "ds_ready", i)
            yield ("commit", "a_free")           # dK_i
            yield ("commit", f"q_free{s}")
            yield ("commit", "dq_full")          # dQ_i
            if i + 1 == n_q:
                break
            yield ("wait", f"q_full{s1}", (i + 1) >> 1)
            yield ("wait", "a_free", i)
            yield ("commit", "s_full")           # S_{i+1}
            yield ("wait", "do_full", i + 1)
            yield ("wait", "dq_free", i)
            yield ("commit", "dp_full")          # dP_{i+1}
        yield ("commit", "fin")

    def reducer():
        for i in range(n_q):
            yield ("wait", "stage_full1", i)
            yield ("arrive", f"q_free{i & 1}")   # after the q~-slot half is read
            if i + 2 < n_q:
                yield ("wait", "q_issued", i)
            yield ("wait", "stage_full0", i)
            yield ("arrive", "stage_free")

    def row_warp():
        for i in range(n_q):
            s = i & 1
            if i >= 2:
                yield ("wait", f"q_free{s}", (i >> 1) - 1)
            yield ("arrive", f"q_ready{s}")

    def compute(cw):
        def dq_load(t):
            yield ("wait", "dq_full", t)
            yield ("arrive", "dq_free")

        def dq_stage(t):
            if head_dim != 128:
                return
            if cw == 0 and t >= 1:
                yield ("wait", "stage_free", t - 1)
            if fixed and cw == 1 and t >= 1:
                yield ("wait", f"q_free{(t - 1) & 1}", (t - 1) >> 1)
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
                yield ("arrive", "p_ready")
                yield ("wait", "dp_full", i)
                yield ("arrive", "ds_ready")
                if i > 0 and cw == 0:
                    yield from dq_stage(i - 1)
            yield from dq_load(n_q - 1)
            yield from dq_stage(n_q - 1)
            yield ("wait", "fin", 0)
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


def _fwd_roles(n_kv, rng, k_stages=3, v_stages=2):
    """attn_fwd_kernel: the K ring (k_stages) and V ring (v_stages), the
    ping-pong MMA order QK_0(j), PV_1(j-1), QK_1(j), PV_0(j), and the two
    softmax warpgroups (one per Q tile), whose O rescale waits for the
    tile's previous PV only when the running max grew (data-dependent:
    drawn at random here)."""

    def producer():
        yield ("tma", "q_full")
        for j in range(n_kv + 1):
            if j < n_kv:
                s = j % k_stages
                if j >= k_stages:
                    yield ("wait", f"k_free{s}", j // k_stages - 1)
                yield ("tma", f"k_full{s}")
            jv = j - 1
            if jv >= 0:
                s = jv % v_stages
                if jv >= v_stages:
                    yield ("wait", f"v_free{s}", jv // v_stages - 1)
                yield ("tma", f"v_full{s}")

    def mma():
        yield ("wait", "q_full", 0)
        yield ("wait", "k_full0", 0)
        yield ("commit", "s_full0")                      # QK_0(0)
        for j in range(n_kv):
            if j > 0:
                yield ("wait", "p_full1", j - 1)
                yield ("commit", "pv_done1")             # PV_1(j-1)
                yield ("commit", f"v_free{(j - 1) % v_stages}")
                yield ("wait", "pv_done1", j - 1)
            yield ("commit", "s_full1")                  # QK_1(j)
            yield ("commit", f"k_free{j % k_stages}")
            yield ("wait", "p_full0", j)
            yield ("wait", f"v_full{j % v_stages}", j // v_stages)
            yield ("commit", "pv_done0")                 # PV_0(j)
            if j + 1 < n_kv:
                yield ("wait", f"k_full{(j + 1) % k_stages}", (j + 1) // k_stages)
                yield ("wait", "pv_done0", j)
                yield ("commit", "s_full0")              # QK_0(j+1)
        yield ("wait", "p_full1", n_kv - 1)
        yield ("commit", "pv_done1")                     # PV_1(n_kv-1)
        yield ("commit", f"v_free{(n_kv - 1) % v_stages}")
        yield ("commit", "final")
        yield ("wait", "final", 0)

    def softmax(a):
        for j in range(n_kv):
            yield ("wait", f"s_full{a}", j)
            if j > 0 and rng.random() < 0.3:
                yield ("wait", f"pv_done{a}", j - 1)     # O rescale
            yield ("arrive", f"p_full{a}")
        yield ("wait", f"pv_done{a}", n_kv - 1)

    return {"producer": producer(), "mma": mma(), "sm0": softmax(0), "sm1": softmax(1)}


def _fwd_barriers(k_stages=3, v_stages=2):
    names = ["q_full", "final", "s_full0", "s_full1", "p_full0", "p_full1", "pv_done0", "pv_done1"]
    names += [f"k_full{s}" for s in range(k_stages)] + [f"k_free{s}" for s in range(k_stages)]
    names += [f"v_full{s}" for s in range(v_stages)] + [f"v_free{s}" for s in range(v_stages)]
    return {n: Barrier(n, 1) for n in names}


def run_schedule(n_q, seed, fixed=True, kernel="bwd", head_dim=128, max_steps=200000):
    """One random interleaving of `kernel`'s protocol over n_q Q tiles
    (backward) or n_q K/V tiles (forward).  Returns None when every role
    finished, or a string describing the deadlock; raises Overrun on a phase
    overrun."""
    rng = random.Random(seed)
    if kernel == "bwd":
        bars, roles = _bwd_barriers(head_dim), _bwd_roles(n_q, fixed, head_dim)
    else:
        bars, roles = _fwd_barriers(), _fwd_roles(n_q, random.Random(seed + 7919))
    nxt = {r: next(g) for r, g in roles.items()}
    weight = {r: rng.choice([0.02, 0.2, 1.0, 1.0, 5.0]) for r in roles}  # some roles run far behind
    tma = []        # issued loads, completing in any order
    commits = []    # tcgen05.commit arrivals, landing in issue order

    def check(role, bar, k):
        c = bars[bar].completed
        if c >= k + 2:
            raise Overrun(f"{role} waits for phase {k} of {bar}, which has completed {c} phases")

    def ready(role):
        op = nxt[role]
        if op is None:
            return False
        if op[0] == "wait":
            check(role, op[1], op[2])
            return (bars[op[1]].completed & 1) != (op[2] & 1)
        return True

    for _ in range(max_steps):
        cands = [r for r in roles if ready(r)]
        agents = (["tma"] if tma else []) + (["commit"] if commits else [])
        if not cands and not agents:
            break
        pool = cands + agents
        w = [weight[r] for r in cands] + [1.0] * len(agents)
        pick = rng.choices(pool, weights=w)[0]
        if pick == "tma":
            bars[tma.pop(rng.randrange(len(tma)))].arrive()
            continue
        if pick == "commit":
            bars[commits.pop(0)].arrive()
            continue
        kind, bar = nxt[pick][0], nxt[pick][1]
        if kind == "arrive":
            bars[bar].arrive()
        elif kind == "tma":
            tma.append(bar)
        elif kind == "commit":
            commits.append(bar)
        nxt[pick] = next(roles[pick], None)
    stuck = {r: op for r, op in nxt.items() if op is not None}
    if stuck:
        return "deadlock: " + ", ".join(f"{r} at {op}" for r, op in stuck.items())
    return None


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("n_q", [1, 2, 3, 4, 5, 8])
def test_bwd_protocol_never_overruns_or_deadlocks(n_q, head_dim):
    for seed in range(300):
        assert run_schedule(n_q, seed, head_dim=head_dim) is None, (n_q, head_dim, seed)


@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 7])
def test_fwd_protocol_never_overruns_or_deadlocks(n_kv):
    for seed in range(300):
        assert run_schedule(n_kv, seed, kernel="fwd") is None, (n_kv, seed)


def test_checker_finds_the_unthrottled_staging_deadlock():
    """Without warpgroup 1's wait for the reducer, some schedule lets it stage
    two dQ halves ahead: stage_full[1] then overruns the reducer's wait."""
    found = False
    for seed in range(2000):
        try:
            out = run_schedule(6, seed, fixed=False)
        except Overrun as e:
            assert "stage_full1" in str(e)
            found = True
            break
        if out is not None:
            found = True
            break
    assert found
