"""A model of the tensor-core forward kernel's mbarrier protocol (no GPU).

The role loops of attn_fwd_tc_kernel (the TMA producer warp, the MMA warp and
the eight softmax warps of the two query tiles) are transcribed here at the
level of their barrier operations. TMA loads land in any order and tcgen05
commits complete in issue order, at random times. For random interleavings
over causal and non-causal item lists (ragged N, odd pair counts, one or many
items per CTA, both ring depths) the model checks two things: no schedule
deadlocks, and every wait observes exactly the phase it targets. mbarrier
try_wait.parity compares parities only, so a barrier two phases ahead of its
waiter (or one behind) would pass or block wrongly on the GPU. The model must
change together with the kernel's role loops.
"""

import random

import pytest


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; `done` counts completed phases."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count, f"{self.name}: too many arrivals"
        if self.pending == self.count:
            self.pending, self.done = 0, self.done + 1


def wait_phase(b, phase):
    """Wait, as try_wait.parity does, for phase `phase` of barrier `b` to complete;
    fail if the barrier is not exactly at that phase or the one after it."""
    while (b.done & 1) == (phase & 1):  # the parity test the hardware makes
        assert b.done == phase, f"{b.name}: waiting for phase {phase} with {b.done} complete"
        yield "blocked"
    assert b.done == phase + 1, f"{b.name}: passed phase {phase} with {b.done} complete"


def items_of(causal, BH, n_pairs, n_kt, G, cta):
    """The (key tiles of query tile 0, of query tile 1) of each item CTA `cta` takes (snake order)."""
    total = BH * n_pairs
    r = 0
    while r * G < total:
        item = r * G + ((G - 1 - cta) if r & 1 else cta)
        if item < total:
            if causal:
                pair = n_pairs - 1 - item // BH
                yield min(2 * pair + 1, n_kt), min(2 * pair + 2, n_kt)
            else:
                yield n_kt, n_kt
        r += 1


def run(seed, causal, BH, N, G, stages):
    rng = random.Random(seed)
    n_kt, n_pairs = (N + 127) // 128, (N + 255) // 256
    G = min(G, BH * n_pairs)  # the persistent grid: at most one CTA per item
    items = list(items_of(causal, BH, n_pairs, n_kt, G, rng.randrange(G)))
    assert items
    bars = {}
    for t in (0, 1):
        for name, count in (("q_full", 1), ("q_empty", 1), ("s_full", 1), ("p_lo", 4), ("p_hi", 4),
                            ("o_full", 1), ("o_empty", 4)):
            bars[f"{name}{t}"] = Barrier(f"{name}{t}", count)
    for i in range(stages):
        bars[f"slot_full{i}"] = Barrier(f"slot_full{i}", 1)
        bars[f"slot_empty{i}"] = Barrier(f"slot_empty{i}", 1)
    loads = []    # landed in any order
    commits = []  # completed in issue order

    def wait(name, phase):
        return wait_phase(bars[name], phase)

    def load(name):
        loads.append(name)

    def commit(name):
        commits.append(name)

    def producer():
        it = nq = 0

        def load_kv():
            nonlocal it
            if it >= stages:
                yield from wait(f"slot_empty{it % stages}", it // stages - 1)
            load(f"slot_full{it % stages}")
            it += 1

        def load_q(t):
            if nq > 0:
                yield from wait(f"q_empty{t}", nq - 1)
            load(f"q_full{t}")

        for k0, k1 in items:
            yield from load_q(0)
            yield from load_kv()
            yield from load_q(1)
            nq += 1
            for _ in range(1, 2 * k1):
                yield from load_kv()

    def mma():
        it = nq = 0
        npv = [0, 0]
        early_v = stages <= 5  # shallow ring: V_j's slot released before the next S, K_{j+1} only tested early
        for k0, k1 in items:
            yield from wait("q_full0", nq)
            yield from wait(f"slot_full{it % stages}", it // stages)
            commit("s_full0")
            if k0 == 1:
                commit("q_empty0")
            yield from wait("q_full1", nq)
            commit("s_full1")
            if k1 == 1:
                commit("q_empty1")
            commit(f"slot_empty{it % stages}")
            it += 1
            for j in range(k1):
                sv = it % stages
                yield from wait(f"slot_full{sv}", it // stages)
                itk = it + 1
                k_bar = f"slot_full{itk % stages}"
                # K_{j+1} before the P waits: a deep ring waits for it there, a
                # shallow one takes it there only if it has landed already
                k_ready = False
                if j + 1 < k1:
                    if early_v:
                        k_ready = bars[k_bar].done == itk // stages + 1
                    else:
                        yield from wait(k_bar, itk // stages)
                        k_ready = True
                for t in (0, 1):
                    kv_end = k1 if t else k0
                    if j < kv_end:
                        if j == 0 and nq > 0:
                            yield from wait(f"o_empty{t}", nq - 1)
                        yield from wait(f"p_lo{t}", npv[t])
                        yield from wait(f"p_hi{t}", npv[t])
                        if t == 1 and early_v:
                            commit(f"slot_empty{sv}")
                        if j + 1 < kv_end:
                            if not k_ready:
                                yield from wait(k_bar, itk // stages)
                                k_ready = True
                            commit(f"s_full{t}")
                            if j + 2 == kv_end:
                                commit(f"q_empty{t}")
                        npv[t] += 1
                        if j == kv_end - 1:
                            commit(f"o_full{t}")
                        if t == 1 and not early_v:
                            commit(f"slot_empty{sv}")
                    elif t == 1:
                        commit(f"slot_empty{sv}")
                if j + 1 < k1:
                    commit(f"slot_empty{itk % stages}")
                it += 2 if j + 1 < k1 else 1
            nq += 1

    def softmax_warp(t):
        ns = nq = 0
        for k0, k1 in items:
            for _ in range(k1 if t else k0):
                yield from wait(f"s_full{t}", ns)
                ns += 1
                yield "work"
                bars[f"p_lo{t}"].arrive()
                yield "work"
                bars[f"p_hi{t}"].arrive()
            yield from wait(f"o_full{t}", nq)
            bars[f"o_empty{t}"].arrive()
            nq += 1

    roles = [producer(), mma()] + [softmax_warp(t) for t in (0, 1) for _ in range(4)]
    alive = list(range(len(roles)))
    idle = 0
    while alive:
        if loads and rng.random() < 0.3:
            bars[loads.pop(rng.randrange(len(loads)))].arrive()
            idle = 0
        if commits and rng.random() < 0.3:
            bars[commits.pop(0)].arrive()
            idle = 0
        r = rng.choice(alive)
        try:
            step = next(roles[r])
        except StopIteration:
            alive.remove(r)
            idle = 0
            continue
        idle = idle + 1 if step == "blocked" else 0
        assert not (idle > 200 * len(alive) and not loads and not commits), f"deadlock, roles {alive} waiting"
    return True


CASES = [(True, 64, 2048, 152, 5), (True, 3, 300, 4, 5), (False, 2, 1000, 3, 8), (True, 1, 37, 1, 8),
         (False, 1, 1892, 2, 8), (True, 2, 640, 2, 5)]


@pytest.mark.parametrize("causal,BH,N,G,stages", CASES)
def test_forward_barrier_protocol_has_no_deadlock_or_phase_aliasing(causal, BH, N, G, stages):
    for seed in range(12):
        assert run(seed, causal, BH, N, G, stages)


def test_the_model_catches_a_barrier_two_phases_ahead():
    # Two completed phases look like none to a parity test: the model must report
    # the waiter that missed one, not let it block (or pass) silently.
    b = Barrier("x", 1)
    b.arrive()
    b.arrive()
    with pytest.raises(AssertionError):
        next(wait_phase(b, 0))
    # one phase ahead is the normal case: the waiter passes
    c = Barrier("y", 1)
    c.arrive()
    with pytest.raises(StopIteration):
        next(wait_phase(c, 0))


def run_backward(seed, items, slots, double_s, skip_acc_free_wait=False):
    """The persistent backward kernel's CTA: producer, MMA warp and the eight pass
    warps over a list of work items (key tiles), item r having items[r] query
    tiles, with `slots` Q/dO slots and, when `double_s`, the next query tile's S^T
    issued into a second buffer during the current pass (the d = 64 layout).
    Steps are numbered across items (T); per-step barriers take phase T, per-slot
    ones phase T // slots, per-item ones (kv, fin, acc_free) phase r.  The next
    item's K/V load waits until the last MMA that reads the current K/V has
    completed (fin), and its first dV/dK products until the epilogue has read the
    previous item's dV/dK out of TMEM (acc_free).  The dS^T shared buffer is
    written by every pass (each warp its own part) and, at d = 128, by each
    item's epilogue, which stages dV and dK there for their stores; every
    step's dQ product reads all of it.  The model checks that no write lands
    while a dQ product that reads the buffer may still be running (for the
    epilogue the last step's drain, which waits for that step's dQ, already
    ensures it), and that no dQ product is issued while a warp is still
    staging its epilogue there."""
    rng = random.Random(seed)
    bars = {name: Barrier(name, count) for name, count in (
        ("kv", 1), ("s_full", 1), ("dq_full", 1), ("drain_done", 8), ("fin", 1), ("acc_free", 8), ("p_full0", 8),
        ("p_full1", 8))}
    for s in range(slots):
        for name, count in (("q_full", 1), ("q_empty", 1), ("stage_free", 8)):
            bars[f"{name}{s}"] = Barrier(f"{name}{s}", count)
    loads, commits = [], []
    total = sum(items)

    def slot(t):
        return t % slots

    def use(t):
        return t // slots  # phase index of slot(t)'s barriers for step t

    def wait(name, phase):
        return wait_phase(bars[name], phase)

    reduced = []
    stored = []
    acc_read = [0] * len(items)  # pass warps that have read item r's dV, dK out of TMEM
    dq_done = [0]                # dQ products completed (the dq_full commit follows each one)
    epi_done = [0] * 8           # items whose epilogue staging each pass warp has finished

    def producer():
        def finish_tile(t):  # dQ of step t staged: reduce-add it, then the slot is free
            yield from wait(f"stage_free{slot(t)}", use(t))
            reduced.append(t)
            yield "work"

        T = 0
        for r, n_it in enumerate(items):
            for it in range(n_it):
                if T >= slots:
                    yield from finish_tile(T - slots)
                loads.append(f"q_full{slot(T)}")
                if it == 0:
                    if r > 0:
                        yield from wait("fin", r - 1)  # the previous item's K/V are no longer read
                        assert bars["fin"].done >= r, "K/V reloaded while the previous item's MMAs may read them"
                    loads.append("kv")
                T += 1
        for t in range(max(0, total - slots), total):
            yield from finish_tile(t)

    def mma():
        T = 0
        for r, n_it in enumerate(items):
            yield from wait("kv", r)
            yield from wait(f"q_full{slot(T)}", use(T))
            if T > 0:
                yield from wait("drain_done", T - 1)  # S^T columns: the previous step's dQ is out
            commits.append("s_full")
            for it in range(n_it):
                s = slot(T)
                if double_s and it + 1 < n_it:
                    yield from wait(f"q_full{slot(T + 1)}", use(T + 1))
                    if it > 0:
                        yield from wait("drain_done", T - 1)
                if it == 0 and r > 0:
                    if not skip_acc_free_wait:
                        yield from wait("acc_free", r - 1)  # dV, dK of the previous item read out
                    # the first dV/dK products of item r overwrite the accumulators
                    assert acc_read[r - 1] == 8, f"item {r} overwrites dV/dK before item {r - 1} was read"
                yield from wait("p_full0", T)
                yield from wait("p_full1", T)
                commits.append(f"q_empty{s}")
                # dQ = dS K reads the whole dS^T buffer: no warp may still be staging an epilogue in it
                assert all(e == r for e in epi_done), f"dQ of step {T} issued during an epilogue's staging"
                commits.append("dq_full")
                if it + 1 < n_it:
                    if not double_s:
                        yield from wait(f"q_full{slot(T + 1)}", use(T + 1))
                        yield from wait("drain_done", T)
                    commits.append("s_full")
                T += 1
            commits.append("fin")
        yield from wait("fin", len(items) - 1)

    def pass_warp(w):
        T = 0
        for r, n_it in enumerate(items):
            for it in range(n_it):
                s = slot(T)
                yield from wait("s_full", T)
                yield from wait(f"q_full{s}", use(T))
                # this pass writes its part of dS^T: every earlier dQ product has read the buffer
                assert dq_done[0] >= T, f"dS^T of step {T} written while an earlier dQ may read it"
                yield "work"
                bars["p_full0"].arrive()
                yield "work"
                bars["p_full1"].arrive()
                yield from wait("dq_full", T)
                yield "work"
                bars["drain_done"].arrive()
                yield from wait(f"q_empty{s}", use(T))
                yield "work"
                bars[f"stage_free{s}"].arrive()
                T += 1
            yield from wait("fin", r)
            # the epilogue stages dV, dK in this warp's part of dS^T: the item's dQ products are done
            assert dq_done[0] >= T, f"item {r}'s epilogue staged while its last dQ may read dS^T"
            yield "work"
            acc_read[r] += 1
            bars["acc_free"].arrive()
            yield "work"  # the stores have read the staging
            epi_done[w] += 1
            if w == 0:
                stored.append(r)

    roles = [producer(), mma()] + [pass_warp(w) for w in range(8)]
    alive = list(range(len(roles)))
    idle = 0
    while alive:
        if loads and rng.random() < 0.3:
            bars[loads.pop(rng.randrange(len(loads)))].arrive()
            idle = 0
        if commits and rng.random() < 0.3:
            c = commits.pop(0)
            if c == "dq_full":
                dq_done[0] += 1
            bars[c].arrive()
            idle = 0
        r = rng.choice(alive)
        try:
            step = next(roles[r])
        except StopIteration:
            alive.remove(r)
            idle = 0
            continue
        idle = idle + 1 if step == "blocked" else 0
        assert not (idle > 200 * len(alive) and not loads and not commits), f"deadlock, roles {alive} waiting"
    assert sorted(reduced) == list(range(total)), "every step's dQ is reduced exactly once"
    assert stored == list(range(len(items))), "every item's dK, dV stored once, in order"
    return True


@pytest.mark.parametrize("items", [[1], [2], [16], [3, 1, 5], [1, 1, 1, 1], [16, 2, 7], [2, 3]])
@pytest.mark.parametrize("slots,double_s", [(2, False), (3, True)])
def test_backward_barrier_protocol_has_no_deadlock_or_phase_aliasing(items, slots, double_s):
    for seed in range(12):
        assert run_backward(seed, items, slots, double_s)


def test_the_backward_model_catches_a_missing_accumulator_hand_off():
    with pytest.raises(AssertionError, match="overwrites dV/dK"):
        for seed in range(50):
            run_backward(seed, [2, 2, 2], 2, False, skip_acc_free_wait=True)
