"""CPU models of the attention kernels' synchronisation (bit_exact_attention_gb300/csrc/
sage2_attention.cu). For attn_pp, the two-tile kernel, the model has a producer, a Q K^T issuer
and a P~V issuer (separate threads with blocking waits in a fixed order, so separate in-order
pipes whose commits track only their own MMAs), and the softmax warps of both tiles. For attn_fwd, the one-tile kernel, it has two issuers
with their own pipes, softmax and fold warps, a 4-slot alpha ring and double-buffered P~ and R.
In both, the agents meet on mbarriers that are waited on by phase parity, as the hardware does.

Random interleavings (seeded) are checked for:
  * parity aliasing: a wait must only pass once the awaited phase has completed, and not when
    its barrier has run two phases further;
  * buffer hazards: S_t, the two P~ buffers of each tile, O_t and the K, V and DeltaS stages are
    only rewritten once every reader of the old contents is done, and only read once written;
  * deadlock: every run finishes.
The models follow the kernels' conditions one for one. Each has deliberately broken variants
that must be caught. For the two-tile kernel these are: QK(n) issued without waiting for
PV(n-2) to complete, one P~V completion barrier per tile instead of one per P~ buffer, and the
DeltaS stage released with the K stage. For
the one-tile kernel: the R-free wait removed, and a single-slot alpha ring (a 2-slot ring fails
as well, while 3 would do; the kernel keeps 4 for mask indexing).
"""
from __future__ import annotations

import random

import pytest


class Hazard(AssertionError):
    pass


class Bar:
    """mbarrier: `count` arrivals complete a phase; waiters test the phase parity."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.c = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.c += 1
            self.pending = self.count

    def passes(self, n):
        """Parity test for phase n (what try_wait.parity(n & 1) answers)."""
        ok = (self.c & 1) != (n & 1)
        if ok and self.c != n + 1:
            raise Hazard(f"{self.name}: wait for phase {n} passed with {self.c} completions")
        return ok


class Model:
    """attn_pp's protocol. Three rings: K (ST stages, released by the Q K^T issuer once QK_0(n)
    and QK_1(n) complete), V (ST stages) and DeltaS*c / K scales (DS stages, read by the softmax),
    both released by the P~V issuer once PV_0(n) and PV_1(n) complete. One producer loads K and
    DeltaS, a second one V. Both issuers take n = 0, 1, ..., tile 0 then tile 1, with blocking
    waits. QK_t(n) is issued once the softmax read S_t(n-1), PV_t(n-2) completed, K(n) and
    DeltaS(n) landed; PV_t(n) once P~_t(n) is written and V(n) landed. pv_done[t][b] completes
    for the PVs of P~ buffer b. The softmax stores P~_t(j), rescales O_t after waiting for
    PV_t(j-1), then hands P~ over."""

    def __init__(self, T0, T1, ST, W, rng, resc_p, qk_after_pv=True, pv_bar_per_buffer=True,
                 DS=4, d_released_by_qk=False, sm_weight=1.0):
        self.T, self.ST, self.DS, self.W, self.rng = (T0, T1), ST, DS, W, rng
        self.Tmax = max(T0, T1)
        self.resc_p, self.qk_after_pv, self.d_released_by_qk = resc_p, qk_after_pv, \
            d_released_by_qk
        self.sm_weight = sm_weight  # < 1: softmax warps take steps less often (slow softmax)
        B = Bar
        self.full = {r: [B(f"{r}_full{s}", 1) for s in range(self.depth(r))] for r in "kvd"}
        self.empty = {r: [B(f"{r}_empty{s}", 1) for s in range(self.depth(r))] for r in "kvd"}
        self.s_full = [B(f"s_full{t}", 1) for t in range(2)]
        self.s_free = [B(f"s_free{t}", W) for t in range(2)]
        self.p_full = [[B(f"p_full{t}{b}", W) for b in range(2)] for t in range(2)]
        if pv_bar_per_buffer:
            self.pv_done = [[B(f"pv_done{t}{b}", 1) for b in range(2)] for t in range(2)]
            self.pv_phase = lambda n: n >> 1
        else:  # one barrier per tile, completed by every PV
            one = [B(f"pv_done{t}", 1) for t in range(2)]
            self.pv_done = [[one[t], one[t]] for t in range(2)]
            self.pv_phase = lambda n: n
        self.pipes = {"qk": [], "pv": []}   # one in-order pipe per issuing thread
        self.stage = {r: [None] * self.depth(r) for r in "kvd"}  # tile held by each stage
        self.stage_users = {r: {} for r in "kvd"}                # tile -> readers not yet done
        self.S = [None, None]                # QK index whose result S_t holds
        self.s_read = [[-1] * W for _ in range(2)]   # last S_t(j) read by each warp
        self.P = [[[None] * W for _ in range(2)] for _ in range(2)]  # P~ tile in buffer
        self.pv_completed = [0, 0]
        self.events = 0                      # steps taken by agents other than the issuers

    # ------------------------------------------------------------ helpers
    def depth(self, ring):
        return self.DS if ring == "d" else self.ST

    def use_stage(self, ring, n, who):
        s = n % self.depth(ring)
        if self.stage[ring][s] != n:
            raise Hazard(f"{who} reads {ring} tile {n} but stage {s} holds {self.stage[ring][s]}")

    def release_stage_user(self, ring, n, who):
        self.stage_users[ring][n].discard(who)

    def pv_wait(self, t, n):
        """The barrier and phase that PV_t(n)'s completion moves."""
        return self.pv_done[t][n & 1], self.pv_phase(n)

    # ------------------------------------------------------------ agents (generators)
    def load(self, ring, j, users):
        d = self.depth(ring)
        s = j % d
        if j >= d:
            yield ("wait", self.empty[ring][s], j // d - 1)
            old = j - d
            if self.stage_users[ring].get(old):
                raise Hazard(f"{ring} stage {s} reloaded while "
                             f"{sorted(self.stage_users[ring][old])} still read tile {old}")
        self.stage[ring][s] = j
        self.stage_users[ring][j] = users
        yield ("act", self.full[ring][s].arrive)

    def producer(self):  # K and DeltaS
        for j in range(self.Tmax):
            live = [t for t in range(2) if j < self.T[t]]
            yield from self.load("k", j, {("QK", t) for t in live})
            yield from self.load("d", j, {("SM", t, w) for t in live for w in range(self.W)})

    def producer_v(self):
        for j in range(self.Tmax):
            yield from self.load("v", j, {("PV", t) for t in range(2) if j < self.T[t]})

    def qk_issuer(self):
        """Fixed order n = 0, 1, ..., tile 0 then tile 1, each condition a blocking wait."""
        for n in range(self.Tmax):
            for t in range(2):
                if n >= self.T[t]:
                    continue
                if n > 0:
                    yield ("wait", self.s_free[t], n - 1)
                if self.qk_after_pv and n >= 2:
                    yield ("wait", *self.pv_wait(t, n - 2))
                yield ("wait", self.full["k"][n % self.ST], n // self.ST)
                yield ("wait", self.full["d"][n % self.DS], n // self.DS)
                if n > 0 and min(self.s_read[t]) < n - 1:
                    raise Hazard(f"QK{t}({n}) issued before S{t}({n - 1}) was read")
                self.pipes["qk"] += [("QK", t, n), ("commit", self.s_full[t])]
            self.pipes["qk"].append(("commit", self.empty["k"][n % self.ST]))
            if self.d_released_by_qk:
                self.pipes["qk"].append(("commit", self.empty["d"][n % self.DS]))

    def pv_issuer(self):
        for n in range(self.Tmax):
            for t in range(2):
                if n >= self.T[t]:
                    continue
                yield ("wait", self.p_full[t][n & 1], n >> 1)
                yield ("wait", self.full["v"][n % self.ST], n // self.ST)
                for w in range(self.W):
                    if self.P[t][n & 1][w] != n:
                        raise Hazard(f"PV{t}({n}) issued but warp {w}'s P~ buffer holds "
                                     f"{self.P[t][n & 1][w]}")
                bar, _ = self.pv_wait(t, n)
                self.pipes["pv"] += [("PV", t, n), ("commit", bar)]
            self.pipes["pv"].append(("commit", self.empty["v"][n % self.ST]))
            if not self.d_released_by_qk:
                self.pipes["pv"].append(("commit", self.empty["d"][n % self.DS]))

    def pipe_step(self, name):
        kind = self.pipes[name].pop(0)
        if kind[0] == "commit":  # at the head: everything issued before it has completed
            kind[1].arrive()
            return
        _, t, n = kind
        if kind[0] == "QK":
            self.use_stage("k", n, f"QK{t}({n})")
            self.S[t] = n
            self.release_stage_user("k", n, ("QK", t))
        else:
            self.use_stage("v", n, f"PV{t}({n})")
            if self.pv_completed[t] != n:
                raise Hazard(f"PV{t}({n}) out of order")
            self.pv_completed[t] += 1
            self.release_stage_user("v", n, ("PV", t))

    def softmax(self, t, w):
        T = self.T[t]
        for j in range(T):
            yield ("wait", self.s_full[t], j)
            if self.S[t] != j:
                raise Hazard(f"softmax{t}.{w} reads S{t}({j}) but S holds {self.S[t]}")
            self.s_read[t][w] = j
            yield ("act", self.s_free[t].arrive)
            yield ("act", lambda: None)  # the logits read DeltaS(j) (landed: QK_t(j) waited)
            self.use_stage("d", j, f"softmax{t}.{w} DeltaS({j})")
            self.release_stage_user("d", j, ("SM", t, w))
            # P~_t(j) is stored while the exponentials run, before the rescale
            if self.pv_completed[t] < j - 1:
                raise Hazard(f"softmax{t}.{w} overwrites P~ buffer {j & 1} before PV{t}({j - 2})")
            self.P[t][j & 1][w] = j
            yield ("act", lambda: None)
            if j > 0 and self.rng.random() < self.resc_p:
                bar, ph = self.pv_wait(t, j - 1)
                yield ("wait", bar, ph)
                if self.pv_completed[t] != j:
                    raise Hazard(f"softmax{t}.{w} rescales O{t} at {j} with "
                                 f"{self.pv_completed[t]} PVs complete")
            yield ("act", self.p_full[t][j & 1].arrive)
        if T > 0:
            bar, ph = self.pv_wait(t, T - 1)
            yield ("wait", bar, ph)
            if self.pv_completed[t] != T:
                raise Hazard(f"epilogue{t}.{w} reads O{t} with {self.pv_completed[t]} of {T} PVs")

    # ------------------------------------------------------------ scheduler
    def run(self, max_steps=300000):
        agents = {"producer": self.producer(), "producer_v": self.producer_v(),
                  "qk": self.qk_issuer(), "pv": self.pv_issuer()}
        for t in range(2):
            for w in range(self.W):
                agents[f"sm{t}{w}"] = self.softmax(t, w)
        pending = {k: None for k in agents}  # the action each agent is blocked on
        idle = set()                         # issuers that polled without progress
        for _ in range(max_steps):
            runnable = []
            for k, req in pending.items():
                if k not in agents:
                    continue
                if req is None:
                    runnable.append(k)
                elif req[0] == "wait":
                    if (req[1].c & 1) != (req[2] & 1):
                        runnable.append(k)
                elif req[0] == "poll":
                    if not (k in idle and not req[1]):
                        runnable.append(k)
            runnable += [("pipe", p) for p in ("qk", "pv") if self.pipes[p]]
            if not runnable:
                if not agents:
                    return
                raise Hazard("deadlock: " + ", ".join(
                    f"{k}:{pending[k][0]} {getattr(pending[k][1], 'name', '')}"
                    for k in agents if pending[k]))
            if self.sm_weight < 1.0:
                fast = [k for k in runnable if not (isinstance(k, str) and k.startswith("sm"))
                        or self.rng.random() < self.sm_weight]
                runnable = fast or runnable
            k = self.rng.choice(runnable)
            if k not in ("qk", "pv"):
                self.events += 1
                idle.clear()
            if isinstance(k, tuple):
                self.pipe_step(k[1])
                continue
            req = pending[k]
            if req is not None and req[0] == "wait":
                req[1].passes(req[2])  # raises on aliasing
            try:
                nxt = next(agents[k])
            except StopIteration:
                del agents[k]
                pending[k] = None
                continue
            if nxt[0] == "act":
                nxt[1]()
                pending[k] = None
                idle.clear()
            else:
                pending[k] = nxt
                if nxt[0] == "poll":
                    if nxt[1]:
                        idle.discard(k)
                    else:
                        idle.add(k)
        raise Hazard("step limit")


CASES = [(T0, T1, ST, DS) for (T0, T1) in [(0, 1), (1, 1), (1, 2), (2, 3), (3, 3), (5, 6), (4, 4),
                                           (0, 3), (6, 2), (9, 10)]
         for ST, DS in ((2, 2), (3, 4), (6, 4), (3, 6))]


@pytest.mark.parametrize("T0,T1,ST,DS", CASES)
def test_two_tile_protocol_has_no_aliasing_hazard_or_deadlock(T0, T1, ST, DS):
    for seed in range(40):
        rng = random.Random(seed * 1009 + T0 * 31 + T1 * 7 + ST + 13 * DS)
        Model(T0, T1, ST, W=2, rng=rng, resc_p=rng.choice([0.0, 0.15, 0.5, 1.0]), DS=DS,
              sm_weight=rng.choice([1.0, 0.1])).run()


def _caught(**kw):
    for seed in range(400):
        rng = random.Random(seed)
        T0, T1 = rng.choice([(3, 4), (4, 4), (5, 6), (2, 3)])
        try:
            Model(T0, T1, 3, W=2, rng=rng, resc_p=rng.choice([0.0, 0.5]),
                  sm_weight=rng.choice([1.0, 0.1]), **kw).run()
        except Hazard:
            return True
    return False


def test_model_catches_qk_issued_before_pv_two_back_completed():
    """QK(n) before PV(n-2) completes lets the softmax refill the P~ buffer that PV(n-2) has not
    read yet."""
    assert _caught(qk_after_pv=False)


def test_model_catches_deltas_stage_released_after_the_qk_products():
    """Releasing a DeltaS*c stage when the Q K^T products complete lets the producer refill it
    while the softmax still reads it."""
    assert _caught(d_released_by_qk=True)


def test_model_catches_one_pv_barrier_per_tile():
    """With one P~V completion barrier per tile, a waiter for PV(n-2) can find PV(n-1) complete
    as well: the barrier is two phases on, the parity test fails and the wait can never end."""
    assert _caught(pv_bar_per_buffer=False)


# ---------------------------------------------------------------------- one-tile kernel
class OneTileModel:
    """attn_fwd's protocol: a Q K^T issuer and a P~V issuer (separate threads, so separate
    in-order pipes whose commits track only their own MMAs), four softmax and four fold warps
    (modelled with W each), a 4-slot alpha ring, double-buffered P~ and R."""

    def __init__(self, T, ST, W, rng, r_free_wait=True, ring=4):
        self.T, self.ST, self.W, self.rng, self.r_free_wait, self.ring = T, ST, W, rng, \
            r_free_wait, ring
        B = Bar
        self.q_full = B("q_full", W)
        self.kv_full = [B(f"kv_full{s}", 1) for s in range(ST)]
        self.kv_empty = [B(f"kv_empty{s}", 1) for s in range(ST)]
        self.s_full, self.s_free = B("s_full", 1), B("s_free", W)
        self.p_full = [B(f"p_full{b}", W) for b in range(2)]
        self.pv_done = [B(f"pv_done{b}", 1) for b in range(2)]
        self.r_free = [B(f"r_free{b}", W) for b in range(2)]
        self.a_full = [B(f"a_full{s}", W) for s in range(ring)]
        self.l_full = B("l_full", W)
        self.pipes = {"qk": [], "pv": []}
        self.stage, self.stage_users = [None] * ST, {}
        self.S, self.s_read = None, [-1] * W
        self.P = [[None] * W for _ in range(2)]
        self.R = [None, None]
        self.r_read = [[-1] * W for _ in range(2)]
        self.alpha = [[None] * W for _ in range(ring)]
        self.pv_completed = 0
        self.qk_completed = 0
        self.folded = [-1] * W

    def use_stage(self, n, who):
        if self.stage[n % self.ST] != n:
            raise Hazard(f"{who} reads KV tile {n} but its stage holds {self.stage[n % self.ST]}")

    def producer(self):
        for j in range(self.T):
            s = j % self.ST
            if j >= self.ST:
                yield ("wait", self.kv_empty[s], j // self.ST - 1)
                if self.stage_users.get(j - self.ST):
                    raise Hazard(f"stage {s} reloaded while {sorted(self.stage_users[j - self.ST])}"
                                 f" still read KV tile {j - self.ST}")
            self.stage[s] = j
            self.stage_users[j] = {"QK", "PV"} | {("SM", w) for w in range(self.W)}
            yield ("act", self.kv_full[s].arrive)

    def qk_issuer(self):
        yield ("wait", self.q_full, 0)
        for j in range(self.T):
            if j:
                yield ("wait", self.s_free, j - 1)
                if min(self.s_read) < j - 1:
                    raise Hazard(f"QK({j}) issued before S({j - 1}) was read")
            yield ("wait", self.kv_full[j % self.ST], j // self.ST)
            self.pipes["qk"] += [("QK", j), ("commit", self.s_full)]

    def pv_issuer(self):
        for j in range(self.T):
            b = j & 1
            yield ("wait", self.p_full[b], j >> 1)
            if j >= 2 and self.r_free_wait:
                yield ("wait", self.r_free[b], (j - 2) >> 1)
            if any(p != j for p in self.P[b]):
                raise Hazard(f"PV({j}) issued but the P~ buffer holds {self.P[b]}")
            if self.qk_completed <= j:
                raise Hazard(f"stage of KV tile {j} released before QK({j}) completed")
            self.pipes["pv"] += [("PV", j), ("commit", self.pv_done[b]),
                                 ("commit", self.kv_empty[j % self.ST])]

    def pipe_step(self, name):
        head = self.pipes[name].pop(0)
        if head[0] == "commit":
            head[1].arrive()
            return
        j = head[1]
        self.use_stage(j, f"{head[0]}({j})")
        if head[0] == "QK":
            self.S = j
            self.qk_completed = j + 1
            self.stage_users[j].discard("QK")
        else:
            b = j & 1
            if j >= 2 and min(self.r_read[b]) < j - 2:
                raise Hazard(f"PV({j}) overwrites R{b} before the fold read R({j - 2})")
            self.R[b] = j
            self.pv_completed = j + 1
            self.stage_users[j].discard("PV")

    def softmax(self, w):
        yield ("act", self.q_full.arrive)
        jprev = None

        def hand_over(n):
            slot = n % self.ring
            if n >= self.ring and self.folded[w] < n - self.ring:
                raise Hazard(f"alpha({n}) overwrites slot {slot} before the fold read "
                             f"alpha({n - self.ring})")
            self.alpha[slot][w] = n

        for j in range(self.T):
            yield ("wait", self.s_full, j)
            if self.S != j:
                raise Hazard(f"softmax {w} reads S({j}) but S holds {self.S}")
            self.s_read[w] = j
            yield ("act", self.s_free.arrive)
            if jprev is not None:
                hand_over(jprev)
                yield ("act", self.p_full[jprev & 1].arrive)
                yield ("act", self.a_full[jprev % self.ring].arrive)
            yield ("wait", self.kv_full[j % self.ST], j // self.ST)
            if j >= 2:
                yield ("wait", self.pv_done[j & 1], (j - 2) >> 1)
            self.use_stage(j, f"softmax {w} DeltaS({j})")
            self.stage_users[j].discard(("SM", w))
            if self.pv_completed < j - 1:
                raise Hazard(f"softmax {w} overwrites P~ buffer {j & 1} before PV({j - 2})")
            self.P[j & 1][w] = j
            jprev = j
        if jprev is not None:
            hand_over(jprev)
            yield ("act", self.p_full[jprev & 1].arrive)
            yield ("act", self.a_full[jprev % self.ring].arrive)
        yield ("act", self.l_full.arrive)

    def fold(self, w):
        for j in range(self.T):
            yield ("wait", self.a_full[j % self.ring], j // self.ring)
            if self.alpha[j % self.ring][w] != j:
                raise Hazard(f"fold {w} reads alpha({j}) but the slot holds "
                             f"{self.alpha[j % self.ring][w]}")
            self.folded[w] = j
            yield ("wait", self.pv_done[j & 1], j >> 1)
            if self.R[j & 1] != j:
                raise Hazard(f"fold {w} reads R({j}) but R{j & 1} holds {self.R[j & 1]}")
            self.r_read[j & 1][w] = j
            yield ("act", self.r_free[j & 1].arrive)
        yield ("wait", self.l_full, 0)
        if self.pv_completed != self.T:
            raise Hazard("epilogue before every PV completed")

    def run(self, max_steps=200000):
        agents = {"producer": self.producer(), "qk": self.qk_issuer(), "pv": self.pv_issuer()}
        for w in range(self.W):
            agents[f"sm{w}"] = self.softmax(w)
            agents[f"fold{w}"] = self.fold(w)
        pending = {k: None for k in agents}
        for _ in range(max_steps):
            choices = [k for k in agents if pending[k] is None or
                       (pending[k][1].c & 1) != (pending[k][2] & 1)]
            choices += [("pipe", p) for p in ("qk", "pv") if self.pipes[p]]
            if not choices:
                if agents:
                    raise Hazard("deadlock: " + ", ".join(
                        f"{k}:{pending[k][1].name}" for k in agents if pending[k]))
                return
            k = self.rng.choice(choices)
            if isinstance(k, tuple):
                self.pipe_step(k[1])
                continue
            if pending[k] is not None:
                pending[k][1].passes(pending[k][2])  # raises on aliasing
            try:
                nxt = next(agents[k])
            except StopIteration:
                del agents[k]
                continue
            if nxt[0] == "act":
                nxt[1]()
                pending[k] = None
            else:
                pending[k] = nxt
        raise Hazard("step limit")


@pytest.mark.parametrize("T,ST", [(T, ST) for T in (1, 2, 3, 5, 8, 13) for ST in (2, 4, 6)])
def test_one_tile_protocol_has_no_aliasing_hazard_or_deadlock(T, ST):
    for seed in range(40):
        OneTileModel(T, ST, W=2, rng=random.Random(seed * 131 + T * 7 + ST)).run()


def test_one_tile_model_catches_a_missing_r_free_wait_and_a_short_alpha_ring():
    def caught(**kw):
        for seed in range(300):
            try:
                OneTileModel(8, 4, W=2, rng=random.Random(seed), **kw).run()
            except Hazard:
                return True
        return False
    assert caught(r_free_wait=False)
    assert caught(ring=1)
