"""A randomized model of the ring protocol of the int8 token-row GEMM
(csrc/gemm_tc_w8.cu), run on the CPU.

Agents: the activation and raw-weight copy producers, four converter groups
taking k-steps in turn, and the MMA issuer.  They share S = 3 converted
stages, 4 raw stages and 12 stage-free barriers indexed by k-step.  The
mbarriers are parity-wait barriers, as in the kernel.  Copies and MMAs
complete after random latencies, and the agents interleave at random.  The
model checks:
  - every read sees the data of the k-step it waits for;
  - no stage is rewritten while the MMA that reads it is still running;
  - nothing deadlocks.
It checks the barrier protocol of both converter orderings:
  - "widen after the stage-free wait" (the kernel's);
  - "read the raw stage into registers, release it, then wait".
The second one was not byte-identical on the GPU; the model finds no
protocol fault in either, which places that fault below the protocol, in
the memory ordering.
"""
import random

import pytest

S, RS, NG, FREE = 3, 4, 4, 12


class Bar:
    """Parity-wait mbarrier: `done(p)` is true once the phase of parity p has
    completed (a fresh barrier reads parity 1 as completed)."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "over-arrival"
        if self.pending == 0:
            self.phase ^= 1
            self.pending = self.count

    def done(self, parity):
        return parity != self.phase


def run(N, staged, seed):
    rng = random.Random(seed)
    ab_empty = [Bar(1) for _ in range(FREE)]
    a_full = [Bar(1) for _ in range(S)]
    b_full = [Bar(1) for _ in range(S)]
    q_full = [Bar(1) for _ in range(RS)]
    q_empty = [Bar(1) for _ in range(RS)]
    rawslot, astage, bstage = [None] * RS, [None] * S, [None] * S
    reading = [None] * S               # k-step whose MMA still reads stage s
    events, now, last_done = [], [0], [0]

    def later(dt, fn):
        events.append((now[0] + dt, fn))

    def stage_free(seq):
        if seq < S:
            return lambda: True
        q = seq - S
        return lambda: ab_empty[q % FREE].done((q // FREE) & 1)

    def a_prod():
        for seq in range(N):
            yield stage_free(seq)
            s = seq % S
            assert reading[s] is None, "activation copy over a stage being read"

            def land(seq=seq, s=s):
                astage[s] = seq
                a_full[s].arrive()
            later(rng.randint(1, 30), land)

    def q_prod():
        for seq in range(N):
            r = seq % RS
            ph = (seq // RS) & 1
            yield (lambda r=r, ph=ph: q_empty[r].done(ph ^ 1))

            def land(seq=seq, r=r):
                rawslot[r] = seq
                q_full[r].arrive()
            later(rng.randint(5, 60), land)

    def conv(g):
        for seq in range(g, N, NG):
            s, r = seq % S, seq % RS
            yield (lambda r=r, seq=seq: q_full[r].done((seq // RS) & 1))
            if staged:
                assert rawslot[r] == seq, "raw stage holds another k-step"
                q_empty[r].arrive()
                yield stage_free(seq)
            else:
                yield stage_free(seq)
                assert rawslot[r] == seq, "raw stage holds another k-step"
            assert reading[s] is None, "widened rows written over a stage being read"
            bstage[s] = seq
            yield (lambda: True)
            b_full[s].arrive()
            if not staged:
                q_empty[r].arrive()

    def mma():
        for seq in range(N):
            s, ph = seq % S, (seq // S) & 1
            yield (lambda s=s, ph=ph: a_full[s].done(ph) and b_full[s].done(ph))
            assert astage[s] == seq and bstage[s] == seq, "MMA reads another k-step"
            reading[s] = seq

            def finish(seq=seq, s=s):
                assert astage[s] == seq and bstage[s] == seq, "stage changed under the MMA"
                reading[s] = None
                ab_empty[seq % FREE].arrive()
            # MMAs complete in issue order (a commit tracks every earlier MMA)
            last_done[0] = max(last_done[0] + 1, now[0] + rng.randint(1, 40))
            events.append((last_done[0], finish))
            yield (lambda: True)

    agents = [a_prod(), q_prod(), mma()] + [conv(g) for g in range(NG)]
    waits = [next(a) for a in agents]
    alive = [True] * len(agents)
    for _ in range(10 ** 6):
        if not any(alive) and not events:
            return
        ready = [i for i in range(len(agents)) if alive[i] and waits[i]()]
        if ready and (not events or rng.random() < 0.7):
            i = rng.choice(ready)
            try:
                waits[i] = next(agents[i])
            except StopIteration:
                alive[i] = False
        elif events:
            events.sort(key=lambda e: e[0])
            t, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
        else:
            raise AssertionError("deadlock")
    raise AssertionError("no progress")


@pytest.mark.parametrize("staged", [False, True])
def test_token_row_int8_ring_protocol(staged):
    for seed in range(400):
        run(72, staged, seed)


def test_model_catches_an_early_stage_free_wait():
    """The model is not vacuous: with the stage-free wait one k-step early
    (for k-step seq - S - 1 instead of seq - S, the stage's last reader),
    some schedule rewrites a stage under its MMA."""
    caught = 0
    for seed in range(100):
        try:
            _run_early(48, seed)
        except AssertionError:
            caught += 1
    assert caught > 0


def _run_early(N, seed):
    """Activation copies and MMAs only, with the early stage-free wait."""
    rng = random.Random(seed)
    ab_empty = [Bar(1) for _ in range(FREE)]
    a_full = [Bar(1) for _ in range(S)]
    astage, reading = [None] * S, [None] * S
    events, now, last_done = [], [0], [0]

    def stage_free(seq):
        if seq < S + 1:
            return lambda: True
        q = seq - S - 1
        return lambda: ab_empty[q % FREE].done((q // FREE) & 1)

    def a_prod():
        for seq in range(N):
            yield stage_free(seq)
            s = seq % S
            assert reading[s] is None, "activation copy over a stage being read"

            def land(seq=seq, s=s):
                astage[s] = seq
                a_full[s].arrive()
            events.append((now[0] + rng.randint(1, 30), land))

    def mma():
        for seq in range(N):
            s, ph = seq % S, (seq // S) & 1
            yield (lambda s=s, ph=ph: a_full[s].done(ph))
            assert astage[s] == seq, "MMA reads another k-step"
            reading[s] = seq

            def finish(seq=seq, s=s):
                reading[s] = None
                ab_empty[seq % FREE].arrive()
            last_done[0] = max(last_done[0] + 1, now[0] + rng.randint(1, 40))
            events.append((last_done[0], finish))
            yield (lambda: True)

    agents = [a_prod(), mma()]
    waits = [next(a) for a in agents]
    alive = [True, True]
    for _ in range(10 ** 5):
        if not any(alive) and not events:
            return
        ready = [i for i in range(2) if alive[i] and waits[i]()]
        if ready and (not events or rng.random() < 0.7):
            i = rng.choice(ready)
            try:
                waits[i] = next(agents[i])
            except StopIteration:
                alive[i] = False
        elif events:
            events.sort(key=lambda e: e[0])
            t, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
        else:
            raise AssertionError("deadlock")
