"""CPU model of the decode GEMV's stage ring (host logic, no GPU).

The kernel has one producer warp and two consumer sets that take alternate
stages; stage i sits in slot i mod R with a full and an empty mbarrier, and
every wait is a parity wait. A data stage lands some time after it is issued
(tensor copies may complete in any order); a mark stage (flush or end mark)
completes at issue. The model runs every actor under random interleavings and
checks that a set only ever consumes its own stage j, after it landed.

With an odd slot count a set's two successive stages in one slot are two
phases apart, and a bare parity wait can pass on the phase before the other
set's stage: the model finds such runs. The kernel's consumers also wait for
the slot's descriptor to carry j (the producer writes it only after the slot's
previous stage was released); with that gate the model finds none, and no
deadlock, for R = 2..6.
"""
from __future__ import annotations

import random


def _try_wait(completed: int, parity: int) -> bool:
    # mbarrier.try_wait.parity: true once the phase of that parity is complete
    return (completed & 1) != parity


def _run(R: int, kinds: list[str], seq_gate: bool, rng: random.Random) -> str:
    T = len(kinds)
    full = [0] * R    # completed phases of each slot's full barrier
    empty = [0] * R   # completed phases of each slot's empty barrier
    desc = [None] * R  # (stage index, kind) last written to the slot
    landed: set[int] = set()
    in_flight: list[int] = []
    nxt = 0
    want = [0, 1]     # each set's next stage
    done = [False, False]
    for _ in range(100000):
        if nxt >= T and all(done) and not in_flight:
            return "ok"
        acts = []
        if nxt < T and _try_wait(empty[nxt % R], ((nxt // R) & 1) ^ 1):
            acts.append(("issue", 0))
        acts += [("land", st) for st in in_flight]
        for s in (0, 1):
            if done[s]:
                continue
            j = want[s]
            k = j % R
            ok = _try_wait(full[k], (j // R) & 1)
            if seq_gate:
                ok = ok and desc[k] is not None and desc[k][0] == j
            if ok:
                acts.append(("consume", s))
        if not acts:
            return "deadlock"
        what, arg = rng.choice(acts)
        if what == "issue":
            k = nxt % R
            desc[k] = (nxt, kinds[nxt])
            if kinds[nxt] == "data":
                in_flight.append(nxt)
            else:
                full[k] += 1
                landed.add(nxt)
            nxt += 1
        elif what == "land":
            in_flight.remove(arg)
            full[arg % R] += 1
            landed.add(arg)
        else:
            s = arg
            j = want[s]
            k = j % R
            if desc[k] is None or desc[k][0] != j or j not in landed:
                return "wrong stage"
            if desc[k][1] == "end":
                done[s] = True
            empty[k] += 1  # the set's eight warps, as one arrival
            want[s] += 2
    return "deadlock"


def _sweep(seq_gate: bool, slots, trials: int, seed: int) -> dict[str, int]:
    rng = random.Random(seed)
    out = {"ok": 0, "wrong stage": 0, "deadlock": 0}
    for R in slots:
        for _ in range(trials):
            T = rng.randint(2, 30)
            kinds = [rng.choice(("data", "data", "mark")) for _ in range(T)] + ["end", "end"]
            out[_run(R, kinds, seq_gate, rng)] += 1
    return out


def test_bare_parity_waits_race_with_odd_slot_counts():
    # the model is sharp enough to see the race the descriptor gate closes
    assert _sweep(False, (3, 5), 400, seed=1)["wrong stage"] > 0
    assert _sweep(False, (2, 4, 6), 400, seed=2)["wrong stage"] == 0


def test_descriptor_gate_orders_every_slot_count():
    r = _sweep(True, (2, 3, 4, 5, 6), 400, seed=3)
    assert r["wrong stage"] == 0 and r["deadlock"] == 0
