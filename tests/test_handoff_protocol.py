"""Model check of the named-barrier handoff in the tile/block-scaled GEMM
(csrc/fp8q_gemm_block.cu): the MMA warp, the relay warp and the eight
promotion warps each walk the same T K blocks, arriving on and waiting at
hardware barriers that cannot time out, so the sequence itself must be proven
balanced.

Barrier semantics modelled (PTX bar.arrive / bar.sync with a thread count):
each warp-wide operation adds 32 threads to the barrier's current generation;
bar.sync blocks until the generation reaches its count, which completes it
and starts the next.  The checks, over random schedules (with one
participant slowed down) and with an abort at a random K block (the MMA warp
then issues nothing and the relay's bounded wait returns at once):
- every generation is completed by operations of one K block only;
- every schedule finishes, with no generation left incomplete.
The same checker must flag three broken variants of the protocol."""
import random

import pytest

COUNT = {"FULL": 32 * 9, "RELM": 32 * 9, "ISS": 64}
PROMOTION_WARPS = 8


def seq_mma(T):
    s = []
    for it in range(T):
        if it >= 2:
            s.append(("sync", "RELM", it % 2, it - 2))
        s.append(("issue", it))
        s.append(("arrive", "ISS", it % 2, it))
    for k in range(max(0, T - 2), T):
        s.append(("sync", "RELM", k % 2, k))
    return s


def seq_relay(T):
    s = []
    for it in range(T):
        s.append(("sync", "ISS", it % 2, it))
        s.append(("pf", it))
        s.append(("arrive", "FULL", it % 2, it))
    return s


def seq_promotion(T):
    s = []
    for it in range(T):
        s.append(("sync", "FULL", it % 2, it))
        s.append(("arrive", "RELM", it % 2, it))
    return s


def simulate(seqs, rng, abort_at, slow):
    pc = {w: 0 for w in seqs}
    blocked, gen = {}, {}
    issued, done = set(), set()
    aborted = False
    for _ in range(200000):
        runnable = []
        for w, s in seqs.items():
            if pc[w] >= len(s) or w in blocked:
                continue
            op = s[pc[w]]
            if op[0] == "pf" and not aborted and op[1] not in done:
                continue                      # waits for that K block's MMAs
            runnable.append(w)
        pending = sorted(i for i in issued if i not in done)
        if not runnable and not pending:
            if all(pc[w] >= len(s) for w, s in seqs.items()) and not blocked:
                return "ok" if not gen else f"incomplete generations {sorted(gen)}"
            return "deadlock"
        if pending and (not runnable or rng.random() < 0.3):
            done.add(pending[0])              # MMAs complete in issue order
            continue
        fast = [x for x in runnable if x != slow]
        w = rng.choice(fast if fast and rng.random() < 0.97 else runnable)
        op = seqs[w][pc[w]]
        if op[0] in ("issue", "pf"):
            if op[0] == "issue":
                if abort_at is not None and op[1] >= abort_at:
                    aborted = True
                else:
                    issued.add(op[1])
            pc[w] += 1
            continue
        kind, bar, parity, tag = op
        g = gen.setdefault((bar, parity), [0, set(), []])
        g[0] += 32
        g[1].add(tag)
        if kind == "sync":
            g[2].append(w)
            blocked[w] = (bar, parity)
        else:
            pc[w] += 1
        if g[0] == COUNT[bar]:
            if len(g[1]) != 1:
                return f"generation of {bar}[{parity}] mixes K blocks {sorted(g[1])}"
            for x in g[2]:
                del blocked[x]
                pc[x] += 1
            del gen[(bar, parity)]
    return "no progress"


def check(make_mma, make_relay, make_prom, seed, trials=150, max_t=9):
    rng = random.Random(seed)
    failures = []
    for T in range(max_t + 1):
        for t in range(trials):
            abort_at = None if t % 3 else rng.randrange(0, T + 1)
            slow = rng.choice([None, "mma", "relay", "p0", "p5"])
            seqs = {"mma": make_mma(T), "relay": make_relay(T)}
            for w in range(PROMOTION_WARPS):
                seqs[f"p{w}"] = make_prom(T)
            r = simulate(seqs, rng, abort_at, slow)
            if r != "ok":
                failures.append((T, abort_at, slow, r))
    return failures


def test_protocol_is_balanced_and_never_mixes_generations():
    assert check(seq_mma, seq_relay, seq_promotion, seed=1) == []


@pytest.mark.parametrize("broken", ["no_issue_barrier", "one_parity", "no_final_syncs"])
def test_checker_catches_broken_protocols(broken):
    mma, relay, prom = seq_mma, seq_relay, seq_promotion
    if broken == "no_issue_barrier":
        # the relay no longer waits for the MMA warp: after an abort it runs ahead
        def relay(T):
            return [op for op in seq_relay(T) if op[1] != "ISS"]

        def mma(T):
            return [op for op in seq_mma(T) if op[1] != "ISS"]
    elif broken == "one_parity":
        def relay(T):
            return [(o[0], o[1], 0, o[3]) if o[1] == "FULL" else o for o in seq_relay(T)]

        def prom(T):
            return [(o[0], o[1], 0, o[3]) if o[1] == "FULL" else o for o in seq_promotion(T)]
    else:
        def mma(T):
            s = seq_mma(T)
            return s[:-1] if T else s
    assert check(mma, relay, prom, seed=2, trials=100) != []
