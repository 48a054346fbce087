"""A discrete-event model of the MLA decode kernel's barrier protocol, checked on CPU.

mla_kernel (softmax_attention_gb300/csrc/mla.cu) streams a sequence's 32-token stages through
a four-slot shared-memory ring (two 64-token tiles).  Four producer warps gather their eight
tokens of each stage with per-thread cp.async groups and publish a stage (32 arrivals per
warp on its full barrier) once their own copies have landed; for a whole tile inside one
large page, one producer thread instead waits for both of the tile's slots, adds the tile's
bytes to the first stage's full barrier and issues two TMA boxes that fill both stages.  The
MMA thread polls: S_j once both stages of tile j are full and S buffer j & 1 is free (P_{j-2}
V has been issued), P_j V_j once P_j is written; P_j V_j's commits release the tile's two
slots.  The softmax warps read S_j, wait for P_{j-1} V_{j-1} (O^T rescale, and the single
shared-memory P buffer), write P_j and arrive.

The model restates those roles over modelled barriers (tests/_protomodel.py) and checks, under
random latencies and random mixes of gathered and TMA tiles, that every agent finishes, that
every parity wait or poll is exact, and that no ring slot, S buffer or P buffer is read
before it is written or overwritten while still needed.  The mutation tests plant protocol
mistakes and check that the model reports them.
"""
import random

import pytest

from tests._protomodel import Bar, Hazard, Sim, TensorPipe

SLOTS = 4  # two 64-token tiles of two 32-token stages


def run_mla(n_tiles, seed, *, tma_prob=0.0, mutate=None):
    rng = random.Random(seed)
    sim = Sim(rng)
    pipe = TensorPipe(sim)
    lat = lambda lo, hi: rng.uniform(lo, hi)
    n_stages = 2 * n_tiles
    partial_last = rng.random() < 0.5
    by_tma = [rng.random() < tma_prob and not (partial_last and j == n_tiles - 1)
              for j in range(n_tiles)]

    bar_q = Bar("q", 1)
    bar_full = [Bar(f"full{s}", 128) for s in range(SLOTS)]
    bar_empty = [Bar(f"empty{s}", 1) for s in range(SLOTS)]
    bar_s = [Bar("s_full0", 1), Bar("s_full1", 1)]
    bar_p = Bar("p_full", 128)
    bar_o = Bar("o_full", 1)

    slot_stage = [None] * SLOTS        # stage whose data a slot holds (or is receiving)
    landed = [set() for _ in range(SLOTS)]
    sbuf = [None, None]                # ("S", j) written, ("read", j) read by the softmax
    p_buf = None                       # ("P", j)
    pv_done = set()
    in_flight = [0]

    def check(cond, what):
        if not cond:
            raise Hazard(what)

    def parts(n):
        return {"ckv", "kpe"} if by_tma[n // 2] else {0, 1, 2, 3}

    def stage_ready(n):
        s = n % SLOTS
        return slot_stage[s] == n and parts(n) <= landed[s]

    def claim(n):
        """A write into stage n's slot starts: the tile that held it must be done."""
        s = n % SLOTS
        if slot_stage[s] != n:
            if n >= SLOTS:
                check((n - SLOTS) // 2 in pv_done, f"stage {n} written over a slot still in use")
            slot_stage[s], landed[s] = n, set()

    def land_later(n, part, on_land=None):
        in_flight[0] += 1

        def land():
            s = n % SLOTS
            check(slot_stage[s] == n, f"stage {n} data landed in a slot now holding {slot_stage[s]}")
            landed[s].add(part)
            in_flight[0] -= 1
            if on_land:
                on_land()
        sim.at(lat(0.2, 3.0), land)

    def producer(pw):
        if pw == 0:
            bar_q.arrive(expect=1)
            sim.at(lat(0.2, 2.0), lambda: bar_q.complete_tx(1))
        issued = published = 0
        group_landed = []
        while published < n_stages:
            can_issue = issued < n_stages and (
                issued < SLOTS or bar_empty[issued % SLOTS].passed(issued // SLOTS - 1))
            if can_issue:
                n, j = issued, issued // 2
                flag = [True]  # a TMA stage leaves this thread an empty cp.async group
                if by_tma[j]:
                    if n % 2 == 0 and pw == 0:
                        if n + 1 >= SLOTS:
                            yield ("wait", lambda n=n: bar_empty[(n + 1) % SLOTS].passed(
                                (n + 1) // SLOTS - 1))
                        claim(n)
                        claim(n + 1)
                        full = bar_full[n % SLOTS]
                        if mutate != "tma_no_expect":
                            full.expect(2)
                        for box in ("ckv", "kpe"):
                            def both(box=box, n=n, full=full):
                                landed[(n + 1) % SLOTS].add(box)
                                if mutate != "tma_no_expect":
                                    full.complete_tx(1)
                            land_later(n, box, both)
                else:
                    claim(n)
                    flag = [False]
                    land_later(n, pw, lambda f=flag: f.__setitem__(0, True))
                group_landed.append(flag)
                issued += 1
                yield ("delay", lat(0.0, 0.05))
            elif published < issued:
                f = group_landed[published]
                if mutate != "publish_early":
                    yield ("wait", lambda f=f: f[0])
                for _ in range(32):
                    bar_full[published % SLOTS].arrive()
                published += 1
            else:
                yield ("wait", lambda i=issued: bar_empty[i % SLOTS].passed(i // SLOTS - 1))

    def issue_s(j):
        def start():
            for n in (2 * j, 2 * j + 1):
                check(stage_ready(n), f"S_{j} reads stage {n} before it is complete")
            check(sbuf[j & 1] in (None, ("read", j - 2)), f"S_{j} overwrites {sbuf[j & 1]}")

        def end():
            sbuf[j & 1] = ("S", j)
        pipe.mma(lat(0.3, 0.8), start, end)
        pipe.commit(bar_s[j & 1])

    def issue_pv(j):
        def start():
            check(p_buf == ("P", j), f"P_{j} V_{j} reads the P buffer holding {p_buf}")
            for n in (2 * j, 2 * j + 1):
                check(stage_ready(n), f"P_{j} V_{j} reads stage {n} before it is complete")

        pipe.mma(lat(0.2, 0.4), start, lambda: pv_done.add(j))
        pipe.commit(bar_o)
        pipe.commit(bar_empty[(2 * j) % SLOTS])
        pipe.commit(bar_empty[(2 * j + 1) % SLOTS])

    def mma():
        yield ("wait", lambda: bar_q.passed(0))
        st = {"s": 0, "pv": 0}

        def can_s():
            j = st["s"]
            gate = mutate == "no_s_gate" or j <= st["pv"] + 1
            return (j < n_tiles and gate and bar_full[(2 * j) % SLOTS].passed((2 * j) // SLOTS)
                    and bar_full[(2 * j + 1) % SLOTS].passed((2 * j + 1) // SLOTS))

        def can_pv():
            return st["pv"] < st["s"] and bar_p.passed(st["pv"])

        while st["pv"] < n_tiles:
            yield ("wait", lambda: can_s() or can_pv())
            if can_s():
                issue_s(st["s"])
                st["s"] += 1
            if can_pv():
                issue_pv(st["pv"])
                st["pv"] += 1

    def softmax():
        nonlocal p_buf
        for j in range(n_tiles):
            yield ("wait", lambda j=j: bar_s[j & 1].passed(j >> 1))
            check(sbuf[j & 1] == ("S", j), f"softmax reads S_{j} from {sbuf[j & 1]}")
            sbuf[j & 1] = ("read", j)
            yield ("delay", lat(0.3, 1.0))
            if j > 0 and mutate != "softmax_skips_o":
                yield ("wait", lambda j=j: bar_o.passed(j - 1))
            if j > 0:
                check(j - 1 in pv_done, f"P_{j} written while P_{j - 1} V_{j - 1} may read P")
            p_buf = ("P", j)
            for _ in range(128):
                bar_p.arrive()
        if n_tiles:
            yield ("wait", lambda: bar_o.passed(n_tiles - 1))
            check(len(pv_done) == n_tiles, "epilogue before every P V finished")
            check(in_flight[0] == 0, "epilogue reuses the ring while a copy is in flight")

    if n_tiles:
        for pw in range(4):
            sim.start(f"producer{pw}", producer(pw))
        sim.start("mma", mma())
        sim.start("softmax", softmax())
    sim.run()
    expected = ({f"producer{pw}" for pw in range(4)} | {"mma", "softmax"}) if n_tiles else set()
    check(sim.finished == expected, f"unfinished: {expected - sim.finished}")


@pytest.mark.parametrize("tma_prob", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("n_tiles", [0, 1, 2, 3, 4, 5, 8])
def test_mla_protocol_is_safe(n_tiles, tma_prob):
    for seed in range(40):
        run_mla(n_tiles, seed, tma_prob=tma_prob)


def _fails(mutate, tma_prob=0.0, n_tiles=6):
    for seed in range(200):
        try:
            run_mla(n_tiles, seed, tma_prob=tma_prob, mutate=mutate)
        except Hazard:
            return True
    return False


def test_s_buffer_gate_is_implied_by_the_ring():
    # S_j needs tile j's two ring slots, which only P_{j-2} V_{j-2} releases, and that needs
    # P_{j-2}, written after the softmax read S_{j-2}: the issuer's explicit gate is redundant
    for seed in range(100):
        run_mla(6, seed, tma_prob=0.5, mutate="no_s_gate")


def test_model_catches_p_written_under_a_running_pv():
    assert _fails("softmax_skips_o")


def test_model_catches_a_stage_published_before_its_copies_land():
    assert _fails("publish_early")


def test_model_catches_tma_bytes_missing_from_the_full_barrier():
    assert _fails("tma_no_expect", tma_prob=1.0)
