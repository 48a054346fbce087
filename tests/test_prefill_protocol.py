"""A discrete-event model of the prefill kernel's barrier protocol, checked on CPU.

prefill_kernel (softmax_attention_gb300/csrc/prefill.cu) runs seven warps that only meet
through mbarriers: a TMA producer, a landing watcher, one MMA-issuing thread and four softmax
warps.  A mistake there hangs or races on the GPU, where it cannot be tried safely, so this
module restates the protocol as agents over modelled barriers and runs it under random
latencies.  For every run it checks that

* every agent finishes (no deadlock);
* every parity wait is unambiguous whenever it polls: the barrier has completed exactly the
  awaited phase's predecessors or one more, never two phases past nor one short (either would
  make the hardware's parity test answer wrongly);
* no shared-memory stage or tensor-memory S/P buffer is read before its data is there, or
  overwritten while a reader still needs it.

The model follows the kernel's structure (one agent per role, the same barriers and phase
arithmetic); the mutation tests at the end plant known protocol mistakes and check that the
model reports them.
"""
import random

import pytest

from tests._protomodel import Hazard, Sim, TensorPipe, Bar


def run_protocol(n, stages, seed, *, paged_tail=False, mutate=None, fault=None):
    """Runs one CTA's KV loop of n tiles with `stages` K/V stages; raises Hazard on a fault.

    fault = (agent, tile) stops that agent at that tile, as if one of its waits had run out
    ("softmax1", "mma" or "watcher"); every wait is then bounded and the others take the
    kernel's error paths.  Returns the agents that recorded an error.
    """
    rng = random.Random(seed)
    sim = Sim(rng)
    pipe = TensorPipe(sim)
    limit = 50.0 if fault else 1e9   # latencies below are at most a few units
    watch_k = stages >= 3                                 # ready[j] also covers K_{j+2}
    watcher_k = watch_k and mutate != "watcher_skips_k"
    watcher_v = mutate != "watcher_skips_v"
    B = lambda name, c=1: Bar(name, c)
    bar_q, bar_qt, bar_done = B("q"), B("q_in_tmem", 128), B("mma_done")
    bar_k = [B(f"k_full{s}") for s in range(stages)]
    bar_v = [B(f"v_full{s}") for s in range(stages)]
    bar_ke = [B(f"k_empty{s}") for s in range(stages)]
    bar_ve = [B(f"v_empty{s}") for s in range(stages)]
    bar_s = [B("s_full0"), B("s_full1")]
    bar_r = [B(f"ready{s}", 128 + (0 if mutate == "ready_count_128" else 1)) for s in range(stages)]
    bar_o = B("o_full")

    kstage, vstage = [None] * stages, [None] * stages   # (tile, landed)
    sbuf = [[None] * 4 for _ in range(2)]               # per buffer, per warp quarter
    s_done, pv_done = set(), set()
    errors = set()
    last_landing = [0.0]
    lat = lambda lo, hi: rng.uniform(lo, hi)

    def check(cond, what):
        if not cond:
            raise Hazard(what)

    def wait(pred):
        return ("twait", pred, limit)

    def stops(agent, j):
        return fault is not None and fault == (agent, j)

    def tma(bar, store, s, j, reader_done):
        if j >= stages:
            check(j - stages in reader_done, f"load of tile {j} over a stage still in use")
        store[s] = (j, False)

        def land():
            store[s] = (j, True)
            bar.complete_tx(1)
        dt = lat(0.2, 3.0)
        last_landing[0] = max(last_landing[0], sim.t + dt)
        sim.at(dt, land)

    def producer():
        bar_q.arrive(expect=1)
        dt = lat(0.2, 2.0)
        last_landing[0] = max(last_landing[0], sim.t + dt)
        sim.at(dt, lambda: bar_q.complete_tx(1))
        issued, k_only = 0, -1
        for j in range(n):
            s = j % stages
            if j >= stages and not (yield wait(lambda s=s, j=j: bar_ke[s].passed(j // stages - 1))):
                errors.add("producer")
                break
            bar_k[s].arrive(expect=1)
            tma(bar_k[s], kstage, s, j, s_done)
            if j >= stages and not (yield wait(lambda s=s, j=j: bar_ve[s].passed(j // stages - 1))):
                errors.add("producer")
                k_only = j
                break
            bar_v[s].arrive(expect=1)
            tma(bar_v[s], vstage, s, j, pv_done)
            issued = j + 1
            yield ("delay", lat(0.0, 0.1))
        if issued < n:
            # A wait ran out: let the copies still in flight land before the CTA exits.  When
            # the producer stopped between a tile's K and V, that K (K_{k_only}) reused the
            # stage of K_{k_only - stages}, and it was issued only after S_{k_only - stages},
            # the reader of that older K, had finished: the older K has landed, and its
            # barrier may already be two phases on, so the drain does not wait for it.  Every
            # other drain wait is exact (the ambiguity check applies) and must not run out.
            drain = [(bar_q, 0)]
            for jj in range(max(0, issued - stages), issued):
                if not (k_only >= 0 and jj == k_only - stages and mutate != "drain_waits_stale_k"):
                    drain.append((bar_k[jj % stages], jj // stages))
                drain.append((bar_v[jj % stages], jj // stages))
            if k_only >= 0:
                drain.append((bar_k[k_only % stages], k_only // stages))
            for bar, phase in drain:
                if not (yield wait(lambda bar=bar, phase=phase: bar.passed(phase))):
                    errors.add("drain ran out")

    def watcher():
        if watcher_k and mutate != "watcher_skips_k01":
            # K_0 and K_1 share barriers with K_S and K_{S+1}, which the watcher waits for
            if not (yield wait(lambda: bar_k[0].passed(0))):
                errors.add("watcher")
                return
            if n > 1 and not (yield wait(lambda: bar_k[1].passed(0))):
                errors.add("watcher")
                return
        for j in range(n):
            s = j % stages
            if stops("watcher", j):
                errors.add("watcher")
                return
            if watcher_v and not (yield wait(lambda s=s, j=j: bar_v[s].passed(j // stages))):
                errors.add("watcher")
                return
            if watcher_k and j + 2 < n:
                s2 = (j + 2) % stages
                if not (yield wait(lambda s2=s2, j=j: bar_k[s2].passed((j + 2) // stages))):
                    errors.add("watcher")
                    return
            bar_r[s].arrive()

    def issue_s(j):
        b, s = j & 1, j % stages

        def start():
            check(kstage[s] == (j, True), f"S_{j} reads K stage {s} holding {kstage[s]}")
            if j >= 2:
                check(j - 2 in pv_done, f"S_{j} overwrites P_{j - 2} before P V read it")

        def end():
            s_done.add(j)
            for w in range(4):
                sbuf[b][w] = ("S", j)
        pipe.mma(lat(0.2, 0.6), start, end)
        pipe.commit(bar_s[b])
        pipe.commit(bar_ke[s])

    def issue_pv(j):
        b, s = j & 1, j % stages

        def start():
            check(all(q == ("P", j) for q in sbuf[b]), f"P_{j} V_{j} reads {sbuf[b]}")
            check(vstage[s] == (j, True), f"P_{j} V_{j} reads V stage {s} holding {vstage[s]}")

        pipe.mma(lat(0.2, 0.6), start, lambda: pv_done.add(j))
        pipe.commit(bar_o)
        pipe.commit(bar_ve[s])

    def mma():
        ok = yield wait(lambda: bar_qt.passed(0))
        ok = ok and (yield wait(lambda: bar_k[0].passed(0)))
        if ok:
            issue_s(0)
        if ok and n > 1:
            ok = yield wait(lambda: bar_k[1].passed(0))
            if ok:
                issue_s(1)
        for j in range(n):
            if not ok:
                break
            s = j % stages
            if stops("mma", j):
                ok = False
                break
            if mutate == "s_before_pv" and j + 2 < n:
                if not watch_k:
                    yield ("wait", lambda j=j: bar_k[(j + 2) % stages].passed((j + 2) // stages))
                yield ("wait", lambda s=s, j=j: bar_r[s].passed(j // stages))
                issue_s(j + 2)
                issue_pv(j)
                continue
            if not (ok := (yield wait(lambda s=s, j=j: bar_r[s].passed(j // stages)))):
                break
            issue_pv(j)
            if j + 2 < n:
                if not watch_k:
                    s2 = (j + 2) % stages
                    if not (ok := (yield wait(lambda s2=s2, j=j: bar_k[s2].passed((j + 2) // stages)))):
                        break
                issue_s(j + 2)
        if not ok:
            errors.add("mma")
        # every MMA issued must finish before tensor memory is released
        pipe.commit(bar_done)
        yield wait(lambda: bar_done.passed(0))

    def softmax(w):
        ok = yield wait(lambda: bar_q.passed(0))
        if ok:
            yield ("delay", lat(0.05, 0.2))
            for _ in range(32):
                bar_qt.arrive()
        for j in range(n):
            if not ok:
                break
            b, s = j & 1, j % stages
            if stops(f"softmax{w}", j):
                ok = False
                break
            if not (ok := (yield wait(lambda b=b, j=j: bar_s[b].passed(j >> 1)))):
                break
            check(sbuf[b][w] == ("S", j), f"softmax {w} reads S_{j} from {sbuf[b][w]}")
            yield ("delay", lat(0.3, 1.0))
            # The kernel waits every tile.  Skipping the wait on tiles with no rescale is unsafe
            # with a single barrier: the epilogue's wait for the last P V could then pass on
            # the phase before it (the skip_o_waits mutation).
            if j > 0 and not (mutate == "skip_o_waits" and rng.random() < 0.8):
                if not (ok := (yield wait(lambda j=j: bar_o.passed(j - 1)))):
                    break
                check(j - 1 in pv_done, f"softmax {w} rescales O before P_{j - 1} V_{j - 1}")
            sbuf[b][w] = ("P", j)
            if paged_tail and j == n - 1:
                if not (ok := (yield wait(lambda s=s, j=j: bar_v[s].passed(j // stages)))):
                    break
            for _ in range(32):
                bar_r[s].arrive()
        if ok and n > 0:
            ok = yield wait(lambda: bar_o.passed(n - 1))
            if ok:
                check(n - 1 in pv_done, "epilogue reads O before the last P V")
        if not ok:
            errors.add(f"softmax{w}")

    if n > 0:
        sim.start("producer", producer())
        sim.start("watcher", watcher())
        sim.start("mma", mma())
        for w in range(4):
            sim.start(f"softmax{w}", softmax(w))
    sim.run()
    expected = {"producer", "watcher", "mma"} | {f"softmax{w}" for w in range(4)} if n else set()
    check(sim.finished == expected, f"unfinished: {expected - sim.finished}")
    if n:
        exit_time = max(sim.finish_time.values())
        check(last_landing[0] <= exit_time, "a copy lands after every warp has finished")
        check(pipe.free_at <= exit_time, "an MMA runs after every warp has finished")
    return errors


@pytest.mark.parametrize("stages", [2, 3, 5])
@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 7, 10])
def test_protocol_is_safe(stages, n):
    for seed in range(40):
        run_protocol(n, stages, seed)
        run_protocol(n, stages, seed + 1000, paged_tail=True)


def _fails(n, stages, mutate):
    for seed in range(200):
        try:
            run_protocol(n, stages, seed, mutate=mutate)
        except Hazard:
            return True
    return False


def test_model_catches_missing_k_landing_wait():
    # ready[j] must cover K_{j+2} when the issuer does not wait for it itself
    assert _fails(8, 3, "watcher_skips_k")


def test_model_catches_s_issued_over_unread_p():
    # S_{j+2} shares P_j's buffer, so it has to follow P_j V_j in the tensor pipe
    assert _fails(8, 3, "s_before_pv")


def test_model_catches_watcher_not_observing_k0_k1():
    # without it, the wait for K_S can pass on K_0's phase when loads complete out of order
    assert _fails(8, 3, "watcher_skips_k01")


def test_model_catches_watcher_not_waiting_for_v():
    assert _fails(8, 3, "watcher_skips_v")


def test_model_catches_ready_count_without_the_watcher():
    # 128 + 1 arrivals per phase; with a count of 128 a phase can close before every P row
    assert _fails(8, 3, "ready_count_128")


def test_model_catches_skipped_o_waits_on_one_barrier():
    assert _fails(9, 3, "skip_o_waits")


@pytest.mark.parametrize("agent", ["softmax1", "mma", "watcher"])
@pytest.mark.parametrize("stages", [2, 3])
def test_error_paths_end_with_nothing_in_flight(agent, stages):
    # a warp stopping mid-loop (as after a wait that ran out): every other wait is bounded,
    # the producer lets its copies in flight land and the issuer's MMAs finish before exit
    for seed in range(30):
        n = 7
        errors = run_protocol(n, stages, seed, fault=(agent, seed % n))
        assert agent in errors and len(errors) > 1
        assert "drain ran out" not in errors


def test_model_catches_drain_waiting_for_a_reused_k_stage():
    # the drain's wait for the K whose stage the last K reused reads a barrier two phases on
    def fails():
        for seed in range(200):
            for agent in ("softmax1", "mma", "watcher"):
                try:
                    run_protocol(7, 3, seed, mutate="drain_waits_stale_k", fault=(agent, seed % 7))
                except Hazard:
                    return True
        return False
    assert fails()
