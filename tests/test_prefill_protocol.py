"""A discrete-event model of the prefill kernel's barrier protocol, checked on CPU.

prefill_kernel (softmax_attention_gb300/csrc/prefill.cu) runs seven warps that only meet
through mbarriers: a TMA producer, two MMA-issuing threads (one for S = Q K^T, one for
O += P V) and four softmax warps, with three S/P buffers in tensor memory.  A mistake there
hangs or races on the GPU, where it cannot be tried safely, so this module restates the
protocol as agents over modelled barriers and runs it under random latencies.  For every run
it checks that

* every agent finishes (no deadlock);
* every parity wait is unambiguous whenever it polls: the barrier has completed exactly the
  awaited phase's predecessors or one more, never two phases past nor one short (either would
  make the hardware's parity test answer wrongly);
* no shared-memory stage or tensor-memory S/P buffer is read before its data is there, or
  overwritten while a reader still needs it, and O is not rescaled under a running P V.

Each issuing thread's MMAs run in order on a pipe of their own, and the two pipes run
independently, so the model allows any interleaving of the two threads' MMAs (the hardware
orders them at least that strictly).  The model follows the kernel's structure (one agent
per role, the same barriers and phase arithmetic); the mutation tests at the end plant known
protocol mistakes and check that the model reports them.
"""
import random

import pytest

from tests._protomodel import Hazard, Sim, TensorPipe, Bar

NS = 3  # S/P buffers


def run_protocol(n, stages, seed, *, paged_tail=False, q_tmem=False, mutate=None, fault=None):
    """Runs one CTA's KV loop of n tiles with `stages` K/V stages; raises Hazard on a fault.

    q_tmem: Q is copied into tensor memory by the softmax warps and the S issuer waits for
    that copy.  fault = (agent, tile) stops that agent at that tile, as if one of its waits
    had run out ("softmax1", "pv" or "s"); every wait is then bounded and the others take the
    kernel's error paths.  Returns the agents that recorded an error.
    """
    rng = random.Random(seed)
    sim = Sim(rng)
    pipe_s, pipe_pv = TensorPipe(sim), TensorPipe(sim)
    limit = 50.0 if fault else 1e9   # latencies below are at most a few units
    B = lambda name, c=1: Bar(name, c)
    bar_q, bar_qt = B("q"), B("q_in_tmem", 128)
    bar_done, bar_sdone = B("pv_issuer_done"), B("s_issuer_done")
    bar_k = [B(f"k_full{s}") for s in range(stages)]
    bar_v = [B(f"v_full{s}") for s in range(stages)]
    bar_ke = [B(f"k_empty{s}") for s in range(stages)]
    bar_ve = [B(f"v_empty{s}") for s in range(stages)]
    bar_s = [B(f"s_full{b}") for b in range(NS)]
    bar_p = [B(f"p_full{b}", 96 if mutate == "p_count_96" else 128) for b in range(NS)]
    bar_pv = [B(f"pv_done{b}") for b in range(NS)]

    kstage, vstage = [None] * stages, [None] * stages   # (tile, landed)
    sbuf = [[None] * 4 for _ in range(NS)]              # per buffer, per warp quarter
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

    def s_issuer():
        q_bar = bar_qt if q_tmem else bar_q
        ok = yield wait(lambda: q_bar.passed(0))
        for j in range(n):
            if not ok:
                break
            b, s = j % NS, j % stages
            if stops("s", j):
                ok = False
                break
            if mutate != "s_skips_k":
                if not (ok := (yield wait(lambda s=s, j=j: bar_k[s].passed(j // stages)))):
                    break
            if j >= NS and mutate != "s_skips_buffer_wait":
                if not (ok := (yield wait(lambda b=b, j=j: bar_pv[b].passed((j - NS) // NS)))):
                    break

            def start(j=j, b=b, s=s):
                check(kstage[s] == (j, True), f"S_{j} reads K stage {s} holding {kstage[s]}")
                if j >= NS:
                    check(j - NS in pv_done, f"S_{j} overwrites P_{j - NS} before P V read it")

            def end(j=j, b=b):
                s_done.add(j)
                for w in range(4):
                    sbuf[b][w] = ("S", j)
            pipe_s.mma(lat(0.2, 0.6), start, end)
            pipe_s.commit(bar_s[b])
            pipe_s.commit(bar_ke[s])
        if not ok:
            errors.add("s")
        pipe_s.commit(bar_sdone)
        yield wait(lambda: bar_sdone.passed(0))

    def pv_issuer():
        ok = True
        for j in range(n):
            b, s = j % NS, j % stages
            if stops("pv", j):
                ok = False
                break
            if mutate != "pv_skips_p":
                if not (ok := (yield wait(lambda b=b, j=j: bar_p[b].passed(j // NS)))):
                    break
            if mutate != "pv_skips_v":
                if not (ok := (yield wait(lambda s=s, j=j: bar_v[s].passed(j // stages)))):
                    break

            def start(j=j, b=b, s=s):
                check(all(q == ("P", j) for q in sbuf[b]), f"P_{j} V_{j} reads {sbuf[b]}")
                check(vstage[s] == (j, True), f"P_{j} V_{j} reads V stage {s} holding {vstage[s]}")
                o_busy[0] = True

            def end(j=j):
                o_busy[0] = False
                pv_done.add(j)
            pipe_pv.mma(lat(0.2, 0.6), start, end)
            pipe_pv.commit(bar_pv[b])
            pipe_pv.commit(bar_ve[s])
        if not ok:
            errors.add("pv")
        # every MMA this thread issued must finish before tensor memory is released
        pipe_pv.commit(bar_done)
        yield wait(lambda: bar_done.passed(0))

    o_busy = [False]

    def softmax(w):
        ok = True
        if q_tmem:
            ok = yield wait(lambda: bar_q.passed(0))
            if ok:
                yield ("delay", lat(0.05, 0.2))
                for _ in range(32):
                    bar_qt.arrive()
        for j in range(n):
            if not ok:
                break
            b, s = j % NS, j % stages
            if stops(f"softmax{w}", j):
                ok = False
                break
            if not (ok := (yield wait(lambda b=b, j=j: bar_s[b].passed(j // NS)))):
                break
            check(sbuf[b][w] == ("S", j), f"softmax {w} reads S_{j} from {sbuf[b][w]}")
            yield ("delay", lat(0.3, 1.0))
            # A warp rescales O (some of its rows' max moved) only after waiting for
            # P_{j-1} V_{j-1}; other tiles do not wait (the rescale_without_wait mutation
            # skips the wait on rescale tiles too).
            rescale = rng.random() < 0.3
            if j > 0 and rescale:
                if mutate != "rescale_without_wait":
                    if not (ok := (yield wait(lambda j=j: bar_pv[(j - 1) % NS].passed((j - 1) // NS)))):
                        break
                check(j - 1 in pv_done and not o_busy[0],
                      f"softmax {w} rescales O before P_{j - 1} V_{j - 1} finished")
            sbuf[b][w] = ("P", j)
            if paged_tail and j == n - 1:
                # the V wait is exact once P_{j-1} V_{j-1} (hence V_{j-stages}) is done
                if j > 0 and not rescale and mutate != "tail_skips_pv_wait":
                    if not (ok := (yield wait(lambda j=j: bar_pv[(j - 1) % NS].passed((j - 1) // NS)))):
                        break
                if not (ok := (yield wait(lambda s=s, j=j: bar_v[s].passed(j // stages)))):
                    break
            for _ in range(32):
                bar_p[b].arrive()
        if ok and n > 0:
            ok = yield wait(lambda: bar_pv[(n - 1) % NS].passed((n - 1) // NS))
            if ok:
                check(n - 1 in pv_done, "epilogue reads O before the last P V")
        if not ok:
            errors.add(f"softmax{w}")

    if n > 0:
        sim.start("producer", producer())
        sim.start("s", s_issuer())
        sim.start("pv", pv_issuer())
        for w in range(4):
            sim.start(f"softmax{w}", softmax(w))
    sim.run()
    expected = {"producer", "s", "pv"} | {f"softmax{w}" for w in range(4)} if n else set()
    check(sim.finished == expected, f"unfinished: {expected - sim.finished}")
    if n:
        exit_time = max(sim.finish_time.values())
        check(last_landing[0] <= exit_time, "a copy lands after every warp has finished")
        check(max(pipe_s.free_at, pipe_pv.free_at) <= exit_time,
              "an MMA runs after every warp has finished")
    return errors


@pytest.mark.parametrize("stages", [2, 3, 5])
@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 7, 10])
def test_protocol_is_safe(stages, n):
    for seed in range(40):
        run_protocol(n, stages, seed, q_tmem=(seed % 2 == 1))
        run_protocol(n, stages, seed + 1000, paged_tail=True)


def _fails(n, stages, mutate, **kw):
    for seed in range(200):
        try:
            run_protocol(n, stages, seed, mutate=mutate, **kw)
        except Hazard:
            return True
    return False


def test_model_catches_s_over_an_unread_p():
    # S_j goes into P_{j-3}'s buffer; without waiting for P_{j-3} V_{j-3} it can overwrite it
    assert _fails(8, 3, "s_skips_buffer_wait")


def test_model_catches_s_before_its_k_lands():
    assert _fails(8, 3, "s_skips_k")


def test_model_catches_pv_before_p():
    assert _fails(8, 3, "pv_skips_p")


def test_model_catches_pv_before_its_v_lands():
    assert _fails(8, 3, "pv_skips_v")


def test_model_catches_p_count_short_of_the_rows():
    # 128 arrivals (4 warps x 32 rows) per phase; with fewer a phase closes before every row
    assert _fails(8, 3, "p_count_96")


def test_model_catches_a_paged_tail_v_wait_without_the_pv_wait():
    # without P_{j-1} V_{j-1} done, V_{j-stages} may not have landed and the parity wait for
    # V_j can pass on its phase
    assert _fails(5, 2, "tail_skips_pv_wait", paged_tail=True)


def test_model_catches_a_rescale_without_the_o_wait():
    assert _fails(9, 3, "rescale_without_wait")


@pytest.mark.parametrize("agent", ["softmax1", "pv", "s"])
@pytest.mark.parametrize("stages", [2, 3])
def test_error_paths_end_with_nothing_in_flight(agent, stages):
    # a warp stopping mid-loop (as after a wait that ran out): every other wait is bounded,
    # the producer lets its copies in flight land and the issuers' MMAs finish before exit
    for seed in range(30):
        n = 7
        errors = run_protocol(n, stages, seed, fault=(agent, seed % n))
        assert agent in errors and len(errors) > 1
        assert "drain ran out" not in errors


def test_model_catches_drain_waiting_for_a_reused_k_stage():
    # the drain's wait for the K whose stage the last K reused reads a barrier two phases on
    def fails():
        for seed in range(200):
            for agent in ("softmax1", "pv", "s"):
                try:
                    run_protocol(7, 3, seed, mutate="drain_waits_stale_k", fault=(agent, seed % 7))
                except Hazard:
                    return True
        return False
    assert fails()
