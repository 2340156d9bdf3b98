"""Host replay of the tensor-memory W8A8 arm's pipeline protocol (no GPU).

The kernel's roles meet on mbarriers with parity waits: a wait names the phase it needs by its
parity only, so it is correct only if, whenever a thread checks, the barrier has completed either
exactly the phase it needs or one fewer; two phases further it would mistake an old phase for its
own.  This test runs the roles' programs, with the slot, phase and period arithmetic written the
way the kernel computes it, under random interleavings and random MMA completion delays, for the
CTA runs the library's own split plans produce, and checks that

  * every wait checks its barrier with the phase it names, or the one before, completed last (the
    parity of an older phase would pass early; two phases on it would block on a phase long gone),
  * no slot is overwritten or read before the role that owns it has finished with it (the weight,
    activation and tensor-memory A rings, the accumulator buffers and their read-out),
  * every role finishes (no deadlock), and
  * every stage is converted, multiplied and retired once, every period's accumulator read once.

Roles (one CTA): the weight producer, the activation producer, sixteen converter warps in four
groups as in the kernel (group g converts the stages q with q % 4 == g into A slot g; every warp
reads out every accumulation period; each arrives once per warp), I issuing threads, and an MMA
engine that completes each issuer's commits in order.  Ring depths are the kernel's (weight 8 /
activations 3 at N = 128, 10 / 4 with two issuers at N = 64; four A slots, two accumulator
buffers).
"""
import random

import pytest

import int8_weight_gemm_gb300 as lib8
from schedule_util import Barrier, run_roles, wait

STAGE_UNITS = 4
PERIOD_STAGES = 4


class Walk:
    """The kernel's schedule walker (segments of one tile, stages of <= 4 units, periods of <= 4
    stages)."""

    def __init__(self, b0, b1, KB):
        self.u, self.b1, self.KB = b0, b1, KB
        self.q = self.sp = self.period = 0
        self._begin_segment()

    def _begin_segment(self):
        self.t = self.u // self.KB
        self.seg_begin = self.u
        self.seg_end = min(self.b1, (self.t + 1) * self.KB)
        self.ns = min(STAGE_UNITS, self.seg_end - self.u)

    def done(self):
        return self.u >= self.b1

    def seg_first(self):
        return self.u == self.seg_begin

    def seg_last(self):
        return self.u + self.ns >= self.seg_end

    def period_first(self):
        return self.sp == 0

    def period_last(self):
        return self.seg_last() or self.sp == PERIOD_STAGES - 1

    def whole_tile(self):
        return self.seg_begin == self.t * self.KB and self.seg_end == (self.t + 1) * self.KB

    def next(self):
        pl, sl = self.period_last(), self.seg_last()
        self.u += self.ns
        self.q += 1
        if pl:
            self.sp = 0
            self.period += 1
        else:
            self.sp += 1
        if self.u >= self.b1:
            return
        if sl:
            self._begin_segment()
        else:
            self.ns = min(STAGE_UNITS, self.seg_end - self.u)


def _run_cta(b0, b1, KB, n_mma, seed, fault=None):
    rng = random.Random(seed)
    NW, NB, kI = (10, 4, 2) if n_mma == 64 else (8, 3, 1)
    NA = GROUPS = 4   # A slots, one per converter group
    C = 16  # converter warps, as many as the kernel runs (one arrival per warp)
    GW = C // GROUPS
    wfull = [Barrier(f"wfull{s}", 1) for s in range(NW)]
    wempty = [Barrier(f"wempty{s}", GW) for s in range(NW)]
    bfull = [Barrier(f"bfull{s}", 1) for s in range(NB)]
    bdone = [Barrier(f"bdone{s}", kI) for s in range(NB)]
    adone = [Barrier(f"adone{a}", kI) for a in range(NA)]
    conv = [Barrier(f"conv{a}", GW) for a in range(NA)]
    dfull = [Barrier(f"dfull{d}", kI) for d in range(2)]
    dempty = [Barrier(f"dempty{d}", C) for d in range(2)]
    sync = Barrier("sync", C)
    pending_commits = [[] for _ in range(kI)]   # per issuer, in issue order: barriers to arrive on
    log = {"converted": [], "issued": [[] for _ in range(kI)], "retired": [[] for _ in range(C)],
           "drained": [[] for _ in range(C)]}

    def w_producer():
        it, q = Walk(b0, b1, KB), 0
        while not it.done():
            s = q % NW
            if q >= NW and fault != "weight producer skips its wait":
                yield from wait(wempty[s], ((q // NW) & 1) ^ 1, q // NW - 1)
            # overwriting slot s: the group that converts stage q - NW has read it
            assert q < NW or wempty[s].completed >= q // NW, "weight slot overwritten before it was read"
            wfull[s].arrive()   # expect_tx + copies; the bytes land eventually
            it.next()
            q += 1
            yield

    def b_producer():
        it, q = Walk(b0, b1, KB), 0
        while not it.done():
            s = q % NB
            if q >= NB and fault != "activation producer skips its wait":
                yield from wait(bdone[s], ((q - NB) // NB) & 1, (q - NB) // NB)
            assert q < NB or bdone[s].completed >= (q - NB) // NB + 1, "activation slot overwritten under the MMAs"
            bfull[s].arrive()
            it.next()
            q += 1
            yield

    def issuer(i):
        it = Walk(b0, b1, KB)
        while not it.done():
            sb, a, db = it.q % NB, it.q % NA, it.period & 1
            if it.period_first() and it.period >= 2 and fault != "issuer skips the read-out wait":
                yield from wait(dempty[db], ((it.period >> 1) - 1) & 1, (it.period >> 1) - 1)
            parity = (it.q // NA) & 1
            yield from wait(conv[a], parity ^ 1 if fault == "issuer waits on the wrong parity" else parity, it.q // NA)
            if fault != "issuer skips the activation wait":
                yield from wait(bfull[sb], (it.q // NB) & 1, it.q // NB)
            # the MMAs read A slot a and activation slot sb of this stage, and write buffer db
            assert conv[a].completed >= it.q // NA + 1, "A slot read before its group wrote it"
            assert bfull[sb].completed >= it.q // NB + 1, "activation slot read before it landed"
            assert it.period < 2 or not it.period_first() or dempty[db].completed >= it.period >> 1, \
                "accumulator buffer overwritten before its read-out"
            steps = [j for j in range(i, 2 * it.ns, kI)]
            assert steps, "every issuer has a k-step in every stage"
            log["issued"][i].append(it.q)
            pending_commits[i].append(bdone[sb])
            pending_commits[i].append(adone[a])
            if it.period_last():
                pending_commits[i].append(dfull[db])
            it.next()
            yield

    def mma_engine():
        while any(pending_commits) or not all(done_issuers):
            live = [i for i in range(kI) if pending_commits[i]]
            if live and rng.random() < 0.5:
                i = rng.choice(live)
                pending_commits[i].pop(0).arrive()   # in order per issuer
            yield

    def converter(w):
        sync_phase = 0
        group = w // GW
        dr = Walk(b0, b1, KB)

        def retire():
            nonlocal sync_phase
            log["retired"][w].append(dr.q)
            if dr.period_last():
                # reading the period's accumulators once its MMAs have completed
                if fault != "converter skips the read-out wait":
                    yield from wait(dfull[dr.period & 1], (dr.period >> 1) & 1, dr.period >> 1)
                assert dfull[dr.period & 1].completed >= (dr.period >> 1) + 1, "accumulators read before their MMAs completed"
                log["drained"][w].append(dr.period)
                dempty[dr.period & 1].arrive()
                if dr.seg_last() and not dr.whole_tile():
                    sync.arrive()
                    yield from wait(sync, sync_phase & 1, sync_phase)
                    sync_phase += 1
                    sync.arrive()
                    yield from wait(sync, sync_phase & 1, sync_phase)
                    sync_phase += 1
            dr.next()

        it = Walk(b0, b1, KB)
        while not it.done():
            # stage q - 4 retires as the walk passes stage q
            if it.q >= GROUPS:
                yield from retire()
            if it.q % GROUPS == group:
                s, a = it.q % NW, group
                yield from wait(wfull[s], (it.q // NW) & 1, it.q // NW)
                if it.q >= GROUPS and fault != "converter skips the MMA wait":
                    yield from wait(adone[a], ((it.q - GROUPS) // NA) & 1, (it.q - GROUPS) // NA)
                # writing A slot a: the MMAs of stage q - 4, which read it, have completed
                assert it.q < NA or adone[a].completed >= (it.q - NA) // NA + 1, "A slot overwritten under the MMAs"
                assert wfull[s].completed >= it.q // NW + 1
                if w == group * GW:
                    log["converted"].append(it.q)
                wempty[s].arrive()
                conv[a].arrive()
            it.next()
            yield
        while not dr.done():
            yield from retire()

    done_issuers = [False] * kI

    def issuer_wrapped(i):
        yield from issuer(i)
        done_issuers[i] = True

    roles = [w_producer(), b_producer(), mma_engine()] + [issuer_wrapped(i) for i in range(kI)] + \
            [converter(w) for w in range(C)]
    run_roles(roles, seed + 1)
    walk = Walk(b0, b1, KB)
    stages = periods = 0
    while not walk.done():
        if walk.period_last():
            periods += 1
        walk.next()
        stages += 1
    assert sorted(log["converted"]) == list(range(stages))
    for i in range(kI):
        assert log["issued"][i] == list(range(stages))
    for w in range(C):
        assert log["retired"][w] == list(range(stages))
        assert log["drained"][w] == list(range(periods))
    return stages


@pytest.mark.parametrize("M,K,N,blocks", [(128, 4096, 1536, 0), (128, 4096, 24576, 0), (64, 12288, 4096, 0),
                                          (100, 2048, 384, 7), (33, 4000, 320, 0), (128, 512, 1024, 3),
                                          (64, 96, 136, 0), (128, 4096, 1536, 1)])
def test_protocol_has_no_aliasing_and_no_deadlock(M, K, N, blocks):
    plan = lib8.w8a8_plan(M, K, N, blocks, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)
    assert plan["tensor_memory"] == 1
    G, KB = plan["blocks"], plan["k_blocks"]
    bounds = lib8.w8a8_split_bounds(K, N, G, M=M)
    n_mma = plan["n8_tiles"] * 8
    picks = sorted(set([0, G - 1, G // 2] + random.Random(M + K + N).sample(range(G), min(G, 5))))
    for i in picks:
        for seed in range(3):
            _run_cta(bounds[i], bounds[i + 1], KB, n_mma, seed=1000 * i + seed)


FAULTS = ["weight producer skips its wait", "activation producer skips its wait", "issuer skips the read-out wait",
          "issuer waits on the wrong parity", "issuer skips the activation wait", "converter skips the MMA wait",
          "converter skips the read-out wait"]


@pytest.mark.parametrize("fault", FAULTS)
@pytest.mark.parametrize("n_mma", [64, 128])
def test_planted_protocol_fault_is_caught(fault, n_mma):
    # The replay's checks are tight enough: each fault, planted in the model, trips one of them on
    # some interleaving.  Runs: long tiles (periods of four stages), and tiles of one stage each
    # (K = 96), where a period is one stage and only the read-out wait keeps the issuer off an
    # accumulator buffer still being read (with four-stage periods the A-ring wait implies it).
    caught = 0
    for (b0, b1, KB) in [(0, 300, 128), (0, 60, 3), (1, 40, 3)]:
        for seed in range(6):
            try:
                _run_cta(b0, b1, KB, n_mma, seed=seed, fault=fault)
            except AssertionError:
                caught += 1
    assert caught > 0, f"not caught: {fault}"


@pytest.mark.parametrize("n_mma", [64, 128])
def test_protocol_on_long_and_short_runs(n_mma):
    # Runs that span several tiles, start mid-tile, or hold a single unit.
    for (b0, b1, KB) in [(0, 1, 1), (3, 4, 128), (0, 37, 8), (5, 300, 128), (100, 140, 7), (0, 512, 128)]:
        for seed in range(4):
            _run_cta(b0, b1, KB, n_mma, seed=seed + b1)
