"""Host replay of the decode W8A8 kernel's barrier protocol (no GPU).

The kernel's producer thread fills an NS-deep ring of stages (four 2 KiB slabs and an activation
box each).  Eight consumer warps take slab w % 4 of the stages of parity w / 4 (M <= 16) or of every
stage (M > 16), release a stage with one arrival per warp, and flush their sums into one of two
segment buffers by segment parity.  With the run split, a combine warp finishes every segment but a
CTA's last (seg_full / seg_free handshakes); the last segment ends at a barrier of all consumers.

The programs below follow the kernel's stage walk and its slot, phase and segment arithmetic, and run
under random interleavings for the CTA runs the library's own plans produce.  Checks: every parity
wait checks its barrier with the phase it names, or the one before, completed last (never an older
phase the parity would pass on, never two phases on), no ring slot is refilled before the
stage's consumers read it, no consumer reads a slot before it landed, no segment buffer is reused
before the combine warp released it, no deadlock, and every stage consumed by every warp that owns
it.
"""
import random

import pytest

import int8_weight_gemm_gb300 as lib8
from schedule_util import Barrier, run_roles, wait

STAGE_SLABS = 4


def _segments(b0, b1, KB):
    """(tile, first slab, end slab) of each segment of the run [b0, b1), in the order the kernel
    walks them: with tiles of at least 128 k-blocks two segments swap when the first is the
    longer and three go first, last, middle; otherwise the natural order."""
    out, u = [], b0
    while u < b1:
        t = u // KB
        end = min(b1, (t + 1) * KB)
        out.append((t, u, end))
        u = end
    if KB >= 128 and len(out) == 2 and out[0][2] - out[0][1] > out[1][2] - out[1][1]:
        out = [out[1], out[0]]
    elif len(out) == 3 and KB >= 128:
        out = [out[0], out[2], out[1]]
    return out


def _run_cta(b0, b1, KB, NS, half_subtiles, multi, seed, fault=None):
    segs = _segments(b0, b1, KB)
    seg_stages = [-(-(e - s) // STAGE_SLABS) for (_, s, e) in segs]
    total = sum(seg_stages)
    stage_warps = 8 if half_subtiles else 4
    full = [Barrier(f"full{s}", 1) for s in range(NS)]
    empty = [Barrier(f"empty{s}", stage_warps) for s in range(NS)]
    seg_bar = Barrier("seg_bar", 8)
    seg_full = [Barrier(f"seg_full{b}", 8) for b in range(2)]
    seg_free = [Barrier(f"seg_free{b}", 1) for b in range(2)]
    consumed = [[] for _ in range(8)]
    buffer_owner = [None, None]   # which segment's sums a buffer holds until released

    def producer():
        pq = 0
        # the first min(NS, total) stages go out before the CTA barrier, with no wait
        while pq < min(NS, total):
            full[pq % NS].arrive()
            pq += 1
        yield
        while pq < total:
            s = pq % NS
            if fault != "producer skips its wait":
                yield from wait(empty[s], ((pq // NS) & 1) ^ 1, pq // NS - 1)
            assert empty[s].completed >= pq // NS, "ring slot refilled before its consumers read it"
            full[s].arrive()
            pq += 1
            yield

    def consumer(w):
        half = w // STAGE_SLABS
        q = 0
        for si, stages in enumerate(seg_stages):
            buf = si & 1
            if multi and si >= 2 and fault != "consumer skips the segment-buffer wait":
                yield from wait(seg_free[buf], ((si - 2) >> 1) & 1, (si - 2) >> 1)
                assert seg_free[buf].completed >= ((si - 2) >> 1) + 1, "segment buffer reused before release"
            if w == 0:
                assert buffer_owner[buf] is None, "segment buffer still holds an unfinished segment"
                buffer_owner[buf] = si
            start = 0 if half_subtiles else ((half - q) & 1)
            step = 1 if half_subtiles else 2
            for i in range(start, stages, step):
                qs = q + i
                s = qs % NS
                parity = (qs // NS) & 1
                yield from wait(full[s], parity ^ 1 if fault == "consumer waits on the wrong parity" else parity,
                                qs // NS)
                assert full[s].completed >= qs // NS + 1
                consumed[w].append(qs)
                empty[s].arrive()
                yield
            q += stages
            if multi and si != len(seg_stages) - 1:
                seg_full[buf].arrive()
                continue
            seg_bar.arrive()
            yield from wait(seg_bar, 0, 0)
            if w == 0:
                buffer_owner[buf] = None
            return

    def combine():
        for si in range(len(seg_stages) - 1):
            buf = si & 1
            if fault != "combine skips its wait":
                yield from wait(seg_full[buf], (si >> 1) & 1, si >> 1)
            assert buffer_owner[buf] == si, "segment buffer released before its consumers filled it"
            buffer_owner[buf] = None
            seg_free[buf].arrive()
            yield

    roles = [producer()] + [consumer(w) for w in range(8)] + ([combine()] if multi else [])
    run_roles(roles, seed)
    for w in range(8):
        half = w // STAGE_SLABS
        own = [qs for qs in range(total)] if half_subtiles else None
        if not half_subtiles:
            # a warp owns the stages of its parity, counted per segment from the segment's first stage
            own, q = [], 0
            for stages in seg_stages:
                own += [q + i for i in range((half - q) & 1, stages, 2)]
                q += stages
        assert consumed[w] == own


@pytest.mark.parametrize("M,K,N,blocks", [(16, 4096, 1536, 0), (16, 4096, 24576, 0), (32, 12288, 4096, 0),
                                          (8, 2048, 4096, 0), (16, 4096, 1536, 3), (32, 4096, 1536, 7),
                                          (1, 512, 256, 0), (24, 96, 136, 0), (16, 4096, 1536, 25)])
def test_decode_protocol_has_no_aliasing_and_no_deadlock(M, K, N, blocks):
    plan = lib8.w8a8_plan(M, K, N, blocks)
    assert plan["tensor_memory"] == 0
    G, KB, NS = plan["blocks"], plan["k_blocks"], plan["stages"]
    half_subtiles = plan["n8_tiles"] >= 3
    multi = plan["threads"] == 320
    bounds = lib8.w8a8_split_bounds(K, N, G)
    picks = sorted(set([0, G - 1, G // 2] + random.Random(M + K + N + G).sample(range(G), min(G, 5))))
    for i in picks:
        for seed in range(3):
            _run_cta(bounds[i], bounds[i + 1], KB, NS, half_subtiles, multi, seed=100 * i + seed)


FAULTS = ["producer skips its wait", "consumer skips the segment-buffer wait", "consumer waits on the wrong parity",
          "combine skips its wait"]


@pytest.mark.parametrize("fault", FAULTS)
@pytest.mark.parametrize("half_subtiles", [False, True])
def test_planted_protocol_fault_is_caught(fault, half_subtiles):
    # The replay's checks are tight enough: each fault, planted in the model, trips one of them on
    # some interleaving of runs with several segments.
    caught = 0
    for (b0, b1, KB) in [(0, 300, 128), (100, 140, 7), (0, 129, 64)]:
        for seed in range(6):
            try:
                _run_cta(b0, b1, KB, 8, half_subtiles, multi=True, seed=seed, fault=fault)
            except AssertionError:
                caught += 1
    assert caught > 0, f"not caught: {fault}"


@pytest.mark.parametrize("NS", [6, 8, 10])
@pytest.mark.parametrize("half_subtiles", [False, True])
def test_decode_protocol_on_long_runs_with_several_segments(NS, half_subtiles):
    for (b0, b1, KB) in [(0, 300, 128), (5, 263, 128), (100, 140, 7), (3, 4, 128), (0, 129, 64),
                         (30, 200, 128), (100, 200, 128), (10, 150, 64)]:
        for seed in range(3):
            _run_cta(b0, b1, KB, NS, half_subtiles, multi=True, seed=seed + b1)
