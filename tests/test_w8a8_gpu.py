"""W8A8 decode GEMM on the GPU against the oracle: bit-exact bf16 outputs and int32 accumulators
(through w8a8_gemm_acc) on every case.

Cases: the five workload families (seeded, full size, compared element by element), ragged
shapes (M not a multiple of 8, N not a multiple of 64), every split count class (one CTA, a few,
one CTA per slab, automatic), adversarial inputs whose large int32 partial sums cancel to small
results (an inexact accumulation would show in the bf16 output), the pack against the oracle's
layout, CUDA-graph replays, and the workspace contract (counters back at zero, status clean).
"""
import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import W8A8Case, bf16_bits

pytestmark = pytest.mark.gpu


def _check(case, x, xs, W, ws, blocks=None):
    """bf16 outputs of w8a8_gemm, and both the outputs and the int32 accumulators of
    w8a8_gemm_acc, bit for bit against the oracle."""
    ref = oracle.w8a8_gemm(x, xs, W, ws)
    out = case.run(blocks=blocks)
    torch.cuda.synchronize()
    got = bf16_bits(out)
    mism = np.count_nonzero(got != ref)
    assert mism == 0, f"{mism} of {ref.size} outputs differ"
    assert case.status() == 0
    out2, acc = case.run_acc(blocks=blocks)
    torch.cuda.synchronize()
    ref_acc = oracle.w8a8_acc(x, W)
    acc_mism = np.count_nonzero(acc.cpu().numpy().astype(np.int64) != ref_acc)
    assert acc_mism == 0, f"{acc_mism} of {ref_acc.size} int32 accumulators differ"
    assert np.array_equal(bf16_bits(out2), ref)
    assert case.status() == 0


def test_small_config_seed0():
    # M=1, K=512, N=256; int8 uniform [-127,127]; scales uniform [1e-3, 2e-2]; seed 0; one call.
    x, xs, W, ws = synth.w8a8_inputs(1, 512, 256, seed=0)
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


def test_pack_matches_oracle_layout():
    for K, N in [(512, 256), (64, 200), (4096, 1536)]:
        W = synth.uniform_int8(7, "pack.W", (K, N), lo=-128, hi=127)
        Wd = torch.from_numpy(W).cuda()
        got = lib8.w8a8_pack_weights(Wd).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.w8a8_pack(W))


@pytest.mark.parametrize("M", [1, 2, 3, 5, 7, 8, 9, 13, 16, 17, 24, 25, 31, 32])
def test_ragged_m(M):
    x, xs, W, ws = synth.w8a8_inputs(M, 1024, 200, seed=M)
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("K,N", [(32, 8), (32, 64), (64, 72), (96, 136), (2048, 520), (416, 4096)])
def test_ragged_shapes(K, N):
    x, xs, W, ws = synth.w8a8_inputs(11, K, N, seed=K + N)
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("blocks", [1, 2, 3, 7, 64, 151, 152, 304, 0, -1])
def test_every_split_count_is_bit_identical(blocks):
    M, K, N = 16, 2048, 384
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=3)
    slabs = (N // 64) * (K // 32)
    b = slabs if blocks == -1 else blocks          # -1: one CTA per slab, every tile split K/32 ways
    case = W8A8Case(x, xs, W, ws, blocks=b)
    _check(case, x, xs, W, ws)


def test_adversarial_cancelling_partial_sums():
    # Runs of +-127*127 products: inside one 512-k accumulation window the partial sums reach up to
    # 512 * 16129 ~ 2^23, across windows they cancel exactly, and one weight per column moved toward
    # zero leaves a small exact result.  With unit scales bf16 holds it exactly, so an inexact
    # accumulation anywhere would show.
    M, K, N = 16, 4096, 256
    x = np.full((M, K), 127, np.int8)
    x[1::2] = -127
    W = np.zeros((K, N), np.int8)
    for n in range(N):
        run = [1, 32, 256, 512, 1024, 2048][n % 6]
        W[:, n] = np.where((np.arange(K) // run) % 2 == 0, 127, -127)
        k0 = (n * 37) % K
        d = n % 3
        W[k0, n] = W[k0, n] - d if W[k0, n] > 0 else W[k0, n] + d
    xs = np.ones(M, np.float32)
    ws = np.ones(N, np.float32)
    acc = oracle.w8a8_acc(x, W)
    assert np.abs(acc).max() <= 256 and np.abs(acc).max() > 0
    for blocks in (0, 1, 37):
        case = W8A8Case(x, xs, W, ws, blocks=blocks)
        _check(case, x, xs, W, ws)


@pytest.mark.parametrize("fill", [127, -128])
def test_extremes(fill):
    M, K, N = 32, 12288, 128
    x = np.full((M, K), fill, np.int8)
    W = np.full((K, N), fill, np.int8)
    xs = np.full(M, 2.0**-10, np.float32)
    ws = np.full(N, 2.0**-12, np.float32)
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("M", [1, 4, 8, 16, 32])
@pytest.mark.parametrize("N,K", [(2560, 4096), (4096, 2048)])
def test_sweep_shapes(M, N, K):
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=1000 * 3 + M)
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


def test_fused_qkv_shape():
    x, xs, W, ws = synth.w8a8_inputs(16, 4096, 1536, seed=1)
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("N,K", [(24576, 4096), (4096, 12288)])
def test_mlp_shapes(N, K):
    x, xs, W, ws = synth.w8a8_inputs(16, K, N, seed=4000 + N, dist="mlp")
    case = W8A8Case(x, xs, W, ws)
    _check(case, x, xs, W, ws)


def test_untouched_rows_and_columns():
    # The output is written in place into a larger buffer: the bytes after [M, N] stay untouched.
    M, K, N = 5, 512, 200
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=5)
    case = W8A8Case(x, xs, W, ws)
    buf = torch.full((M * N + 64,), 3.0, dtype=torch.bfloat16, device="cuda")
    res = case.run(out=buf[: M * N].view(M, N))
    torch.cuda.synchronize()
    assert (buf[M * N:] == 3.0).all()
    np.testing.assert_array_equal(bf16_bits(res), oracle.w8a8_gemm(x, xs, W, ws))


def test_counters_return_to_zero_and_calls_repeat():
    M, K, N = 16, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=2)
    case = W8A8Case(x, xs, W, ws, blocks=3072)     # workspace sized for the largest split count
    ref = oracle.w8a8_gemm(x, xs, W, ws)
    for blocks in (0, 1, 304, 3072, 5, 0):
        got = bf16_bits(case.run(blocks=blocks))
        np.testing.assert_array_equal(got, ref)
    # Between calls the whole workspace past its status word is zero again: each split-tile
    # accumulator word is returned to zero by the element's last arrival.
    torch.cuda.synchronize()
    assert (case.ws[4:] == 0).all()
    assert case.status() == 0


def test_graph_replay_is_bitwise_the_direct_call():
    M, K, N = 16, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=8)
    case = W8A8Case(x, xs, W, ws)
    direct = bf16_bits(case.run())
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        case.run(out=out)                  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        case.run(out=out)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(out), direct)
    np.testing.assert_array_equal(direct, oracle.w8a8_gemm(x, xs, W, ws))
    assert case.status() == 0


def test_a_changed_weight_byte_changes_exactly_its_column():
    M, K, N = 4, 512, 256
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=12)
    base = bf16_bits(W8A8Case(x, xs, W, ws).run())
    W2 = W.copy()
    W2[100, 77] = np.int8(-W2[100, 77] if W2[100, 77] != 0 else 5)
    got = bf16_bits(W8A8Case(x, xs, W2, ws).run())
    np.testing.assert_array_equal(got, oracle.w8a8_gemm(x, xs, W2, ws))
    changed = np.nonzero((got != base).any(axis=0))[0]
    assert set(changed.tolist()) <= {77}


@pytest.mark.parametrize("M,K,N,blocks", [(16, 4096, 1536, 0), (5, 2048, 4096, 7), (32, 1024, 520, 0)])
def test_weights_rewritten_just_before_a_call_are_the_ones_read(M, K, N, blocks):
    # Every call is launched as a programmatic dependent of the work before it; without
    # W8A8_FLAG_PDL it must still behave as plain stream order.  Here the packed weight buffer is
    # repacked with new values by the kernel right before each call, on the same stream, with no
    # synchronisation: a call that read its weight before the pack had finished would see the old
    # values.  The activations and scales are rewritten the same way.
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=M + K + N)
    x2, xs2, W2, ws2 = synth.w8a8_inputs(M, K, N, seed=M + K + N + 1)
    dev = torch.device("cuda")
    xd = torch.from_numpy(x).to(dev)
    xsd = torch.from_numpy(xs).to(dev)
    wsd = torch.from_numpy(ws).to(dev)
    Wd = [torch.from_numpy(W).to(dev), torch.from_numpy(W2).to(dev)]
    srcs = [(torch.from_numpy(x).to(dev), torch.from_numpy(xs).to(dev), torch.from_numpy(ws).to(dev)),
            (torch.from_numpy(x2).to(dev), torch.from_numpy(xs2).to(dev), torch.from_numpy(ws2).to(dev))]
    refs = [oracle.w8a8_gemm(x, xs, W, ws), oracle.w8a8_gemm(x2, xs2, W2, ws2)]
    wsp = lib8.alloc_workspace(lib8.w8a8_workspace_bytes(M, K, N, blocks), dev)
    Wp = lib8.w8a8_pack_weights(Wd[0], ws=wsp)
    torch.cuda.synchronize()
    outs = []
    for i in range(6):
        j = i % 2
        lib8.w8a8_pack_weights(Wd[j], W_packed=Wp)       # rewrites the whole packed weight
        xd.copy_(srcs[j][0])
        xsd.copy_(srcs[j][1])
        wsd.copy_(srcs[j][2])
        outs.append(lib8.w8a8_gemm(xd, xsd, Wp, wsd, wsp, N, blocks=blocks))
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        np.testing.assert_array_equal(bf16_bits(o), refs[i % 2])
    assert lib8.w8a8_workspace_status(wsp) == 0


@pytest.mark.parametrize("blocks", [0, 7, 3072])
def test_pdl_calls_back_to_back_are_bit_identical(blocks):
    # Programmatic dependent launch: consecutive calls overlap (the next call prefetches its weight
    # during the previous call's tail) and must still produce the oracle's bits, call after call.
    M, K, N = 16, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=21)
    case = W8A8Case(x, xs, W, ws, blocks=blocks)
    torch.cuda.synchronize()            # the packed weight is complete before any call prefetches it
    ref = oracle.w8a8_gemm(x, xs, W, ws)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    for o in outs:
        case.run(out=o, flags=lib8.W8A8_FLAG_PDL)
    torch.cuda.synchronize()
    for o in outs:
        np.testing.assert_array_equal(bf16_bits(o), ref)
    assert case.status() == 0


def test_pdl_graph_replay_chain():
    # A captured chain of PDL calls on different weights, each reading the previous call's output
    # as nothing but a buffer it overwrites: every replay reproduces the oracle.
    M, K, N = 8, 2048, 4096
    cases = []
    for seed in (31, 32, 33):
        x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=seed)
        cases.append((W8A8Case(x, xs, W, ws), oracle.w8a8_gemm(x, xs, W, ws)))
    torch.cuda.synchronize()
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in cases]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for (c, _), o in zip(cases, outs):
            c.run(out=o, flags=lib8.W8A8_FLAG_PDL)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (c, _), o in zip(cases, outs):
            c.run(out=o, flags=lib8.W8A8_FLAG_PDL)
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for (_, ref), o in zip(cases, outs):
            np.testing.assert_array_equal(bf16_bits(o), ref)
    del out


@pytest.mark.parametrize("fx,fw", [(-128, -128), (127, -128), (-128, 127)])
def test_two_element_combine_at_its_range_limits(fx, fw):
    # K = 4096 with constant extremes drives every element's partial sums to the edge of the
    # two-element word's fields (|sum| up to K * 2^14 = 2^26 in 28-bit fields), with 128 CTAs per
    # tile (the count field's 8 bits near full).
    M, K, N = 32, 4096, 128
    x = np.full((M, K), fx, np.int8)
    W = np.full((K, N), fw, np.int8)
    x[5] = -x[5] if fx != -128 else 127
    xs = np.full(M, 2.0**-12, np.float32)
    ws = np.full(N, 2.0**-14, np.float32)
    for blocks in (256, 0, 5):
        case = W8A8Case(x, xs, W, ws, blocks=blocks)
        if blocks == 256:
            assert lib8.w8a8_plan(M, K, N, blocks)["combine_pack_bits"] == 28
        _check(case, x, xs, W, ws)


def test_read_probe_runs_and_leaves_its_input_alone():
    buf = torch.randint(0, 256, (1 << 22,), dtype=torch.uint8, device="cuda")
    ref = buf.clone()
    sink = torch.zeros(1, dtype=torch.int64, device="cuda")
    lib8.w8a8_read_probe(buf, sink)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref)


@pytest.mark.parametrize("K,N,blocks", [(65536, 256, 3), (65536, 256, 1), (4096, 256, 3), (4096, 512, 3),
                                        (2048, 512, 3), (4096, 1536, 10)])
def test_multi_segment_ctas_with_both_word_formats(K, N, blocks):
    # Fewer CTAs than tiles: each CTA streams a run across several tiles, and the combine warp
    # finishes every segment but a CTA's last.  K = 65536 leaves no room for two elements per word
    # (one-element words); the others use two-element words.  The runs go in 4-slab units, and the
    # walk orders of a CTA's segments all occur: two swapped (K = 65536 and 4096 with N = 256),
    # three as first, last, middle (K = 4096, N = 512 and 1536), three or more in natural order
    # (K = 2048, and the runs of four segments).
    M = 5
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=K + blocks)
    plan = lib8.w8a8_plan(M, K, N, blocks)
    assert plan["threads"] == 320 and plan["split_unit"] == 4
    assert plan["combine_pack_bits"] == (0 if K == 65536 else {4096: 28, 2048: 27}[K])
    case = W8A8Case(x, xs, W, ws, blocks=blocks)
    _check(case, x, xs, W, ws)
    torch.cuda.synchronize()
    assert (case.ws[4:] == 0).all()
