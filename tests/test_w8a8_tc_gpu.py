"""W8A8 GEMM for 32 < M <= 128 (the tcgen05 arm) on the GPU against the oracle, bit for bit.

The arm reads the same packed weight as the decode arm, so every case packs once and calls
w8a8_gemm with M > 32.  Cases: ragged M on both MMA widths (64 and 128 activation rows), an odd
number of 64-row packed tiles (the last 128-row tile has one half), ragged K (partial stages),
every split-count class, adversarial partial sums that reach 2^23 inside one 512-k accumulation
window and cancel across windows, int32 extremes, the sweep and MLP shapes (full-size MLP outputs
compared on sampled columns the oracle computes one by one), graph replay, programmatic dependent
launch, and the workspace contract.
"""
import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import W8A8Case, bf16_bits


class TcCase(W8A8Case):
    """A W8A8 case whose calls always run the tensor-memory arm (the automatic plan may run 32-row
    decode chunks instead on small weights; those are tested in test_w8a8_route_gpu.py)."""

    base_flags = lib8.W8A8_FLAG_TENSOR_MEMORY_ARM

pytestmark = pytest.mark.gpu


def _zeroed_end(N):
    # End of the regions that are zero between calls (header word aside): counters and int32 planes
    # of the 128-row tiles; the fp16 activations follow them.
    T = -(-N // 128)
    return 256 + -(-T * 4 // 256) * 256 + T * 128 * 128 * 4


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


def test_plan_uses_the_tensor_memory_arm():
    for M, n8 in ((33, 8), (64, 8), (65, 16), (128, 16)):
        pl = lib8.w8a8_plan(M, 4096, 1536, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)
        assert pl["tensor_memory"] == 1 and pl["tile_rows"] == 128 and pl["n8_tiles"] == n8
    assert lib8.w8a8_plan(32, 4096, 1536)["tensor_memory"] == 0


@pytest.mark.parametrize("M", [33, 40, 48, 63, 64, 65, 96, 127, 128])
def test_ragged_m(M):
    x, xs, W, ws = synth.w8a8_inputs(M, 1024, 200, seed=M)
    case = TcCase(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("M", [48, 128])
@pytest.mark.parametrize("K,N", [(32, 8), (96, 136), (4000, 320), (4096, 320), (416, 4096), (2048, 520)])
def test_ragged_shapes(M, K, N):
    # N = 320: five packed tiles, so the third 128-row tile has only its first half; K = 4000 and
    # K = 416: the last stage of a segment holds fewer than four 32-k units.
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=K + N + M)
    case = TcCase(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("blocks", [1, 2, 3, 7, 64, 151, 152, 192, 0])
def test_every_split_count_is_bit_identical(blocks):
    # 3 tiles of 128 rows x 64 units: one CTA per tile up to one CTA per unit.
    M, K, N = 100, 2048, 384
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=3)
    case = TcCase(x, xs, W, ws, blocks=blocks)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("M", [64, 128])
def test_adversarial_cancelling_partial_sums(M):
    # Runs of +-127*127 products: inside one 512-k accumulation window the partial sums reach up to
    # 512 * 16129 ~ 2^23, across windows they cancel, and one weight per column moved toward zero
    # leaves a small exact result; unit scales make bf16 hold it exactly.
    K, N = 4096, 256
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
        case = TcCase(x, xs, W, ws, blocks=blocks)
        _check(case, x, xs, W, ws)


@pytest.mark.parametrize("fill", [127, -128])
def test_extremes(fill):
    M, K, N = 128, 12288, 128
    x = np.full((M, K), fill, np.int8)
    W = np.full((K, N), fill, np.int8)
    xs = np.full(M, 2.0**-10, np.float32)
    ws = np.full(N, 2.0**-12, np.float32)
    case = TcCase(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("M", [64, 128])
@pytest.mark.parametrize("N,K", [(1536, 4096), (2560, 4096), (4096, 2048)])
def test_sweep_shapes(M, N, K):
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=1000 * 3 + M)
    case = TcCase(x, xs, W, ws)
    _check(case, x, xs, W, ws)


@pytest.mark.parametrize("N,K", [(24576, 4096), (4096, 12288)])
def test_mlp_shapes_on_sampled_columns(N, K):
    # The full output is too large for the oracle in a test: columns are independent, so the
    # oracle computes a seeded sample of whole columns (every tile's first and last column among
    # them) and those are compared bit for bit.
    M = 128
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=4000 + N, dist="mlp")
    case = TcCase(x, xs, W, ws)
    out, acc = case.run_acc()
    torch.cuda.synchronize()
    got = bf16_bits(out)
    rng = np.random.default_rng(N + K)
    cols = np.unique(np.concatenate([rng.choice(N, 96, replace=False), [0, 127, 128, N - 128, N - 1]]))
    Wc = np.ascontiguousarray(W[:, cols])
    np.testing.assert_array_equal(got[:, cols], oracle.w8a8_gemm(x, xs, Wc, ws[cols]))
    np.testing.assert_array_equal(acc.cpu().numpy()[:, cols].astype(np.int64), oracle.w8a8_acc(x, Wc))
    assert case.status() == 0


def test_untouched_rows_and_columns():
    M, K, N = 70, 512, 200
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=5)
    case = TcCase(x, xs, W, ws)
    buf = torch.full((M * N + 64,), 3.0, dtype=torch.bfloat16, device="cuda")
    res = case.run(out=buf[: M * N].view(M, N))
    torch.cuda.synchronize()
    assert (buf[M * N:] == 3.0).all()
    np.testing.assert_array_equal(bf16_bits(res), oracle.w8a8_gemm(x, xs, W, ws))


def test_counters_and_planes_return_to_zero_and_calls_repeat():
    M, K, N = 128, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=2)
    case = TcCase(x, xs, W, ws, blocks=1536)      # workspace sized for the largest split count
    ref = oracle.w8a8_gemm(x, xs, W, ws)
    for blocks in (0, 1, 152, 1536, 5, 0):
        got = bf16_bits(case.run(blocks=blocks))
        np.testing.assert_array_equal(got, ref)
    torch.cuda.synchronize()
    assert (case.ws[4:_zeroed_end(N)] == 0).all()
    assert case.status() == 0


def test_decode_and_tensor_memory_arms_share_one_workspace():
    # One workspace sized for M_max = 128 serves calls of both arms in turn.
    K, N = 2048, 1024
    _, _, W, ws = synth.w8a8_inputs(1, K, N, seed=40)
    size = lib8.w8a8_workspace_bytes(128, K, N)
    work = lib8.alloc_workspace(size)
    Wp = lib8.w8a8_pack_weights(torch.from_numpy(W).cuda())
    wsd = torch.from_numpy(ws).cuda()
    for M in (16, 128, 32, 33, 1, 64, 128, 40, 128, 8):
        x, xs, _, _ = synth.w8a8_inputs(M, K, N, seed=40 + M)
        out = lib8.w8a8_gemm(torch.from_numpy(x).cuda(), torch.from_numpy(xs).cuda(), Wp, wsd, work, N,
                             flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM if M > 32 else 0)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(out), oracle.w8a8_gemm(x, xs, W, ws))
    assert (work[4:_zeroed_end(N)] == 0).all()
    assert lib8.w8a8_workspace_status(work) == 0


def test_graph_replay_is_bitwise_the_direct_call():
    M, K, N = 96, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=8)
    case = TcCase(x, xs, W, ws)
    direct = bf16_bits(case.run())
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        case.run(out=out)
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


@pytest.mark.parametrize("blocks", [0, 7, 384])
def test_pdl_calls_back_to_back_are_bit_identical(blocks):
    M, K, N = 128, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=21)
    case = TcCase(x, xs, W, ws, blocks=blocks)
    torch.cuda.synchronize()
    ref = oracle.w8a8_gemm(x, xs, W, ws)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    for o in outs:
        case.run(out=o, flags=lib8.W8A8_FLAG_PDL)
    torch.cuda.synchronize()
    for o in outs:
        np.testing.assert_array_equal(bf16_bits(o), ref)
    assert case.status() == 0
