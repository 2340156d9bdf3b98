"""CPU tests of the C-ABI library: it loads, exports every symbol include/w8a8.h declares, and its
host-only logic (sizes, plans, split bounds, argument checks) is right.  No kernel runs here."""
import ctypes
import os
import re

import numpy as np
import pytest

import int8_weight_gemm_gb300 as lib8
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("W8A8_GB300")))


def test_header_declares_the_expected_entry_points():
    names = _declared_functions()
    for required in ("w8a8_pack_weights", "w8a8_gemm", "q8_0_gemv"):
        assert required in names
    assert set(names) == set(lib8.SIGNATURES), (set(names) ^ set(lib8.SIGNATURES))


def test_library_exports_every_declared_symbol():
    L = lib8.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_version_and_status_strings():
    assert lib8.w8a8_version() >= 100
    assert lib8.lib().w8a8_status_string(0) == b"ok"
    assert lib8.lib().w8a8_status_string(4) == b"workspace too small"


@pytest.mark.parametrize("K,N", [(512, 256), (4096, 1536), (32, 8), (96, 200), (12288, 4096)])
def test_packed_bytes_match_oracle_layout(K, N):
    assert lib8.w8a8_packed_weight_bytes(K, N) == oracle.w8a8_packed_bytes(K, N)


@pytest.mark.parametrize("K,N,blocks", [(512, 256, 0), (4096, 1536, 0), (4096, 1536, 7), (4096, 24576, 0),
                                        (64, 200, 0), (64, 200, 8), (12288, 4096, 304), (32, 8, 1),
                                        (4096, 2560, 0), (2048, 4096, 0), (4096, 1536, 3072), (4096, 1536, 25),
                                        (4096, 1536, 24), (4096, 1536, 23), (96, 136, 0)])
def test_split_bounds_cover_every_slab_once(K, N, blocks):
    plan = lib8.w8a8_plan(1, K, N, blocks)
    G, U, KB, T = plan["blocks"], plan["slabs"], plan["k_blocks"], plan["n_tiles"]
    assert U == -(-N // 64) * (K // 32) == T * KB
    b = np.array(lib8.w8a8_split_bounds(K, N, G))
    assert b[0] == 0 and b[-1] == U and len(b) == G + 1
    sizes = np.diff(b)
    assert (sizes >= 1).all()                         # no empty run (the combine relies on it)
    # Brute force: the CTAs whose runs touch each tile.
    owner = np.searchsorted(b[1:], np.arange(U), side="right")
    contrib = [sorted(set(owner[t * KB:(t + 1) * KB].tolist())) for t in range(T)]
    for cs in contrib:
        assert cs == list(range(cs[0], cs[-1] + 1))  # a tile's contributors are consecutive CTAs
    if G >= T:
        # Tile-aligned: no run crosses a tile, tile t has c + 1 parts if t < G % T else c, and the
        # parts of one tile are equal to within one slab.
        assert all(b0 // KB == (b1 - 1) // KB for b0, b1 in zip(b[:-1], b[1:]))
        c, e = G // T, G % T
        for t, cs in enumerate(contrib):
            assert len(cs) == (c + 1 if t < e else c)
            part = sizes[cs[0]:cs[-1] + 1]
            assert part.max() - part.min() <= 1
    else:
        # Linear: runs of a + 1 units of q slabs, then runs of a; the kernel counts a tile's
        # contributors from the owners of its first and last slab with this arithmetic.
        q = plan["split_unit"]
        assert q in (1, 4) and U % q == 0
        a, r = (U // q) // G, (U // q) % G
        assert (sizes[:r] == q * (a + 1)).all() and (sizes[r:] == q * a).all()
        def owner_of(u):
            u //= q
            head = r * (a + 1)
            return u // (a + 1) if u < head else r + (u - head) // a
        for t, cs in enumerate(contrib):
            assert owner_of(t * KB + KB - 1) - owner_of(t * KB) + 1 == len(cs)


@pytest.mark.parametrize("K,N,blocks,unit", [
    (4096, 24576, 0, 4),    # 49152 slabs over 304 CTAs: runs of 164 / 160 against 162 / 161 slabs
    (4096, 24576, 304, 4),
    (4096, 1536, 0, 1),     # tile-aligned split: units do not apply
    (96, 24576, 0, 1),      # K / 32 = 3 k-blocks: no 4-slab unit inside a tile
    (128, 25600, 0, 1),     # 1600 slabs: whole units would make the longest run 8 against 6 slabs
    (8192, 32768, 0, 4),
    (4096, 24576, 7, 4),
])
def test_linear_split_unit_follows_its_rule(K, N, blocks, unit):
    plan = lib8.w8a8_plan(16, K, N, blocks)
    assert plan["split_unit"] == unit
    b = np.array(lib8.w8a8_split_bounds(K, N, plan["blocks"]))
    if unit == 4:
        assert (b % 4 == 0).all()   # every run starts on an 8 KiB boundary of the packed weight
        U, G = plan["slabs"], plan["blocks"]
        assert np.diff(b).max() * 100 <= -(-U // G) * 103
    # The tensor-memory arm keeps runs of single 32-k units.
    assert lib8.w8a8_plan(64, K, N, 0, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)["split_unit"] == 1


def test_automatic_split_keeps_every_cta_inside_one_tile_for_small_outputs():
    # The fused-QKV-like shape: 24 tiles over 304 CTAs, 16 tiles cut 13 ways and 8 cut 12 ways,
    # runs of 9 to 11 slabs, and no CTA finishing two tile segments.
    b = np.array(lib8.w8a8_split_bounds(4096, 1536, 304))
    sizes = np.diff(b)
    assert sizes.min() == 9 and sizes.max() == 11
    assert all(b0 // 128 == (b1 - 1) // 128 for b0, b1 in zip(b[:-1], b[1:]))


@pytest.mark.parametrize("M", [1, 8, 16, 24, 32])
@pytest.mark.parametrize("K,N", [(4096, 1536), (4096, 2560), (2048, 4096), (4096, 6144), (4096, 8192),
                                 (4096, 12288), (1024, 4096), (12288, 4096), (14336, 4096), (8192, 1536),
                                 (4096, 24576), (512, 256)])
def test_automatic_count_cuts_every_tile_equally_up_to_k_4096(M, K, N):
    # The automatic CTA count: two per SM (152 SMs without a GPU), at most one per slab; with
    # K <= 4096 and at least one CTA per tile, the largest multiple of the tile count that fits,
    # so every tile is cut into the same number of parts, each within one slab of KB / c.
    p = lib8.w8a8_plan(M, K, N)
    T, KB, G = p["n_tiles"], p["k_blocks"], p["blocks"]
    g = min(2 * 152, T * KB)
    if KB <= 128 and g >= T:
        assert G == T * (g // T)
        c = G // T
        sizes = np.diff(np.array(lib8.w8a8_split_bounds(K, N, G, M=M)))
        assert sizes.max() - sizes.min() <= 1 and sizes.max() == -(-KB // c)
    else:
        assert G == g


def test_split_slices_reproduce_the_oracle_sums():
    # Host replay of the plan: summing each CTA's k-slices of every tile in int32, in ascending CTA
    # order, must give the oracle's sums (the invariant behind the combine).
    M, K, N, G = 3, 256, 128, 5
    x, _, W, _ = synth.w8a8_inputs(M, K, N, seed=4)
    ref = oracle.w8a8_acc(x, W)
    b = lib8.w8a8_split_bounds(K, N, G)
    KB = K // 32
    for t in range(N // 64):
        cuts = sorted(set([0, K] + [32 * (u - t * KB) for u in b if t * KB < u < (t + 1) * KB]))
        cols = slice(64 * t, 64 * t + 64)
        np.testing.assert_array_equal(oracle.w8a8_acc_split(x, W[:, cols], cuts), ref[:, cols])


def test_plan_shape_and_limits():
    p = lib8.w8a8_plan(16, 4096, 1536)
    assert p["n8_tiles"] == 2 and p["n_tiles"] == 24 and p["k_blocks"] == 128
    assert p["blocks"] == 288                                   # 12 parts of each of the 24 tiles (<= 2 CTAs per SM)
    assert lib8.w8a8_plan(32, 2048, 4096)["blocks"] == 256       # 4 parts of each of the 64 tiles
    assert lib8.w8a8_plan(16, 12288, 4096)["blocks"] == 304      # K > 4096: two CTAs per SM (152 SMs without a GPU)
    assert lib8.w8a8_plan(16, 4096, 24576)["blocks"] == 304      # fewer CTAs than tiles: two per SM
    assert lib8.w8a8_plan(1, 512, 256)["blocks"] == 64           # never more CTAs than slabs
    # a combine warp only when some CTA finishes more than one tile segment (fewer CTAs than tiles)
    assert p["threads"] == 288 and lib8.w8a8_plan(16, 4096, 24576)["threads"] == 320
    assert p["smem_bytes"] * 2 <= 228 * 1024          # two CTAs per SM fit
    for M in (1, 8, 9, 16, 17, 24, 25, 32):
        q = lib8.w8a8_plan(M, 4096, 1536)
        assert q["n8_tiles"] == (M + 7) // 8
        # consumer warps take stages by parity: an even ring keeps each slot with one parity group
        assert q["stages"] % 2 == 0
    # the size query covers every M up to M_max
    big = lib8.w8a8_workspace_bytes(32, 4096, 1536)
    assert all(lib8.w8a8_plan(M, 4096, 1536)["workspace_bytes"] <= big for M in range(1, 33))


def test_tensor_memory_arm_plan():
    # 32 < M <= 128: 128-row tiles (two packed tiles), one CTA per SM, MMA N = 64 or 128.
    p = lib8.w8a8_plan(128, 4096, 1536, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)
    assert p["tensor_memory"] == 1 and p["tile_rows"] == 128 and p["n8_tiles"] == 16
    assert p["n_tiles"] == 12 and p["k_blocks"] == 128 and p["slabs"] == 12 * 128
    assert p["blocks"] == 152 and p["threads"] == 608 and p["smem_bytes"] <= 227 * 1024
    q = lib8.w8a8_plan(33, 4096, 320, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)
    assert q["n8_tiles"] == 8 and q["n_tiles"] == 3 and q["threads"] == 640
    assert lib8.w8a8_plan(32, 4096, 320)["tensor_memory"] == 0
    # header, counters (one per tile, padded to 256 bytes), int32 planes [tile][128][128] whatever
    # M (so that no region moves with M), then the fp16 activations [M][K]
    assert p["workspace_bytes"] == 256 + 256 + 12 * 128 * 128 * 4 + 128 * 4096 * 2
    assert q["workspace_bytes"] == 256 + 256 + 3 * 128 * 128 * 4 + 33 * 4096 * 2
    # with at least as many 128-row tiles as SMs, a CTA count dividing the tile count (whole tiles)
    assert lib8.w8a8_plan(128, 4096, 24576)["blocks"] == 96
    assert lib8.w8a8_plan(128, 12288, 4096)["blocks"] == 152
    # the size query for M_max covers both arms, forced or automatic, and the row-chunk plans
    big = lib8.w8a8_workspace_bytes(128, 4096, 1536)
    for f in (0, lib8.W8A8_FLAG_TENSOR_MEMORY_ARM):
        assert all(lib8.w8a8_plan(M, 4096, 1536, flags=f)["workspace_bytes"] <= big for M in range(1, 129))
    assert lib8.w8a8_workspace_bytes(129, 4096, 1536) == 0


def test_automatic_plan_routes_mid_m_by_the_cost_model():
    # 32 < M <= 128: decode row chunks on small weights, the tensor-memory arm on large ones; the
    # flag or an explicit CTA count forces the tensor-memory arm.
    p = lib8.w8a8_plan(64, 4096, 2560)
    assert p["tensor_memory"] == 0 and p["row_chunks"] == 2 and p["n8_tiles"] == 4
    assert lib8.w8a8_plan(96, 4096, 1536)["row_chunks"] == 3
    assert lib8.w8a8_plan(40, 4096, 1536)["row_chunks"] == 2
    g = lib8.w8a8_plan(128, 4096, 24576)
    assert g["tensor_memory"] == 1 and g["row_chunks"] == 1
    assert lib8.w8a8_plan(64, 4096, 2560, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)["tensor_memory"] == 1
    assert lib8.w8a8_plan(64, 4096, 2560, blocks=40)["tensor_memory"] == 1
    assert all(lib8.w8a8_plan(M, 4096, 1536)["row_chunks"] == 1 for M in range(1, 33))
    # every M in (32, 128] at these shapes is either arm, and the size query covers both
    for (K, N) in ((4096, 1536), (2048, 4096), (4096, 24576)):
        big = lib8.w8a8_workspace_bytes(128, K, N)
        for M in range(33, 129):
            p = lib8.w8a8_plan(M, K, N)
            assert p["workspace_bytes"] <= big
            assert p["tensor_memory"] == 1 or p["row_chunks"] == -(-M // 32)


@pytest.mark.parametrize("M,K,N,blocks", [(64, 4096, 1536, 0), (128, 4096, 24576, 0), (100, 2048, 384, 7),
                                          (33, 4000, 320, 0), (128, 32, 8, 1), (65, 12288, 4096, 304)])
def test_tensor_memory_arm_split_bounds(M, K, N, blocks):
    plan = lib8.w8a8_plan(M, K, N, blocks, flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)
    G, U, KB, T = plan["blocks"], plan["slabs"], plan["k_blocks"], plan["n_tiles"]
    assert T == -(-N // 128) and U == T * KB
    b = np.array(lib8.w8a8_split_bounds(K, N, G, M=M))
    assert b[0] == 0 and b[-1] == U and len(b) == G + 1 and (np.diff(b) >= 1).all()
    if G >= T:
        assert all(b0 // KB == (b1 - 1) // KB for b0, b1 in zip(b[:-1], b[1:]))


def test_tensor_memory_arm_operands_emulated():
    # CPU replay of the tensor-memory arm's operand layout: each converter thread writes its packed
    # 16-byte chunk with the 16x256b store (thread t: lanes t/4 and t/4 + 8, columns 2(t%4), 2(t%4)+1
    # and those plus 8), and the fp16 activation copy reorders each 32-k unit's groups of four as
    # 0, 2, 4, 6, 1, 3, 5, 7.  Column j of a row then pairs with activation positions 2j, 2j + 1, and
    # the dot product over all columns must equal x @ W exactly.
    M, K, N = 3, 64, 128
    x = synth.uniform_int8(6, "tc.x", (M, K), lo=-128, hi=127).astype(np.int64)
    W = synth.uniform_int8(5, "tc.W", (K, N), lo=-128, hi=127)
    packed = oracle.w8a8_pack(W).astype(np.int64)
    KB = K // 32

    def sbyte(b):
        b ^= 0x80
        return b - 256 if b >= 128 else b

    # tensor memory A: [row][unit][column j] -> (k0, k1) weight values
    A = np.zeros((128, KB, 16, 2), np.int64)
    for quad in range(4):
        half = quad >> 1
        for unit in range(KB):
            for r in range(2):
                s16 = 2 * (quad & 1) + r
                for t in range(32):
                    off = (half * KB + unit) * 2048 + (s16 * 32 + t) * 16
                    words = [[sbyte(int(packed[off + 4 * wi + b])) for b in range(4)] for wi in range(4)]
                    # four conversions -> eight registers of two values (natural pairs)
                    h = []
                    for wi in range(4):
                        h += [words[wi][0:2], words[wi][2:4]]
                    g, c = t // 4, t % 4
                    lane_of = [g, g, g + 8, g + 8, g, g, g + 8, g + 8]
                    col_of = [2 * c, 2 * c + 1, 2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c, 8 + 2 * c, 9 + 2 * c]
                    # registers: v0 = h0 (row g), v1 = h1, v2 = h2 (row g+8), v3 = h3, v4 = h4, ...
                    for v in range(8):
                        A[32 * quad + 16 * r + lane_of[v], unit, col_of[v]] = h[v]
    # fp16 activation copy: groups of four reordered 0, 2, 4, 6, 1, 3, 5, 7 within each unit
    order = [0, 2, 4, 6, 1, 3, 5, 7]
    B = np.zeros((M, KB, 32), np.int64)
    for m in range(M):
        for unit in range(KB):
            for gi, src in enumerate(order):
                B[m, unit, 4 * gi:4 * gi + 4] = x[m, 32 * unit + 4 * src:32 * unit + 4 * src + 4]
    got = np.einsum("nujq,mujq->mn", A, B.reshape(M, KB, 16, 2))
    np.testing.assert_array_equal(got, x @ W.astype(np.int64))


def test_two_element_combine_words():
    # Field width from K (partial sums of an element are at most K * 2^14 in magnitude) and the
    # arrival count in the remaining bits; one element per word when the count would not fit.
    assert lib8.w8a8_plan(16, 4096, 1536)["combine_pack_bits"] == 28
    assert lib8.w8a8_plan(16, 12288, 4096)["combine_pack_bits"] == 29
    assert lib8.w8a8_plan(16, 4096, 1536, 3072)["combine_pack_bits"] == 28      # 128 CTAs per tile
    assert lib8.w8a8_plan(32, 12288, 128)["combine_pack_bits"] == 0             # 152 > 63 per tile
    assert lib8.w8a8_plan(1, 65536, 64, 1)["combine_pack_bits"] == 0            # fields too wide


def test_two_element_word_arithmetic():
    # Host emulation of the combine word: every CTA adds 2^(2f) + b * 2^f + a (mod 2^64) and
    # decodes the sums and count of the partials added before its own from the returned word.
    rng = np.random.default_rng(5)
    M64 = (1 << 64) - 1
    def sext(v, f):
        v &= (1 << f) - 1
        return v - (1 << f) if v >> (f - 1) else v
    for K, n in ((4096, 13), (4096, 255), (12288, 63), (32, 1000)):
        f = (K << 14).bit_length() + 1
        assert 64 - 2 * f >= 1 and n < 1 << (64 - 2 * f)
        lim = K << 14
        for trial in range(20):
            # partials of n CTAs over disjoint k-ranges: their sum stays within +-K * 2^14
            cuts = np.sort(rng.choice(np.arange(1, K), size=min(n - 1, K - 1), replace=False)) if n > 1 else []
            ks = np.diff(np.concatenate([[0], cuts, [K]])).astype(np.int64)
            extreme = trial % 3
            pa = [int(k) * (16384 if extreme == 0 else -16256 if extreme == 1 else int(rng.integers(-16384, 16385)))
                  for k in ks]
            pb = [int(k) * int(rng.integers(-16384, 16385)) for k in ks]
            w = 0
            for i, (a, b) in enumerate(zip(pa, pb)):
                old = w
                a_old = sext(old, f)
                w1 = ((old - a_old) & M64) >> f
                b_old = sext(w1, f)
                cnt = ((w1 - b_old) & M64) >> f
                assert (a_old, b_old, cnt) == (sum(pa[:i]), sum(pb[:i]), i)
                w = (old + (1 << (2 * f)) + (b << f) + a) & M64
            assert abs(sum(pa)) <= lim and abs(sum(pb)) <= lim


@pytest.mark.parametrize("M,K,N,blocks,code", [
    (0, 512, 256, 0, 1), (129, 512, 256, 0, 1), (1, 0, 256, 0, 1), (1, 512, 0, 0, 1),
    (64, 500, 256, 0, 2), (64, 512, 250, 0, 2), (64, 512, 256, 10**6, 1),
    (1, 500, 256, 0, 2), (1, 512, 250, 0, 2), (1, 512, 256, -1, 1), (1, 512, 256, 10**6, 1)])
def test_plan_rejects_bad_shapes(M, K, N, blocks, code):
    p = lib8.PlanT()
    assert lib8.lib().w8a8_plan(M, K, N, blocks, ctypes.byref(p)) == code
    assert lib8.w8a8_workspace_bytes(M, K, N, blocks) == 0 or code == 0


def test_read_probe_checks_its_arguments_on_the_host():
    L = lib8.lib()
    a = ctypes.c_void_p(1 << 20)
    assert L.w8a8_read_probe(None, 1 << 20, a, None) == 1
    assert L.w8a8_read_probe(a, 8, a, None) == 1
    assert L.w8a8_read_probe(ctypes.c_void_p((1 << 20) + 8), 1 << 20, a, None) == 3
    assert L.w8a8_read_probe(a, 1 << 20, ctypes.c_void_p((1 << 20) + 4), None) == 3


def test_mma_rate_probe_checks_its_arguments_on_the_host():
    L = lib8.lib()
    a = ctypes.c_void_p(1 << 20)
    assert L.w8a8_mma_rate_probe(2, 10, a, None) == 1          # unknown kind
    assert L.w8a8_mma_rate_probe(0, 0, a, None) == 1           # no iterations
    assert L.w8a8_mma_rate_probe(1, 10, None, None) == 1       # no sink
    assert L.w8a8_mma_rate_probe(0, 10, ctypes.c_void_p((1 << 20) + 4), None) == 3


def test_quantisation_entry_points_check_arguments_on_the_host():
    L = lib8.lib()
    a = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert L.w8a8_quantize_activations(None, a, a, 16, 4096, None) == 1
    assert L.w8a8_quantize_activations(a, a, a, 0, 4096, None) == 1
    assert L.w8a8_quantize_activations(a, a, a, 16, 4100, None) == 2
    assert L.w8a8_quantize_activations(odd, a, a, 16, 4096, None) == 3
    assert L.q8_0_quantize(a, a, a, 4010, 320, None) == 2
    assert L.q8_0_quantize(a, odd, a, 4096, 320, None) == 3
    assert L.q8_0_split_from_blocks(a, odd, a, 4096, 320, None) == 3
    assert L.q8_0_split_from_blocks(ctypes.c_void_p((1 << 20) + 1), a, a, 4096, 320, None) == 3
    assert L.q8_0_blocks_from_split(a, a, a, 4096, 0, None) == 1


def test_rms_read_checks_its_arguments_on_the_host():
    L = lib8.lib()
    a = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    qws = lib8.q8_0_workspace_bytes(6, 4096, 320)
    f = ctypes.c_float
    assert L.q8_0_gemv_rms(a, None, f(1e-6), a, a, a, 6, 4096, 320, 0, a, qws, None) == 1      # no gamma
    assert L.q8_0_gemv_rms(a, a, f(-1.0), a, a, a, 6, 4096, 320, 0, a, qws, None) == 1        # eps < 0
    assert L.q8_0_gemv_rms(a, a, f(float("nan")), a, a, a, 6, 4096, 320, 0, a, qws, None) == 1
    assert L.q8_0_gemv_rms(a, a, f(float("inf")), a, a, a, 6, 4096, 320, 0, a, qws, None) == 1
    assert L.q8_0_gemv_rms(a, odd, f(1e-6), a, a, a, 6, 4096, 320, 0, a, qws, None) == 3      # gamma misaligned
    assert L.q8_0_gemv_rms(a, a, f(1e-6), a, a, a, 6, 4096, 320, 0, a, qws - 1, None) == 4
    assert L.q8_0_gemv_rms(a, a, f(1e-6), a, a, a, 9, 4096, 320, 0, a, qws, None) == 1        # T > 8
    assert L.q8_0_gemv_rms(a, a, f(1e-6), a, a, a, 6, 4016, 320, 0, a, qws, None) == 2        # K % 32
    assert L.q8_0_gemv_rms(a, a, f(1e-6), a, a, a, 6, 4096, 320, 2, a, qws, None) == 1        # unknown flag


def test_calls_with_null_pointers_fail_before_any_launch():
    L = lib8.lib()
    null = ctypes.c_void_p(0)
    assert L.w8a8_gemm(null, null, null, null, null, 1, 512, 256, 0, 0, null, 0, null) == 1
    assert L.q8_0_gemv(null, null, null, null, 1, 512, 256, 0, null, 0, null) == 1
    assert L.w8a8_pack_weights(null, 512, 256, null, null, 0, null) == 1
    assert L.w8a8_workspace_init(null, 0, null) == 1


def test_misaligned_and_short_workspace_are_rejected_on_the_host():
    # Fake (never dereferenced) device addresses: the checks run before any launch.
    L = lib8.lib()
    a = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    ws_need = lib8.w8a8_workspace_bytes(16, 4096, 1536)
    assert L.w8a8_gemm(odd, a, a, a, a, 16, 4096, 1536, 0, 0, a, ws_need, None) == 3
    assert L.w8a8_gemm(a, a, odd, a, a, 16, 4096, 1536, 0, 0, a, ws_need, None) == 3
    assert L.w8a8_gemm(a, a, a, a, a, 16, 4096, 1536, 0, 0, a, ws_need - 1, None) == 4
    assert L.w8a8_gemm(a, a, a, a, a, 16, 4096, 1536, 0, 4, a, ws_need, None) == 1      # unknown flag
    qws = lib8.q8_0_workspace_bytes(6, 4096, 320)
    assert L.q8_0_gemv(odd, a, a, a, 6, 4096, 320, 0, a, qws, None) == 3
    assert L.q8_0_gemv(a, a, a, a, 6, 4096, 320, 0, a, qws - 1, None) == 4
    assert L.q8_0_gemv(a, a, a, a, 9, 4096, 320, 0, a, qws, None) == 1
    assert L.q8_0_gemv(a, a, a, a, 6, 4016, 320, 0, a, qws, None) == 2      # K % 32 != 0


# ------------------------------------------------------------------------------------------
# CPU emulation of the GEMM kernel's fragment bookkeeping (documented layout + PTX fragments)
# ------------------------------------------------------------------------------------------

def _frag_a(words):
    """mma.m16n8k16 A fragment of one lane from the kernel's conversion of 4 packed words.

    Each word's bytes (0,2) form one register and bytes (1,3) another (as
    offset_bytes_to_subnormal_pairs): a byte b of the packed weight (offset binary, b = w + 128)
    becomes the fp16 subnormal b * 2^-24, so the fragment carries the unsigned bytes themselves, in
    units of 2^-24.  Registers a0..a3 of one k16 step are (row g, slots 2c,2c+1), (row g+8, ...),
    (row g, slots 2c+8,2c+9), (row g+8, ...) per the PTX fragment layout; the kernel feeds
    {lo(w_row_g), lo(w_row_g8), hi(w_row_g), hi(w_row_g8)}."""
    def lohi(w):
        b = [(w >> (8 * i)) & 0xFF for i in range(4)]
        return (b[0], b[2]), (b[1], b[3])
    return [lohi(w) for w in words]


def test_emulated_fragment_path_reproduces_x_at_w():
    """The MMA sums (w + 128) * x in units of 2^-24; the activation sums that the lanes gather
    with dp4a (each lane 8 bytes of row 8j + g per slab, the four lanes of a row 32 k) take
    128 * sum_k x off once, which leaves exactly x @ W."""
    M, K, N = 12, 64, 128
    x, _, W, _ = synth.w8a8_inputs(M, K, N, seed=21)
    packed = oracle.w8a8_pack(W)
    KB = K // 32
    NT8 = (M + 7) // 8
    acc = np.zeros((N, 8 * NT8), dtype=np.int64)         # rows n, columns m (out^T)
    xp = np.zeros((8 * NT8, K), dtype=np.int64)
    xp[:M] = x
    for t in range(N // 64):
        for kb in range(KB):
            for s in range(4):
                base = (((t * KB + kb) * 4 + s) * 32) * 16
                for lane in range(32):
                    g, c = lane // 4, lane % 4
                    wbytes = packed[base + lane * 16: base + lane * 16 + 16]
                    words = [int.from_bytes(bytes(wbytes[4 * i:4 * i + 4]), "little") for i in range(4)]
                    frag = _frag_a(words)
                    for step in range(2):
                        (r0l, r0h), (r1l, r1h) = frag[2 * step], frag[2 * step + 1]
                        # slot -> k mapping used for both operands: slots (2c, 2c+1) <- k 8c+4step+{0,2};
                        # slots (2c+8, 2c+9) <- k 8c+4step+{1,3}
                        k0 = 32 * kb + 8 * c + 4 * step
                        a_rows = {g: {2 * c: r0l[0], 2 * c + 1: r0l[1], 2 * c + 8: r0h[0], 2 * c + 9: r0h[1]},
                                  g + 8: {2 * c: r1l[0], 2 * c + 1: r1l[1], 2 * c + 8: r1h[0], 2 * c + 9: r1h[1]}}
                        slot_k = {2 * c: k0 + 0, 2 * c + 1: k0 + 2, 2 * c + 8: k0 + 1, 2 * c + 9: k0 + 3}
                        for row, slots in a_rows.items():
                            n = 64 * t + 16 * s + row
                            for slot, a in slots.items():
                                acc[n, :] += a * xp[:, slot_k[slot]]
    # the lanes' activation sums: lane (g, c) adds bytes k = 32 kb + 8c ... 8c + 7 of row 8j + g
    xsum = np.zeros(8 * NT8, dtype=np.int64)
    for kb in range(KB):
        for g in range(8):
            for c in range(4):
                for j in range(NT8):
                    xsum[8 * j + g] += int(xp[8 * j + g, 32 * kb + 8 * c: 32 * kb + 8 * c + 8].sum())
    assert np.array_equal(xsum, xp.sum(axis=1))
    acc -= 128 * xsum[None, :]
    ref = oracle.w8a8_acc(x, W)
    np.testing.assert_array_equal(acc[:N, :M].T, ref)


def test_workspace_query_covers_every_smaller_m_across_shapes():
    # The size query's promise: a workspace of w8a8_workspace_bytes(M_max, K, N, blocks) bytes
    # serves every call with M <= M_max, whichever arm and kernel variant that M runs.
    rng = np.random.default_rng(17)
    shapes = [(32, 8), (96, 136), (512, 256), (4096, 1536), (4096, 2560), (12288, 4096), (4096, 24576)]
    for K, N in shapes:
        for M_max in (1, 8, 17, 32, 33, 64, 65, 100, 128):
            for blocks in (0, 1, int(rng.integers(2, 64))):
                big = lib8.w8a8_workspace_bytes(M_max, K, N, blocks)
                if big == 0:      # some M <= M_max has no plan with this many CTAs
                    continue
                for M in range(1, M_max + 1):
                    assert lib8.w8a8_plan(M, K, N, blocks)["workspace_bytes"] <= big, (M, M_max, K, N, blocks)
