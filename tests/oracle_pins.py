"""Pins for the CPU oracle: checks against what the page and plain mathematics fix.

Each pin takes the tag of an oracle build so the mutation test can run the same
battery against deliberately broken copies.  Sources are "MNN LLM inference on
the SpacemiT K3": section 3 eqs. (1)-(3) and section 4 (prefill data flow).
No pin re-types the oracle's own formula: each compares it with a closed form,
a hand-derived fixture, an invariant, or a differently-structured computation
(dense fp64 dequantise-then-matmul, exact integer identities).
"""
import numpy as np

import oracle
from golden_cases import linear_hand_cases, quant_tie_rule
from w4a8_block_quantized_gb300 import synth

BLOCK = 64


def pin_half_decode(tag):
    """The oracle's fp16 decoder agrees with numpy's IEEE binary16 on all 65536 patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.half_to_double(bits, tag=tag)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_quant_golden(tag):
    """Hand-derived tie-rule fixture (section 4 step 1; round half away from zero)."""
    x, a_q, s_a, rs = quant_tie_rule()
    ga, gs, gr = oracle.quant_pack(x, tag=tag)
    assert np.array_equal(gs, s_a), (gs, s_a)
    assert np.array_equal(ga, a_q)
    assert np.array_equal(gr, rs)


def pin_quant_closed_forms(tag):
    """Single-spike rows: x = v e_j gives s_a = |v|/127 (fp32) and a_q = sign(v) 127 e_j."""
    K = 256
    vals = [3.7, -0.001, 1e-20, -5e4, 127.0, 1.0]
    x = np.zeros((len(vals), K), np.float32)
    js = [0, 63, 64, 100, 200, 255]
    for r, (v, j) in enumerate(zip(vals, js)):
        x[r, j] = np.float32(v)
    a_q, s_a, rs = oracle.quant_pack(x, tag=tag)
    for r, (v, j) in enumerate(zip(vals, js)):
        assert s_a[r] == np.float32(abs(np.float32(v))) / np.float32(127.0)
        exp = np.zeros(K, np.int8)
        exp[j] = 127 if v > 0 else -127
        assert np.array_equal(a_q[r], exp)
        exp_rs = np.zeros(K // BLOCK, np.int32)
        exp_rs[j // BLOCK] = exp[j]
        assert np.array_equal(rs[r], exp_rs)


def pin_quant_tiny_scales(tag):
    """Rows whose scale sits in or below the subnormal range, in units u = 2^-149 (the
    smallest fp32 subnormal), where every step is exact integer arithmetic on multiples of u:
      - absmax 7u or 63u: absmax / 127 < u / 2 rounds to s_a = 0, and the row quantizes like
        a zero row (codes 0, row sums 0);
      - absmax 64u or 143u: absmax / 127 lies in (u/2, 3u/2), so s_a = u and each code is the
        element's multiple of u, clamped to +-127 (143 -> 127);
      - absmax 1e-38 and 1e-36 (s_a subnormal with 16 and 23 significant bits): a single
        spike still maps to +-127 and s_a = RN(|v| / 127)."""
    u = np.float32(2.0 ** -149)
    K = 128
    x = np.zeros((6, K), np.float32)
    x[0, [3, 70]] = [7 * u, -5 * u]
    x[1, [0, 1, 127]] = [-63 * u, 62 * u, u]
    x[2, [5, 6, 64]] = [64 * u, -64 * u, 3 * u]
    x[3, [0, 9, 10, 100]] = [143 * u, 71 * u, -100 * u, -u]
    x[4, 17] = np.float32(1e-38)
    x[5, 90] = np.float32(-1e-36)
    a_q, s_a, rs = oracle.quant_pack(x, tag=tag)
    assert s_a[0] == 0 and s_a[1] == 0
    assert not a_q[:2].any() and not rs[:2].any()
    assert s_a[2] == u and s_a[3] == u
    e2 = np.zeros(K, np.int8)
    e2[[5, 6, 64]] = [64, -64, 3]
    e3 = np.zeros(K, np.int8)
    e3[[0, 9, 10, 100]] = [127, 71, -100, -1]
    assert np.array_equal(a_q[2], e2) and np.array_equal(a_q[3], e3)
    assert np.array_equal(rs[2], [0, 3]) and np.array_equal(rs[3], [127 + 71 - 100, -1])
    for r, j, v in ((4, 17, 1e-38), (5, 90, -1e-36)):
        assert s_a[r] == np.float32(abs(np.float32(v))) / np.float32(127.0)
        assert 0 < s_a[r] < np.float32(2.0 ** -126)
        exp = np.zeros(K, np.int8)
        exp[j] = 127 if v > 0 else -127
        assert np.array_equal(a_q[r], exp)


def pin_quant_invariants(tag):
    """On seeded workload-style rows: codes within +-127, the absmax element maps to
    +-127, the reconstruction error is at most half a step, and the per-64 sums are
    the block sums of the codes."""
    d = synth.random_small(64, 1024, 8, seed=3, outlier=20.0)
    x = d["x"]
    a_q, s_a, rs = oracle.quant_pack(x, tag=tag)
    assert np.abs(a_q.astype(np.int32)).max() <= 127
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s_a, (amax / np.float32(127.0)).astype(np.float32))
    for m in range(x.shape[0]):
        j = int(np.argmax(np.abs(x[m])))
        assert abs(int(a_q[m, j])) == 127
    err = np.abs(a_q.astype(np.float64) * s_a[:, None].astype(np.float64) - x.astype(np.float64))
    assert np.all(err <= s_a[:, None].astype(np.float64) * (0.5 + 1e-6))
    blocks = a_q.astype(np.int64).reshape(x.shape[0], -1, BLOCK).sum(axis=2)
    assert np.array_equal(rs.astype(np.int64), blocks)


def pin_nibble_identity(tag):
    """Section 3 eq. (3) over all 256 int8 values, and the oracle's nibble-split path
    equals its direct path on every int8 value (including -128) and every u4 code."""
    a = np.arange(-128, 128, dtype=np.int32)
    assert np.array_equal(16 * (a >> 4) + (a & 0x0F), a)
    assert (a >> 4).min() == -8 and (a >> 4).max() == 7
    # every (a, q) pair appears: 256 activation values x 16 codes, K = 4096 = 64 blocks
    K = 4096
    a_q = np.tile(np.arange(-128, 128, dtype=np.int16), 16).astype(np.int8)[None, :]
    q = np.repeat(np.arange(16, dtype=np.uint8), 256)[None, :]
    wq = synth.pack_u4(q)
    direct = oracle.block_acc(a_q, wq, 1, tag=tag)
    nib = oracle.block_acc(a_q, wq, 1, nibble=True, tag=tag)
    assert np.array_equal(direct, nib)
    ref = (a_q.astype(np.int64) * q.astype(np.int64)).reshape(1, 1, K // BLOCK, BLOCK).sum(-1)
    assert np.array_equal(direct.astype(np.int64), ref)


def pin_block_acc_matches_codes(tag):
    """Per-block accumulators equal an int64 matmul of a_q with the generator's own
    codes q (not the packed bytes), block by block, on a window with ragged edges."""
    rng = np.random.default_rng(5)
    M, N, K = 9, 7, 192
    a_q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    wq = synth.pack_u4(q)
    acc = oracle.block_acc(a_q, wq, N, m0=2, mc=5, n0=1, nc=6, tag=tag)
    A = a_q.astype(np.int64).reshape(M, K // BLOCK, BLOCK)
    Q = q.astype(np.int64).reshape(N, K // BLOCK, BLOCK)
    ref = np.einsum("mbi,nbi->mnb", A, Q)[2:7, 1:7]
    assert np.array_equal(acc.astype(np.int64), ref)
    nib = oracle.block_acc(a_q, wq, N, m0=2, mc=5, n0=1, nc=6, nibble=True, tag=tag)
    assert np.array_equal(nib.astype(np.int64), ref)


def pin_zero_point_decomposition(tag):
    """Section 3 eq. (2) in exact integers: with fp16 z in [6, 9], 256 z is an integer,
    so sum_i a_i (256 q_i - 256 z) must equal 256 acc - (256 z) rs exactly, where acc
    and rs come from the oracle and the left side is formed directly."""
    d = synth.random_small(16, 512, 12, seed=11)
    a_q, s_a, rs = oracle.quant_pack(d["x"], tag=tag)
    acc = oracle.block_acc(a_q, d["wq"], 12, tag=tag).astype(np.int64)
    z256 = d["z_w"].astype(np.float64) * 256.0
    assert np.all(z256 == np.round(z256))
    z256 = z256.astype(np.int64)                                  # [N, B]
    A = a_q.astype(np.int64).reshape(16, -1, BLOCK)               # [M, B, 64]
    Q = d["q"].astype(np.int64).reshape(12, -1, BLOCK)            # [N, B, 64]
    lhs = np.einsum("mbi,nbi->mnb", A, 256 * Q) - np.einsum("mbi,nb->mnb", A, z256)
    rhs = 256 * acc - z256[None, :, :] * rs.astype(np.int64)[:, None, :]
    assert np.array_equal(lhs, rhs)


def _dense_fp64(a_q, s_a, q, s_w, z_w, bias):
    """Dequantise then matmul in fp64: w = s_w (q - z) (eq. (1)), a = s_a a_q."""
    nb = q.shape[1] // BLOCK
    sw = np.repeat(s_w.astype(np.float64), BLOCK, axis=1)
    zw = np.repeat(z_w.astype(np.float64), BLOCK, axis=1)
    w = sw * (q.astype(np.float64) - zw)
    a = s_a.astype(np.float64)[:, None] * a_q.astype(np.float64)
    y = a @ w.T
    assert w.shape[1] == nb * BLOCK
    if bias is not None:
        y = y + bias.astype(np.float64)[None, :]
    return y


def pin_bruteforce_fp64(tag):
    """Tiny shapes: the oracle's block-wise output equals dense fp64 dequantise-then-
    matmul to 1e-9 relative (of the larger of |y| and the sum of block magnitudes)."""
    seed = 100
    for M in (1, 3, 8):
        for N in (1, 2, 5, 8):
            for K in (64, 128, 192):
                seed += 1
                d = synth.random_small(M, K, N, seed=seed, bias=(seed % 2 == 0))
                a_q, s_a, rs = oracle.quant_pack(d["x"], tag=tag)
                y, bound = oracle.linear(a_q, s_a, rs, d["wq"], d["s_w"], d["z_w"], d["bias"], tag=tag)
                ref = _dense_fp64(a_q, s_a, d["q"], d["s_w"], d["z_w"], d["bias"])
                scale = np.maximum(np.abs(ref), bound) + 1e-300
                assert np.all(np.abs(y - ref) <= 1e-9 * scale), (M, N, K)
    # one bigger seeded case in the shape of the tiny workload
    d = synth.random_small(32, 1024, 64, seed=7, bias=True)
    a_q, s_a, rs = oracle.quant_pack(d["x"], tag=tag)
    y, bound = oracle.linear(a_q, s_a, rs, d["wq"], d["s_w"], d["z_w"], d["bias"], tag=tag)
    ref = _dense_fp64(a_q, s_a, d["q"], d["s_w"], d["z_w"], d["bias"])
    assert np.all(np.abs(y - ref) <= 1e-9 * (np.maximum(np.abs(ref), bound) + 1e-300))


def pin_linear_golden(tag):
    """Hand-derived outputs (section 3 eq. (2) per block, bias in the epilogue)."""
    for c in linear_hand_cases():
        y, _, _, _, _ = oracle.prefill_linear(c["x"], c["wq"], c["s_w"], c["z_w"], c["bias"], tag=tag)
        assert np.array_equal(y, c["y"]), (c["name"], y, c["y"])


def pin_special_cases(tag):
    """Degenerate cases with exact answers: q == z everywhere gives y = bias; an all-zero
    row gives y = bias; a spike row x = v e_j gives y = s_a 127 sign(v) s_w (q_j - z) + bias."""
    rng = np.random.default_rng(9)
    M, N, K = 4, 6, 256
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[1] = 0.0
    bias = rng.standard_normal(N).astype(np.float32)
    c = 9
    q = np.full((N, K), c, np.uint8)
    s_w = rng.uniform(0.005, 0.02, (N, K // BLOCK)).astype(np.float16)
    z_w = np.full((N, K // BLOCK), c, np.float16)
    y, _, _, _, _ = oracle.prefill_linear(x, synth.pack_u4(q), s_w, z_w, bias, tag=tag)
    assert np.array_equal(y, np.broadcast_to(bias.astype(np.float64), (M, N)))
    # zero row with random weights
    q2 = rng.integers(0, 16, (N, K)).astype(np.uint8)
    z2 = rng.uniform(6, 9, (N, K // BLOCK)).astype(np.float16)
    y2, _, _, _, _ = oracle.prefill_linear(x, synth.pack_u4(q2), s_w, z2, bias, tag=tag)
    assert np.array_equal(y2[1], bias.astype(np.float64))
    # spike row
    j, v = 77, np.float32(-2.75)
    xs = np.zeros((1, K), np.float32)
    xs[0, j] = v
    y3, _, a_q, s_a, _ = oracle.prefill_linear(xs, synth.pack_u4(q2), s_w, z2, None, tag=tag)
    b = j // BLOCK
    exp = (float(s_a[0]) * -127.0 * s_w[:, b].astype(np.float64)
           * (q2[:, j].astype(np.float64) - z2[:, b].astype(np.float64)))
    assert np.allclose(y3[0], exp, rtol=1e-13, atol=0.0)


def pin_epilogue_store(tag):
    """The epilogue's store (section 4 step 3: clamp, then the output type).  bf16 rounding
    against hand-worked values (ties to the even significand) and, on random values, against
    the nearer of the two bf16 neighbours built from their bit patterns (numpy's float32 view
    of a 16-bit pattern shifted left by 16); the clamp against its closed form; fp32 against
    numpy's own float32 cast."""
    r = oracle.bf16_round
    assert r(1.0) == 1.0 and r(-3.0) == -3.0 and r(0.0) == 0.0
    assert r(1.0 + 2.0 ** -8) == 1.0                        # tie, even neighbour below
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6        # tie, even neighbour above
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert r(-(1.0 + 2.0 ** -8 + 2.0 ** -20)) == -(1.0 + 2.0 ** -7)
    assert r(1.0 / 3.0) == 0.333984375                      # 0x3EAB
    assert r(255.5) == 256.0 and r(254.5) == 254.0          # step 2 in [128, 256): 255.5 -> 256
    rng = np.random.default_rng(17)
    v = rng.standard_normal(4000) * np.exp2(rng.integers(-30, 30, 4000))
    got = r(v)
    # neighbours from bit patterns: truncate the float32 of v toward zero to a bf16 pattern
    f32 = v.astype(np.float32)
    hi16 = (f32.view(np.uint32) >> 16).astype(np.uint32)
    lo = (hi16 << 16).view(np.float32).astype(np.float64)
    nxt = ((hi16 + 1) << 16).view(np.float32).astype(np.float64)
    for val, a, b, g in zip(v, lo, nxt, got):
        lo_, hi_ = min(a, b), max(a, b)
        if not (lo_ <= val <= hi_):                         # the float32 cast crossed a neighbour
            continue
        da, db = abs(val - lo_), abs(hi_ - val)
        assert g in (lo_, hi_)
        if da != db:
            assert g == (lo_ if da < db else hi_)
    y = np.array([-2.0, -0.5, 0.1, 0.75, 3.0])
    assert np.array_equal(oracle.epilogue(y, -0.5, 0.75, "f32"), [-0.5, -0.5, np.float64(np.float32(0.1)), 0.75, 0.75])
    assert np.array_equal(oracle.epilogue(y, out_dtype="f32"), y.astype(np.float32).astype(np.float64))
    assert np.array_equal(oracle.epilogue(y, -1.0, 1.0, "bf16"), r(np.clip(y, -1.0, 1.0)))


ALL_PINS = [
    pin_half_decode,
    pin_quant_golden,
    pin_quant_closed_forms,
    pin_quant_tiny_scales,
    pin_quant_invariants,
    pin_nibble_identity,
    pin_block_acc_matches_codes,
    pin_zero_point_decomposition,
    pin_bruteforce_fp64,
    pin_linear_golden,
    pin_special_cases,
    pin_epilogue_store,
]
