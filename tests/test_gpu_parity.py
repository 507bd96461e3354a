"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same
seeded inputs.  Integer stages bit-exact; fp32 output within the stated tolerance."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_y, dev, inputs_to_dev, to_dev
from w4a8_block_quantized_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a8_block_quantized_gb300 import binding, build
    build.build()
    binding.load()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    assert binding.sync_status() == 0


def B():
    from w4a8_block_quantized_gb300 import binding
    return binding


# ------------------------------------------------------------------ pre-pass
@pytest.mark.parametrize("M,K", [(1, 64), (3, 128), (128, 1024), (129, 1024), (77, 2048), (40, 4096),
                                 (9, 6144), (33, 14336), (5, 16384), (3, 20480)])
def test_quant_pack_bitexact(M, K):
    d = synth.random_small(M, K, 1, seed=M * 7 + K)
    x = d["x"]
    a_q, s_a, rs = B().quant_pack(to_dev(x))
    ra, rsa, rrs = oracle.quant_pack(x)
    assert np.array_equal(s_a.cpu().numpy(), rsa)
    assert np.array_equal(a_q.cpu().numpy(), ra)
    assert np.array_equal(rs.cpu().numpy(), rrs)


def test_quant_pack_golden_and_degenerate_rows():
    from golden_cases import quant_tie_rule
    x, a_q, s_a, rs = quant_tie_rule()
    ga, gs, gr = B().quant_pack(to_dev(x))
    assert np.array_equal(gs.cpu().numpy(), s_a)
    assert np.array_equal(ga.cpu().numpy(), a_q)
    assert np.array_equal(gr.cpu().numpy(), rs)


def _tiny_scale_rows(K, rng):
    """Rows whose scale is subnormal without a finite reciprocal (absmax 1e-38, deep
    subnormal multiples of u = 2^-149 where |x / s| can pass 127), subnormal with one
    (1e-36), or rounds to 0 (absmax 1e-44 and 63u), next to an ordinary row."""
    u = np.float32(2.0 ** -149)
    rows = [rng.standard_normal(K) * np.float32(1e-38 / 4), rng.standard_normal(K) * np.float32(1e-36 / 4),
            rng.integers(-143, 144, K) * u, rng.integers(-63, 64, K) * u, np.full(K, np.float32(1e-44)),
            rng.standard_normal(K)]
    x = np.stack([np.asarray(r, np.float32) for r in rows])
    x[0, 1] = np.float32(1e-38)
    x[2, 2] = 143 * u
    return x


@pytest.mark.parametrize("K", [1024, 4096, 20480])
def test_quant_tiny_scales_bitexact(K):
    """Scales in and below the subnormal range through the pre-pass (register-resident rows,
    the 512-thread rows and the two-pass long rows): codes, scales and row sums bit for bit;
    the fused call (operand records) within tolerance and equal to the separate calls."""
    rng = np.random.default_rng(K)
    # 16 rows, so that the linear takes the tensor-core form
    x = np.concatenate([_tiny_scale_rows(K, rng), rng.standard_normal((10, K)).astype(np.float32)])
    a_q, s_a, rs = B().quant_pack(to_dev(x))
    ra, rsa, rrs = oracle.quant_pack(x)
    assert np.array_equal(s_a.cpu().numpy(), rsa)
    assert np.array_equal(a_q.cpu().numpy(), ra)
    assert np.array_equal(rs.cpu().numpy(), rrs)
    assert rsa[3] == 0 and rsa[4] == 0 and not ra[3:5].any()
    d = synth.random_small(x.shape[0], K, 100, seed=K, bias=True)
    d["x"] = x
    y_fused, y_sep = _run_both(d)
    y_ref, bound, _, _, _ = oracle.prefill_linear(x, d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_fused, y_ref, bound, f"tiny scales K={K}")
    assert torch.equal(y_fused, y_sep)


@pytest.mark.parametrize("K", [1024, 2048])
def test_decode_quantizer_tiny_scales(K):
    """The few-token kernel's own quantizer (M * K <= 16384) on the same rows: its outputs
    equal those of the pre-pass + kernel path, whose codes match the oracle bit for bit."""
    rng = np.random.default_rng(K + 1)
    x = _tiny_scale_rows(K, rng)
    d = synth.random_small(x.shape[0], K, 300, seed=K + 1, bias=True)
    d["x"] = x
    y_fused, y_sep = _run_both(d)
    assert B().prefill_workspace_bytes(x.shape[0], 300, K) == 0   # the kernel quantized itself
    y_ref, bound, _, _, _ = oracle.prefill_linear(x, d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_fused, y_ref, bound, f"decode tiny scales K={K}")
    assert torch.equal(y_fused, y_sep)


# ------------------------------------------------------------------ block accumulators
def _acc_case(a_q, q, m0=0, mc=None, n0=0, nc=None):
    N = q.shape[0]
    wq = synth.pack_u4(q)
    got = B().debug_block_acc(to_dev(a_q), to_dev(wq), N, m0, mc, n0, nc).cpu().numpy()
    ref = oracle.block_acc(a_q, wq, N, m0, mc, n0, nc)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} accumulators differ"


def test_block_acc_exact_extremes():
    """Largest magnitudes and cancellation patterns the int8 x u4 block sums can take."""
    K, M, N = 512, 130, 70
    a = np.zeros((M, K), np.int8)
    q = np.zeros((N, K), np.uint8)
    a[0] = 127
    a[1] = -127
    a[2] = -128
    a[3, 0::2], a[3, 1::2] = 127, -127           # alternating signs
    a[4] = 1
    a[4, ::64] = 127                              # one large term + many small ones
    a[5] = -1
    a[5, 5::64] = -128
    rng = np.random.default_rng(0)
    a[6:] = rng.integers(-128, 128, size=(M - 6, K)).astype(np.int8)
    q[0] = 15
    q[1, 0::2], q[1, 1::2] = 15, 0
    q[2] = 1
    q[3, ::3] = 15
    q[4:] = rng.integers(0, 16, size=(N - 4, K)).astype(np.uint8)
    _acc_case(a, q)


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (1, 64, 64), (127, 63, 128), (128, 256, 192), (129, 257, 256),
                                   (300, 200, 1024), (64, 1000, 128), (200, 512, 2048)])
def test_block_acc_random(M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K)
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    _acc_case(a, q)


def test_block_acc_windows():
    rng = np.random.default_rng(3)
    M, N, K = 400, 700, 256
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    _acc_case(a, q, m0=5, mc=131, n0=3, nc=300)
    _acc_case(a, q, m0=399, mc=1, n0=699, nc=1)
    _acc_case(a, q, m0=128, mc=200, n0=256, nc=444)


@pytest.mark.parametrize("M,N,K", [(4096, 129, 256), (4097, 200, 128), (4352, 300, 192), (4100, 1, 64)])
def test_block_acc_wide_contraction(M, N, K):
    """M >= 4096 runs the 256-token kernel (N = 256 MMAs): its per-block accumulators, bit for
    bit, over whole problems with ragged token tails (4097 and 4100 leave 1 and 4 rows in the
    last tile; 4352 = 17 full tiles) and ragged or single weight rows."""
    rng = np.random.default_rng(M + 7 * N + K)
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    a[:3] = np.array([127, -127, -128], np.int8)[:, None]   # the extremes, in whole rows
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    q[0] = 15
    _acc_case(a, q)


def test_block_acc_wide_windows():
    """Windows of an 8192-token problem (the 256-token kernel): crossing token-tile and
    weight-tile boundaries, the last rows and columns, a single accumulator."""
    rng = np.random.default_rng(17)
    M, N, K = 8192, 700, 1024
    a = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    _acc_case(a, q, m0=3900, mc=600, n0=100, nc=300)
    _acc_case(a, q, m0=8000, mc=192, n0=572, nc=128)
    _acc_case(a, q, m0=8191, mc=1, n0=699, nc=1)


# ------------------------------------------------------------------ full linear
def _run_both(d):
    g = inputs_to_dev(d)
    y_fused = B().prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    a_q, s_a, rs = B().quant_pack(g["x"])
    y_sep = B().linear(a_q, s_a, rs, g["wq"], g["s_w"], g["z_w"], g["bias"])
    return y_fused, y_sep


@pytest.mark.parametrize("M,K,N,bias", [(1, 64, 1, False), (1, 64, 16, True), (7, 128, 33, True),
                                        (128, 1024, 256, False), (129, 192, 257, True), (255, 1024, 130, True),
                                        (300, 2048, 513, False), (64, 64, 4000, True), (513, 4096, 64, False),
                                        (17, 16384, 100, True), (9, 20480, 70, False), (256, 1024, 3000, True)])
def test_linear_small_shapes(M, K, N, bias):
    """The fused call against the oracle and against w4a8_quant_pack + w4a8_linear.  Rows of
    1024 or less take four, two or one warps per row in the pre-pass, whichever keeps its launch
    in one wave: (128, 1024) four, (256, 1024, 3000) two (its weight job takes 192 CTAs)."""
    d = synth.random_small(M, K, N, seed=M + K + N, bias=bias)
    y_fused, y_sep = _run_both(d)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_fused, y_ref, bound, f"fused {M}x{K}->{N}")
    assert torch.equal(y_fused, y_sep), "fused and separate calls differ"


@pytest.mark.parametrize("M,K,N,bias", [(4096, 512, 256, True), (4100, 1024, 300, False), (4352, 128, 1000, True),
                                        (4097, 2048, 129, True)])
def test_linear_wide_token_tiles(M, K, N, bias):
    """M >= 4096 takes the 256-token records and the N = 256 contraction: ragged token and
    weight tails, every output against the oracle, the fused call against the separate and
    the prepared calls bit for bit."""
    d = synth.random_small(M, K, N, seed=M + 3 * K + N, bias=bias)
    y_fused, y_sep = _run_both(d)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_fused, y_ref, bound, f"wide {M}x{K}->{N}")
    assert torch.equal(y_fused, y_sep), "fused and separate calls differ"
    g = inputs_to_dev(d)
    act = B().prepare_activations(g["x"])
    pw = B().prepare_weights(g["wq"], g["s_w"], g["z_w"])
    assert torch.equal(B().linear_prepared(act, pw, M, N, K, bias=g["bias"]), y_fused), "prepared call differs"


@pytest.mark.parametrize("key", ["c0", "c1", "c2", "c3"])
def test_workloads_full(key):
    _, specs = synth.workload(key)
    for spec in specs:
        d = synth.make_linear(spec)
        y_fused, y_sep = _run_both(d)
        y_ref, bound, a_q, s_a, rs = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
        check_y(y_fused, y_ref, bound, f"{key}/{spec.name}")
        assert torch.equal(y_fused, y_sep)
        ga, gs, gr = B().quant_pack(to_dev(d["x"]))
        assert np.array_equal(ga.cpu().numpy(), a_q) and np.array_equal(gs.cpu().numpy(), s_a)
        assert np.array_equal(gr.cpu().numpy(), rs)


def test_workload_c4_sampled():
    """7B-class sizes in the benchmark's launch configuration: codes, scales and row sums
    bit-exact on every row; outputs on 48 sampled rows; accumulators on a window."""
    _, specs = synth.workload("c4")
    for spec in specs:
        d = synth.make_linear(spec)
        g = inputs_to_dev(d)
        ws = B().workspace(B().prefill_workspace_bytes(spec.M, spec.N, spec.K), dev())
        y = torch.full((spec.M, spec.N), float("nan"), device=dev())
        B().prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y, ws=ws)
        rows = np.unique(np.concatenate([np.linspace(0, spec.M - 1, 40).astype(np.int64),
                                         [127, 128, 4095, 4096, 8063, 8064, 8190, 8191]]))
        y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"], rows=rows)
        check_y(y[torch.from_numpy(rows).to(dev())], y_ref, bound, f"c4/{spec.name}")
        assert not torch.isnan(y).any(), "unwritten outputs"
        a_q, s_a, rs = B().quant_pack(g["x"])
        ra, rsa, rrs = oracle.quant_pack(d["x"])
        assert np.array_equal(a_q.cpu().numpy(), ra)
        assert np.array_equal(s_a.cpu().numpy(), rsa)
        assert np.array_equal(rs.cpu().numpy(), rrs)
        # the 256-token contraction the linear ran, on windows across tiles and at both ends
        for m0, mc, n0, nc in ((4000, 160, spec.N - 300, 300), (0, 256, 0, 128), (8060, 132, 200, 260)):
            got = B().debug_block_acc(a_q, g["wq"], spec.N, m0, mc, n0, nc).cpu().numpy()
            ref = oracle.block_acc(ra, d["wq"], spec.N, m0, mc, n0, nc)
            assert np.array_equal(got, ref), f"c4/{spec.name} window {(m0, mc, n0, nc)}"

        del g, y, ws
        torch.cuda.empty_cache()


# ------------------------------------------------------------------ edge cases
def test_hand_cases_exact():
    from golden_cases import linear_hand_cases
    for c in linear_hand_cases():
        g = inputs_to_dev(c)
        y = B().prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"]).cpu().numpy()
        assert np.array_equal(y.astype(np.float64), c["y"]), (c["name"], y, c["y"])


def test_degenerate_inputs():
    rng = np.random.default_rng(11)
    M, N, K = 130, 70, 256
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0] = 0.0                      # zero row
    x[1] = 0.0
    x[1, 17] = -3.5                 # single spike
    x[2] = 1.0                      # constant row: every code 127
    x[3] = 1e-30                    # tiny values
    x[4] = 3e30                     # huge values
    c = 9
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    q[:5] = c                       # q == z exactly for the first 5 outputs
    s_w = rng.uniform(0.005, 0.02, (N, K // 64)).astype(np.float16)
    z_w = rng.uniform(6, 9, (N, K // 64)).astype(np.float16)
    z_w[:5] = c
    bias = rng.standard_normal(N).astype(np.float32)
    d = dict(x=x, wq=synth.pack_u4(q), s_w=s_w, z_w=z_w, bias=bias)
    y_fused, y_sep = _run_both(d)
    y_ref, bound, _, _, _ = oracle.prefill_linear(x, d["wq"], s_w, z_w, bias)
    check_y(y_fused, y_ref, bound, "degenerate")
    y = y_fused.cpu().numpy()
    assert np.array_equal(y[0], bias)                      # zero row -> bias
    assert np.array_equal(y[:, :5], np.broadcast_to(bias[:5], (M, 5)))  # q == z -> bias exactly
    assert torch.equal(y_fused, y_sep)


def test_empty_and_invalid():
    b = B()
    x = torch.zeros((0, 128), device=dev())
    a_q, s_a, rs = b.quant_pack(x)
    assert a_q.shape == (0, 128)
    wq = torch.zeros((16, 64), dtype=torch.uint8, device=dev())
    sw = torch.ones((16, 2), dtype=torch.float16, device=dev())
    y = b.prefill_linear(x, wq, sw, sw)
    assert y.shape == (0, 16)
    with pytest.raises(b.W4A8Error) as e:
        b.quant_pack(torch.zeros((4, 96), device=dev()))
    assert e.value.status == b.W4A8_ERR_SHAPE
    flat = torch.zeros(4 * 128 + 1, device=dev())
    with pytest.raises(b.W4A8Error) as e:
        b.quant_pack(flat[1:].view(4, 128))                 # contiguous, base off by 4 bytes
    assert e.value.status in (b.W4A8_ERR_ALIGN,)
    assert b.sync_status() == 0


def test_deterministic_and_fully_written():
    d = synth.random_small(300, 1024, 700, seed=5, bias=True)
    g = inputs_to_dev(d)
    y1 = torch.full((300, 700), float("nan"), device=dev())
    y2 = torch.full((300, 700), float("nan"), device=dev())
    B().prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y1)
    B().prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y2)
    assert not torch.isnan(y1).any()
    assert torch.equal(y1, y2)


def test_bounded_wait_times_out_and_reports():
    b = B()
    assert b.sync_status() == 0
    b.selftest_wait_timeout(20000)                          # 20 ms limit on a barrier nobody completes
    assert b.sync_status() == b.W4A8_ERR_TIMEOUT
    assert b.sync_status() == 0                             # status word cleared
    d = synth.random_small(64, 128, 64, seed=2)             # the context is still usable
    g = inputs_to_dev(d)
    y = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y, y_ref, bound, "after timeout")
    assert b.sync_status() == 0


def test_split_calls_equal_fused():
    """prepare_activations + prepare_weights + linear_prepared == prefill_linear, bit for bit;
    one prepared activation buffer serves several linears that read the same input."""
    b = B()
    M, K = 300, 2048
    d0 = synth.random_small(M, K, 512, seed=21, bias=True)
    x = to_dev(d0["x"])
    act = b.prepare_activations(x)
    for N, seed in ((512, 21), (130, 22), (1000, 23)):
        d = synth.random_small(M, K, N, seed=seed, bias=True)
        g = inputs_to_dev(d)
        pw = b.prepare_weights(g["wq"], g["s_w"], g["z_w"])
        y_split = b.linear_prepared(act, pw, M, N, K, bias=g["bias"])
        y_fused = b.prefill_linear(x, g["wq"], g["s_w"], g["z_w"], g["bias"])
        assert torch.equal(y_split, y_fused)
        y_ref, bound, _, _, _ = oracle.prefill_linear(d0["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
        check_y(y_split, y_ref, bound, f"split N={N}")


@pytest.mark.parametrize("M,K,N", [(512, 2048, 6144), (640, 1024, 4096), (1000, 256, 20480)])
def test_wide_tiles_below_4096_tokens(M, K, N):
    """Shapes whose 128-token tiles would take more waves of the 152 SMs (192, 160 and 1280
    tiles) run the one-call entry points on 256-token tiles (96, 96 and 640 tiles; 640 and 1000
    rows leave a half and a ragged last tile).  The prepared-operand calls keep 128-token records:
    without the K split both kernels sum every output in block order, so all of them agree bit
    for bit, and the per-block accumulators (the 256-token kernel's) are exact."""
    b = B()
    d = synth.random_small(M, K, N, seed=M + N, bias=True)
    g = inputs_to_dev(d)
    y_fused = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    act = b.prepare_activations(g["x"])
    pw = b.prepare_weights(g["wq"], g["s_w"], g["z_w"])
    assert torch.equal(b.linear_prepared(act, pw, M, N, K, bias=g["bias"]), y_fused)
    a_q, s_a, rs = b.quant_pack(g["x"])
    assert torch.equal(b.linear(a_q, s_a, rs, g["wq"], g["s_w"], g["z_w"], g["bias"]), y_fused)
    yh = b.prefill_linear_host(_pinned(d["x"]), g["wq"], g["s_w"], g["z_w"], g["bias"])
    torch.cuda.synchronize()
    assert torch.equal(yh, y_fused.cpu())
    rows = np.unique(np.linspace(0, M - 1, 48).astype(np.int64))
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"], rows=rows)
    check_y(y_fused[torch.from_numpy(rows).to(dev())], y_ref, bound, f"wide tiles {M}x{K}->{N}")
    a_np = a_q.cpu().numpy()
    for m0, mc, n0, nc in ((0, 300, 0, 200), (M - 140, 140, N - 130, 130)):
        got = b.debug_block_acc(a_q, g["wq"], N, m0, mc, n0, nc).cpu().numpy()
        ref = oracle.block_acc(a_np, d["wq"], N, m0, mc, n0, nc)
        assert np.array_equal(got, ref), f"{int((got != ref).sum())} accumulators differ"
    assert b.sync_status() == 0


@pytest.mark.parametrize("M,K,N", [(9, 64, 1), (300, 1024, 513), (512, 1088, 3072), (129, 6144, 130),
                                   (4100, 512, 300)])
def test_linear_act_equals_fused(M, K, N):
    """w4a8_linear_act (prepared activations, the packed weights as given) equals the fused
    call bit for bit -- below 4096 tokens the contraction expands the u4 codes in shared
    memory (one 64-block, odd K/64, a ragged weight tile), at 4100 the weights go through the
    workspace -- also right after the weights were rewritten by the previous kernel in the
    stream, and one prepared activation buffer serves two weight sets."""
    b = B()
    d = synth.random_small(M, K, N, seed=M + 5 * K + N, bias=True)
    g = inputs_to_dev(d)
    y_fused = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    act = b.prepare_activations(g["x"])
    assert torch.equal(b.linear_act(act, g["wq"], g["s_w"], g["z_w"], M, N, K, bias=g["bias"]), y_fused)
    wq2, sw2, zw2 = torch.zeros_like(g["wq"]), torch.zeros_like(g["s_w"]), torch.zeros_like(g["z_w"])
    wq2.copy_(g["wq"])        # written by the kernel just before the call
    sw2.copy_(g["s_w"])
    zw2.copy_(g["z_w"])
    assert torch.equal(b.linear_act(act, wq2, sw2, zw2, M, N, K, bias=g["bias"]), y_fused)
    d2 = synth.random_small(M, K, 70, seed=M + K, bias=False)
    g2 = inputs_to_dev(d2)
    y2 = b.linear_act(act, g2["wq"], g2["s_w"], g2["z_w"], M, 70, K)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d2["wq"], d2["s_w"], d2["z_w"], None)
    check_y(y2, y_ref, bound, f"linear_act {M}x{K}->70")
    assert b.sync_status() == 0


def test_quant_pack_near_ties_bitexact():
    """Activations placed on and around the rounding boundaries (k + 1/2) * s_a, for scales
    that are not powers of two: the codes must match the oracle's IEEE-division rounding
    bit for bit (the kernel divides only near such boundaries)."""
    rng = np.random.default_rng(123)
    rows = []
    for absmax in (1.0, 3.7, 0.013, 255.99, 1e-3, 77.77, 1.0e6, 0.3333333):
        a32 = np.float32(absmax)
        s = np.float32(a32 / np.float32(127.0))
        xs = [a32, -a32]
        for k in range(-126, 127, 3):
            c = np.float32((k + 0.5) * np.float64(s))
            xs += [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
            c2 = np.nextafter(np.nextafter(c, np.float32(np.inf)), np.float32(np.inf))
            xs += [c2, np.nextafter(c2, np.float32(np.inf))]
        xs = np.array(xs, np.float32)
        xs = xs[np.abs(xs) <= a32]
        K = ((len(xs) + 63) // 64) * 64
        row = np.zeros(K, np.float32)
        row[:len(xs)] = rng.permutation(xs)
        rows.append(row)
    K = max(len(r) for r in rows)
    x = np.zeros((len(rows), K), np.float32)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    a_q, s_a, rs = B().quant_pack(to_dev(x))
    ra, rsa, rrs = oracle.quant_pack(x)
    assert np.array_equal(s_a.cpu().numpy(), rsa)
    assert np.array_equal(a_q.cpu().numpy(), ra)
    assert np.array_equal(rs.cpu().numpy(), rrs)


@pytest.mark.parametrize("M,K,N,launches", [(8192, 4096, 14336, 200), (2048, 4096, 14336, 200)])
def test_repeated_launches_complete_and_identical(M, K, N, launches):
    """Many back-to-back launches of large persistent grids (thousands of pipeline stages per
    CTA, both token-tile widths): every launch ends with a clean status word and writes the
    same bits.  A stage consumed before its copies land, or a wait that alias-matches an
    earlier phase, shows up here as a timeout or as a differing output."""
    b = B()
    d = synth.make_linear(synth.LinearSpec("stress", M, K, N, True))
    g = inputs_to_dev(d)
    act = b.prepare_activations(g["x"])
    pw = b.prepare_weights(g["wq"], g["s_w"], g["z_w"])
    y0 = b.linear_prepared(act, pw, M, N, K, bias=g["bias"])
    assert b.sync_status() == 0
    y = torch.empty_like(y0)
    for i in range(launches):
        b.linear_prepared(act, pw, M, N, K, bias=g["bias"], y=y)
        if i % 20 == 19:
            assert b.sync_status() == 0, f"launch {i}"
            assert torch.equal(y, y0), f"launch {i}"
    # the first output itself, on sampled rows, against the oracle
    rows = np.linspace(0, M - 1, 6).astype(np.int64)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"][rows], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y0[torch.from_numpy(rows).to(dev())], y_ref, bound, f"rows of {M}x{K}x{N}")


# ------------------------------------------------------------------ few-token (decode) form
@pytest.mark.parametrize("M,K,N,bias", [(1, 64, 1, True), (1, 1024, 3072, True), (1, 1088, 257, False),
                                        (2, 2048, 1023, True), (3, 6144, 2048, False), (4, 192, 5, True),
                                        (5, 3136, 130, False), (6, 4096, 64, True), (7, 16384, 33, True),
                                        (8, 2048, 6144, False), (1, 20480, 3, True), (8, 64, 2, False)])
def test_decode_shapes(M, K, N, bias):
    """M <= 8 streams the packed weights: K chunk tails (K % 1024 != 0), odd N (the last row
    pair half empty), N below a CTA's rows, every token count; every output against the
    oracle, the fused call equal to quant_pack + linear bit for bit, and w4a8_linear with no
    workspace at all."""
    b = B()
    d = synth.random_small(M, K, N, seed=11 * M + K + N, bias=bias)
    g = inputs_to_dev(d)
    y_fused = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    a_q, s_a, rs = b.quant_pack(g["x"])
    y_sep = torch.empty_like(y_fused)
    rc = b.load().w4a8_linear(b._ptr(a_q), b._ptr(s_a), b._ptr(rs), b._ptr(g["wq"]), b._ptr(g["s_w"]),
                              b._ptr(g["z_w"]), b._ptr(g["bias"]), b._ptr(y_sep), M, N, K, None, 0,
                              b._stream(None))
    assert rc == 0
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_fused, y_ref, bound, f"decode {M}x{K}->{N}")
    assert torch.equal(y_fused, y_sep), "fused and separate calls differ"
    assert b.sync_status() == 0


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096), (2048, 6144), (6144, 2048)])
def test_decode_model_shapes_full(K, N):
    """One token through the 7B- and 1.7B-class projections, every output against the oracle;
    the no-alloc entry point gives the same bits."""
    b = B()
    d = synth.make_linear(synth.LinearSpec("decode", 1, K, N, True))
    g = inputs_to_dev(d)
    y = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y, y_ref, bound, f"decode 1x{K}->{N}")
    assert torch.equal(b.prefill_linear_noalloc(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"]), y)


@pytest.mark.parametrize("M,K,N", [(1, 1088, 257), (3, 6144, 130), (8, 2048, 301), (2, 192, 5), (1, 4096, 14336)])
def test_decode_offset_scale_views(M, K, N):
    """s_w and z_w as views that start 2 and 6 bytes into their allocations (so no span of a
    tile's rows begins or ends on a 16-byte boundary): the outputs equal the call on fresh
    arrays bit for bit and lie within tolerance of the oracle."""
    b = B()
    d = synth.random_small(M, K, N, seed=13 * M + K + N, bias=True)
    g = inputs_to_dev(d)
    y = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    nel = N * (K // 64)
    sbuf = torch.zeros(nel + 8, dtype=torch.float16, device=dev())
    zbuf = torch.zeros(nel + 8, dtype=torch.float16, device=dev())
    sw = sbuf[1:1 + nel].view(N, K // 64)
    zw = zbuf[3:3 + nel].view(N, K // 64)
    sw.copy_(g["s_w"])
    zw.copy_(g["z_w"])
    assert sw.data_ptr() % 16 == 2 and zw.data_ptr() % 16 == 6
    y_off = b.prefill_linear(g["x"], g["wq"], sw, zw, g["bias"])
    assert torch.equal(y_off, y)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_off, y_ref, bound, f"offset views {M}x{K}->{N}")
    assert b.sync_status() == 0


@pytest.mark.parametrize("M,K_N", [(1, ((2048, 4096), (2048, 2048), (2048, 12288), (6144, 2048))),
                                   (1, ((4096, 14336), (14336, 4096))),
                                   (1, ((1024, 3072), (3072, 1024))),
                                   (4, ((2048, 2048), (2048, 2048))),
                                   (2, ((1024, 3072), (2048, 1000), (1088, 257))),
                                   (1, tuple((64 * (i + 1), 100 + 37 * i) for i in range(8))),
                                   (1, tuple((1024, 512) for _ in range(9)))])
def test_batch_of_independent_linears(M, K_N):
    """Independent entries, which the few-token batch runs in one launch where they fit (a
    decoder layer's four groups, the 7B-class pair, two small pairs, ragged K / odd N at two
    tokens, the most entries one launch takes, and one entry more): every output equals the
    separate call's bit for bit."""
    b = B()
    ds = [synth.random_small(M, K, N, seed=300 + 7 * i + K + N, bias=i % 2 == 0) for i, (K, N) in enumerate(K_N)]
    gs = [inputs_to_dev(d) for d in ds]
    ents = [dict(x=g["x"], wq=g["wq"], s_w=g["s_w"], z_w=g["z_w"], bias=g["bias"]) for g in gs]
    ys = b.prefill_linear_batch(ents)
    for i, (e, y, d) in enumerate(zip(ents, ys, ds)):
        assert torch.equal(y, b.prefill_linear(e["x"], e["wq"], e["s_w"], e["z_w"], e["bias"])), f"entry {i}"
        y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
        check_y(y, y_ref, bound, f"entry {i}")
    assert b.sync_status() == 0


@pytest.mark.parametrize("M", [1, 3, 8, 300])
def test_batch_equals_separate_calls(M):
    """w4a8_prefill_linear_batch over a decoder layer's linears (hidden 2048: q/k/v and gate/up
    as row-concatenated groups, o, down) and one more entry whose x is the previous entry's y:
    every y equals the separate fused call's bit for bit (few-token kernels after the first
    stream their weights while the previous kernel runs), and lies within tolerance of the
    oracle."""
    b = B()
    shapes = [(2048, 4096), (2048, 2048), (2048, 12288), (6144, 2048)]
    ds = [synth.random_small(M, K, N, seed=200 + i, bias=i == 0) for i, (K, N) in enumerate(shapes)]
    gs = [inputs_to_dev(d) for d in ds]
    ents = [dict(x=g["x"], wq=g["wq"], s_w=g["s_w"], z_w=g["z_w"], bias=g["bias"]) for g in gs]
    # a fifth entry reading the fourth's output (K 2048 = the fourth's N)
    d5 = synth.random_small(M, 2048, 512, seed=205, bias=True)
    g5 = inputs_to_dev(d5)
    ents.append(dict(x=None, wq=g5["wq"], s_w=g5["s_w"], z_w=g5["z_w"], bias=g5["bias"]))
    y4 = torch.empty((M, 2048), device=dev())
    ents[3]["y"] = y4
    ents[4]["x"] = y4
    ys = b.prefill_linear_batch(ents)
    torch.cuda.synchronize()
    for i, (e, y) in enumerate(zip(ents, ys)):
        ref = b.prefill_linear(e["x"], e["wq"], e["s_w"], e["z_w"], e["bias"])
        assert torch.equal(y, ref), f"entry {i}"
    for i, (d, y) in enumerate(zip(ds, ys)):
        y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
        check_y(y, y_ref, bound, f"batch entry {i} M={M}")
    assert b.sync_status() == 0


@pytest.mark.parametrize("M", [1, 4])
def test_batch_pair_reading_its_own_output(M):
    """Two few-token entries where the second reads the first's y: the pair may not share a
    launch, and both outputs equal the separate calls in order, bit for bit, and the oracle's
    within tolerance (the second against the first's device output as its input)."""
    b = B()
    d1 = synth.random_small(M, 1024, 3072, seed=410, bias=True)
    d2 = synth.random_small(M, 3072, 1024, seed=411, bias=False)
    g1, g2 = inputs_to_dev(d1), inputs_to_dev(d2)
    y1 = torch.empty((M, 3072), device=dev())
    ents = [dict(x=g1["x"], wq=g1["wq"], s_w=g1["s_w"], z_w=g1["z_w"], bias=g1["bias"], y=y1),
            dict(x=y1, wq=g2["wq"], s_w=g2["s_w"], z_w=g2["z_w"], bias=None)]
    ys = b.prefill_linear_batch(ents)
    torch.cuda.synchronize()
    r1 = b.prefill_linear(g1["x"], g1["wq"], g1["s_w"], g1["z_w"], g1["bias"])
    r2 = b.prefill_linear(r1, g2["wq"], g2["s_w"], g2["z_w"], None)
    assert torch.equal(ys[0], r1) and torch.equal(ys[1], r2)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d1["x"], d1["wq"], d1["s_w"], d1["z_w"], d1["bias"])
    check_y(ys[0], y_ref, bound, f"first of the pair M={M}")
    y_ref, bound, _, _, _ = oracle.prefill_linear(r1.cpu().numpy(), d2["wq"], d2["s_w"], d2["z_w"], None)
    check_y(ys[1], y_ref, bound, f"second of the pair M={M}")
    assert b.sync_status() == 0


def test_batch_rejects_before_launch():
    """An invalid entry anywhere in the batch: its status, and no entry's y is written."""
    b = B()
    d = synth.random_small(1, 1024, 256, seed=7, bias=False)
    g = inputs_to_dev(d)
    lib = b.load()
    ys = [torch.full((1, 256), 3.0, device=dev()) for _ in range(2)]
    refs = (b.LinearRef * 2)()
    for i in range(2):
        refs[i] = b.LinearRef(g["x"].data_ptr(), g["wq"].data_ptr(), g["s_w"].data_ptr(), g["z_w"].data_ptr(), None,
                              ys[i].data_ptr(), 256, 1024, None, 0)
    refs[1].K = 1000                                      # not a multiple of 64
    import ctypes
    assert lib.w4a8_prefill_linear_batch(ctypes.cast(refs, ctypes.c_void_p), 2, 1, b._stream(None)) == \
        b.W4A8_ERR_SHAPE
    torch.cuda.synchronize()
    assert all(bool((y == 3.0).all()) for y in ys)
    assert b.sync_status() == 0


def test_decode_boundary_tokens():
    """8 tokens take the weight-streaming form, 9 the tensor-core form: both within the
    tolerance of the same definition on the same rows."""
    b = B()
    d = synth.random_small(9, 2048, 777, seed=99, bias=True)
    g = inputs_to_dev(d)
    y9 = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    y8 = b.prefill_linear(g["x"][:8].contiguous(), g["wq"], g["s_w"], g["z_w"], g["bias"])
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y9, y_ref, bound, "9 tokens")
    check_y(y8, y_ref[:8], bound[:8], "8 tokens")


# ------------------------------------------------------------------ epilogue variants
@pytest.mark.parametrize("M,K,N", [(300, 1024, 700), (4100, 512, 300), (1, 2048, 1000), (5, 4096, 777),
                                   (2, 1024, 129)])
def test_epilogue_clamp_and_bf16(M, K, N):
    """The *_ex calls: fp32 with the default bounds equals the plain call bit for bit; the
    clamp against the clamped oracle output; bf16 within the fp32 tolerance plus half a bf16
    step; the split and prepared forms give the fused form's bits.  Covers the 128- and
    256-token contractions and both few-token paths (in-kernel and separate pre-pass)."""
    from gpu_util import ABS_TOL, REL_TOL
    b = B()
    d = synth.random_small(M, K, N, seed=3 * M + K + 7 * N, bias=True)
    g = inputs_to_dev(d)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    lo, hi = (float(v) for v in np.quantile(y_ref, [0.2, 0.85]))
    y_plain = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    assert torch.equal(b.prefill_linear_ex(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"]), y_plain)
    clipped = np.clip(y_ref, lo, hi)
    yc = b.prefill_linear_ex(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], clamp=(lo, hi))
    check_y(yc, clipped, bound, f"clamp {M}x{K}->{N}")
    assert float(yc.min()) >= np.float32(lo) and float(yc.max()) <= np.float32(hi)
    yb = b.prefill_linear_ex(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], out_dtype=torch.bfloat16,
                             clamp=(lo, hi))
    assert yb.dtype == torch.bfloat16
    got = yb.float().cpu().numpy().astype(np.float64)
    allowed = REL_TOL * bound + ABS_TOL
    allowed = allowed + 2.0 ** -8 * (np.abs(clipped) + allowed)
    err = np.abs(got - clipped)
    assert np.all(err <= allowed), f"bf16: {int((err > allowed).sum())} outputs outside tolerance"
    e_ref = oracle.epilogue(y_ref, lo, hi, "bf16")
    assert np.mean(got == e_ref) > 0.95  # the same bf16 value except next to rounding boundaries
    a_q, s_a, rs = b.quant_pack(g["x"])
    ys = b.linear_ex(a_q, s_a, rs, g["wq"], g["s_w"], g["z_w"], g["bias"], out_dtype=torch.bfloat16, clamp=(lo, hi))
    assert torch.equal(ys, yb), "split form differs"
    if M > 8:
        act = b.prepare_activations(g["x"])
        pw = b.prepare_weights(g["wq"], g["s_w"], g["z_w"])
        yp = b.linear_prepared_ex(act, pw, M, N, K, bias=g["bias"], out_dtype=torch.bfloat16, clamp=(lo, hi))
        assert torch.equal(yp, yb), "prepared form differs"
    assert b.sync_status() == 0


def test_epilogue_argument_checks():
    b = B()
    d = synth.random_small(4, 64, 8, seed=1, bias=False)
    g = inputs_to_dev(d)
    y = torch.empty((4, 8), device=dev())
    lib = b.load()
    args = (b._ptr(g["x"]), b._ptr(g["wq"]), b._ptr(g["s_w"]), b._ptr(g["z_w"]), None, b._ptr(y))
    assert lib.w4a8_prefill_linear_ex(*args, 7, -1.0, 1.0, 4, 8, 64, None, 0, b._stream(None)) == b.W4A8_ERR_ARG
    assert lib.w4a8_prefill_linear_ex(*args, 0, 1.0, -1.0, 4, 8, 64, None, 0, b._stream(None)) == b.W4A8_ERR_ARG
    assert lib.w4a8_prefill_linear_ex(*args, 0, float("nan"), 1.0, 4, 8, 64, None, 0, b._stream(None)) == \
        b.W4A8_ERR_ARG
    assert b.sync_status() == 0



def test_binding_checks_every_tensor_before_launch():
    """The binding checks each tensor's device, dtype, shape and (for the opaque prepared
    buffers, which the C call receives without a length) size, so a mismatched argument
    raises in Python and nothing is launched."""
    b = B()
    M, N, K = 4, 8, 128
    d = synth.random_small(M, K, N, seed=2, bias=True)
    g = inputs_to_dev(d)
    x, wq, sw, zw, bias = g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"]
    bad = {
        "y shape": lambda: b.prefill_linear(x, wq, sw, zw, bias, y=torch.empty((M, N + 1), device=dev())),
        "y dtype": lambda: b.prefill_linear(x, wq, sw, zw, bias, y=torch.empty((M, N), device=dev(),
                                                                             dtype=torch.float16)),
        "y on host": lambda: b.prefill_linear(x, wq, sw, zw, bias, y=torch.empty((M, N))),
        "bias on host": lambda: b.prefill_linear(x, wq, sw, zw, bias.cpu()),
        "bias length": lambda: b.prefill_linear(x, wq, sw, zw, bias[:N - 1]),
        "scale shape": lambda: b.prefill_linear(x, wq, sw[:, :1].contiguous(), zw, bias),
        "zero dtype": lambda: b.prefill_linear(x, wq, sw, zw.float(), bias),
        "wq depth": lambda: b.prefill_linear(x[:, :64].contiguous(), wq, sw, zw, bias),
        "strided x": lambda: b.prefill_linear(torch.empty((M, 2 * K), device=dev())[:, :K], wq, sw, zw, bias),
        "ws on host": lambda: b.linear(*b.quant_pack(x), wq, sw, zw, bias, ws=torch.empty(1 << 20,
                                                                                         dtype=torch.uint8)),
        "rowsum shape": lambda: b.linear(b.quant_pack(x)[0], b.quant_pack(x)[1],
                                         torch.zeros((M, 1), dtype=torch.int32, device=dev()), wq, sw, zw),
        "act too small": lambda: b.linear_prepared(torch.empty(64, dtype=torch.uint8, device=dev()),
                                                   b.prepare_weights(wq, sw, zw), M, N, K),
        "pw too small": lambda: b.linear_prepared_ex(b.prepare_activations(x),
                                                     torch.empty(64, dtype=torch.uint8, device=dev()), M, N, K),
        "debug wq rows": lambda: b.debug_block_acc(b.quant_pack(x)[0], wq, N + 1),
        "debug window": lambda: b.debug_block_acc(b.quant_pack(x)[0], wq, N, m0=2, m_cnt=3),
    }
    y = torch.zeros((M, N), device=dev())
    for what, call in bad.items():
        with pytest.raises((TypeError, ValueError)):
            call()
    b.prefill_linear(x, wq, sw, zw, bias, y=y)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y, y_ref, bound, "after rejected calls")
    assert b.sync_status() == 0



def test_temporary_workspace_follows_the_call_stream(monkeypatch):
    """A call on a stream that is not the current one, with no workspace given: the binding's
    temporary workspace is held for that stream's work, so a block allocated on the current
    stream right after the call is not the same memory while the call is still queued."""
    b = B()
    M, K, N = 512, 1024, 640
    d = synth.random_small(M, K, N, seed=8, bias=True)
    g = inputs_to_dev(d)
    ref = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    torch.cuda.synchronize()
    made = []
    orig = b.workspace

    def spy(nbytes, device):
        t = orig(nbytes, device)
        made.append(t.data_ptr())
        return t

    monkeypatch.setattr(b, "workspace", spy)
    s = torch.cuda.Stream()
    y = torch.empty_like(ref)
    with torch.cuda.stream(s):
        torch.cuda._sleep(50_000_000)            # keeps the side stream busy for some milliseconds
    b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y, stream=s)
    assert len(made) == 1
    other = torch.empty(b.prefill_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev())
    assert other.data_ptr() != made[0], "the temporary workspace was handed out while still in use"
    other.fill_(0xA5)
    s.synchronize()
    assert torch.equal(y, ref)
    assert b.sync_status() == 0


# ------------------------------------------------------------------ host-buffer call
def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("M,K,N", [(1500, 1024, 2560), (2048, 2048, 4096), (8300, 512, 256), (9000, 512, 1536),
                                   (16384, 1024, 1024), (512, 1024, 640), (700, 256, 200), (255, 512, 96),
                                   (4096, 128, 64), (3, 1024, 256), (255, 2048, 96), (512, 16384, 1024)])
def test_host_call_equals_fused(M, K, N):
    """x and y in page-locked host memory, chunked copies overlapping the computation: the
    outputs equal the device-buffer fused call's bit for bit -- two chunks with a ragged
    last one; six chunks over four compute streams (streams and activation buffers reused);
    chunks of whole 256-row tiles below 4096 rows each through the 256-token kernel; eight
    chunks; the full sixteen; in place on the mapped buffers (128-token tiles, a ragged last
    tile, fewer than two tiles, 256-token tiles); the few-token form; in place with K split
    over CTA pairs; four chunks of a linear whose K is split over CTA pairs (each chunk told
    the uncut call's split) -- and lie within tolerance of the oracle."""
    b = B()
    d = synth.random_small(M, K, N, seed=70 + M + N, bias=True)
    g = inputs_to_dev(d)
    xh = _pinned(d["x"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y_dev = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], stream=s)
        yh = b.prefill_linear_host(xh, g["wq"], g["s_w"], g["z_w"], g["bias"], stream=s)
    s.synchronize()
    assert torch.equal(yh, y_dev.cpu())
    rows = np.unique(np.linspace(0, M - 1, min(M, 64)).astype(np.int64))
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"], rows=rows)
    check_y(yh[rows], y_ref, bound, f"host call {M}x{K}->{N}")
    assert b.sync_status() == 0


def test_host_call_reuses_a_workspace_in_stream_order():
    """Three calls on one stream through one workspace, each with its own host x and y: the
    later calls' copies in wait for the earlier calls to finish, so every y is its own x's."""
    b = B()
    M, K, N = 1024, 2048, 2048
    ds = [synth.random_small(M, K, N, seed=90 + i, bias=i == 1) for i in range(3)]
    ws = b.workspace(b.prefill_host_workspace_bytes(M, N, K), dev())
    s = torch.cuda.Stream()
    outs = []
    for d in ds:
        gw = inputs_to_dev(d)
        xh = _pinned(d["x"])   # held until the stream is synchronized: torch cannot see the library's copies
        outs.append((d, gw, xh, b.prefill_linear_host(xh, gw["wq"], gw["s_w"], gw["z_w"], gw["bias"], ws=ws,
                                                       stream=s)))
    s.synchronize()
    for d, gw, _, yh in outs:
        ref = b.prefill_linear(to_dev(d["x"]), gw["wq"], gw["s_w"], gw["z_w"], gw["bias"])
        assert torch.equal(yh, ref.cpu())
    assert b.sync_status() == 0


def test_tape_counts_its_kernels():
    """w4a8_tape_kernels: the kernel launches one replay makes -- a fused call (pre-pass and
    contraction), a quantizing few-token call (one kernel), a decoder layer's four few-token
    groups in one batch call (one launch), a pair of 3 MB of weights as a batch (one launch),
    and the 7B-class pair as a batch (a launch each: 58.7 MB of weights)."""
    b = B()
    s = torch.cuda.Stream()

    def count(fn):
        with torch.cuda.stream(s):
            fn()                      # one ordinary call before recording
            with b.Tape(s) as t:
                fn()
        s.synchronize()
        n = t.kernels()
        t.free()
        return n

    def ents(M, shapes, seed):
        out = []
        for i, (K, N) in enumerate(shapes):
            g = inputs_to_dev(synth.random_small(M, K, N, seed=seed + i, bias=True))
            out.append(dict(x=g["x"], wq=g["wq"], s_w=g["s_w"], z_w=g["z_w"], bias=g["bias"]))
        return out

    g = ents(300, [(1024, 640)], 80)[0]
    assert count(lambda: b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], stream=s)) == 2
    g = ents(1, [(1024, 640)], 81)[0]
    assert count(lambda: b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], stream=s)) == 1
    layer = b.Batch(ents(1, [(2048, 4096), (2048, 2048), (2048, 12288), (6144, 2048)], 82), s)
    assert count(lambda: layer.run(s)) == 1
    small = b.Batch(ents(1, [(1024, 3072), (3072, 1024)], 84), s)
    assert count(lambda: small.run(s)) == 1
    pair = b.Batch(ents(1, [(4096, 14336), (14336, 4096)], 86), s)
    assert count(lambda: pair.run(s)) == 2
    assert b.sync_status() == 0


def test_tape_records_the_host_call():
    """Host-buffer calls recorded into a tape -- one cut into chunks (its side streams joined
    back into the capture), one small enough to work on the mapped host buffers in place --
    replay bit for bit, and follow new contents of the same host x."""
    b = B()
    shapes = [(2048, 1024, 2048), (512, 1024, 320)]
    ds = [synth.random_small(M, K, N, seed=95 + i, bias=True) for i, (M, K, N) in enumerate(shapes)]
    gs = [inputs_to_dev(d) for d in ds]
    xs = [_pinned(d["x"]) for d in ds]
    ys = [torch.empty((M, N)).pin_memory() for M, K, N in shapes]
    wss = [b.workspace(b.prefill_host_workspace_bytes(M, N, K), dev()) for M, K, N in shapes]
    s = torch.cuda.Stream()

    def calls():
        for g, xh, yh, ws in zip(gs, xs, ys, wss):
            b.prefill_linear_host(xh, g["wq"], g["s_w"], g["z_w"], g["bias"], y=yh, ws=ws, stream=s)

    with torch.cuda.stream(s):
        calls()
        s.synchronize()
        eager = [y.clone() for y in ys]
        with b.Tape(s) as tape:
            calls()
    for y in ys:
        y.fill_(float("nan"))
    tape.replay(s)
    s.synchronize()
    for y, e in zip(ys, eager):
        assert torch.equal(y, e)
    for xh in xs:
        xh.mul_(-0.5)
    refs = [b.prefill_linear(xh.to(dev()), g["wq"], g["s_w"], g["z_w"], g["bias"]).cpu() for xh, g in zip(xs, gs)]
    tape.replay(s)
    s.synchronize()
    for y, r in zip(ys, refs):
        assert torch.equal(y, r)
    tape.free()
    assert b.sync_status() == 0


def test_host_call_rejects_pageable_memory():
    """A host pointer the driver does not know as page-locked is refused (nothing launched)."""
    b = B()
    M, K, N = 256, 128, 64
    d = synth.random_small(M, K, N, seed=3, bias=False)
    g = inputs_to_dev(d)
    xp = torch.from_numpy(d["x"].copy())                  # pageable
    yp = torch.empty((M, N))
    ws = b.workspace(b.prefill_host_workspace_bytes(M, N, K), dev())
    lib = b.load()
    rc = lib.w4a8_prefill_linear_host(b._ptr(xp), b._ptr(g["wq"]), b._ptr(g["s_w"]), b._ptr(g["z_w"]), None,
                                      b._ptr(yp), M, N, K, b._ptr(ws), ws.numel(), b._stream(None))
    assert rc == b.W4A8_ERR_ARG
    assert b.sync_status() == 0


# ------------------------------------------------------------------ command tapes
def test_tape_replays_a_mixed_sequence():
    """A tape recording the fused call at three forms (128-token, 256-token, few-token), the
    bf16 variant, and one pre-pass shared by two prepared linears, replays bit for bit what
    the same calls give eagerly -- and again after the inputs change in place."""
    b = B()
    stream = torch.cuda.Stream()
    shapes = [(300, 1024, 700), (4100, 512, 300), (1, 2048, 1000), (3, 4096, 200)]
    ds = [synth.random_small(M, K, N, seed=40 + i, bias=True) for i, (M, K, N) in enumerate(shapes)]
    gs = [inputs_to_dev(d) for d in ds]
    outs = [torch.empty((M, N), device=dev()) for M, K, N in shapes]
    wss = [b.workspace(b.prefill_workspace_bytes(M, N, K), dev()) for M, K, N in shapes]
    yb = torch.empty((300, 700), dtype=torch.bfloat16, device=dev())
    # shared pre-pass: one input, two prepared weight sets
    dq = synth.random_small(256, 2048, 512, seed=50, bias=False)
    dk = synth.random_small(256, 2048, 384, seed=51, bias=True)
    xq = to_dev(dq["x"])
    pq = b.prepare_weights(to_dev(dq["wq"]), to_dev(dq["s_w"]), to_dev(dq["z_w"]))
    pk = b.prepare_weights(to_dev(dk["wq"]), to_dev(dk["s_w"]), to_dev(dk["z_w"]))
    act = b.workspace(b.prepared_activations_bytes(256, 2048), dev())
    yq = torch.empty((256, 512), device=dev())
    yk = torch.empty((256, 384), device=dev())
    bk = to_dev(dk["bias"])

    def calls(s):
        for g, y, ws in zip(gs, outs, wss):
            b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y, ws=ws, stream=s)
        b.prefill_linear_ex(gs[0]["x"], gs[0]["wq"], gs[0]["s_w"], gs[0]["z_w"], gs[0]["bias"], y=yb,
                            clamp=(-1.0, 1.0), ws=wss[0], stream=s)
        b.prepare_activations(xq, act=act, stream=s)
        b.linear_prepared(act, pq, 256, 512, 2048, y=yq, stream=s)
        b.linear_prepared(act, pk, 256, 384, 2048, bias=bk, y=yk, stream=s)

    results = lambda: [o.clone() for o in outs] + [yb.clone(), yq.clone(), yk.clone()]
    with torch.cuda.stream(stream):
        calls(stream)
    stream.synchronize()
    eager = results()
    with torch.cuda.stream(stream):
        with b.Tape(stream) as tape:
            calls(stream)
    for o in outs + [yq, yk]:
        o.fill_(float("nan"))
    yb.fill_(float("nan"))
    tape.replay(stream)
    stream.synchronize()
    for e, r in zip(eager, results()):
        assert torch.equal(e, r)
    # new inputs, same buffers: the replay follows them
    for g in gs:
        g["x"].mul_(-0.5)
    xq.add_(0.25)
    with torch.cuda.stream(stream):
        calls(stream)
    stream.synchronize()
    eager2 = results()
    for o in outs + [yq, yk]:
        o.zero_()
    tape.replay(stream)
    stream.synchronize()
    for e, r in zip(eager2, results()):
        assert torch.equal(e, r)
    assert not torch.equal(eager[0], eager2[0])
    tape.free()
    assert b.sync_status() == 0


@pytest.mark.parametrize("M", [512, 1])
def test_row_concatenated_group_equals_members(M):
    """q/k/v stored as one row-concatenated weight matrix: one call gives each member's
    outputs in its column range -- every output within tolerance of the oracle, and, for the
    tensor-core form (whose per-output arithmetic does not depend on N), bit for bit the
    separate calls' outputs."""
    b = B()
    Ns = (512, 256, 256)
    K = 2048
    ds = [synth.random_small(M, K, N, seed=60 + i, bias=True) for i, N in enumerate(Ns)]
    x = ds[0]["x"]
    g = {k: to_dev(np.concatenate([d[k] for d in ds])) for k in ("wq", "s_w", "z_w", "bias")}
    y = b.prefill_linear(to_dev(x), g["wq"], g["s_w"], g["z_w"], g["bias"])
    off = 0
    for d, N in zip(ds, Ns):
        gi = inputs_to_dev(d)
        yi = b.prefill_linear(to_dev(x), gi["wq"], gi["s_w"], gi["z_w"], gi["bias"])
        y_ref, bound, _, _, _ = oracle.prefill_linear(x, d["wq"], d["s_w"], d["z_w"], d["bias"])
        check_y(y[:, off:off + N], y_ref, bound, f"group member N={N}")
        if M > 8:
            assert torch.equal(y[:, off:off + N], yi)
        off += N


@pytest.mark.parametrize("M,K,N,launches", [(1, 4096, 14336, 300), (1, 14336, 4096, 300), (8, 4096, 3000, 200)])
def test_decode_repeated_launches_complete_and_identical(M, K, N, launches):
    """Back-to-back few-token calls (one launch each when the kernel quantizes, pre-pass plus
    kernel at M = 8, K = 4096): a clean status word and the same bits every time; the first
    output against the oracle."""
    b = B()
    d = synth.make_linear(synth.LinearSpec("stress", M, K, N, True))
    g = inputs_to_dev(d)
    y0 = b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"])
    assert b.sync_status() == 0
    ws = b.workspace(b.prefill_workspace_bytes(M, N, K), dev())
    y = torch.empty_like(y0)
    for i in range(launches):
        b.prefill_linear(g["x"], g["wq"], g["s_w"], g["z_w"], g["bias"], y=y, ws=ws)
        if i % 50 == 49:
            assert b.sync_status() == 0, f"launch {i}"
            assert torch.equal(y, y0), f"launch {i}"
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y0, y_ref, bound, f"decode {M}x{K}->{N}")


@pytest.mark.parametrize("M,K,N,bias", [(4096, 64, 129, True), (4095, 64, 257, False), (4096, 1024, 1, True),
                                        (4097, 64, 64, False), (9, 64, 1, True), (8, 16384, 7, False)])
def test_form_boundaries(M, K, N, bias):
    """Shapes at the routing boundaries: exactly 4096 tokens (the first 256-token-tile size)
    and one below and above it, a single 64-block per tile (K = 64), one output column, 9
    tokens (the smallest tensor-core call) and 8 tokens whose row does not fit the kernel's
    own quantizer (separate pre-pass); every output against the oracle, fused = separate."""
    d = synth.random_small(M, K, N, seed=5 * M + K + N, bias=bias)
    y_fused, y_sep = _run_both(d)
    y_ref, bound, _, _, _ = oracle.prefill_linear(d["x"], d["wq"], d["s_w"], d["z_w"], d["bias"])
    check_y(y_fused, y_ref, bound, f"boundary {M}x{K}->{N}")
    assert torch.equal(y_fused, y_sep), "fused and separate calls differ"
    assert B().sync_status() == 0
