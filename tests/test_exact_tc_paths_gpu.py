"""The bf16 exact tier's tensor-core kernel, path by path, against the oracle.

The kernel computes the literal algorithm's bits (Carbon README, "How It
Works": float64 products, 256-wide chunks summed with KBN left to right, the
chunk values combined with KBN) from exact integer chunk sums.  Each test
below builds operands that drive one of its paths and checks the float64
value before rounding and the rounded output bit for bit against the CPU
oracle; where the library's path counters can show that the path ran, the
test asserts that too:

* rounded chunk values: KBN steps inside a chunk round, the chunk value is the
  exact chunk sum rounded once to float64;
* chunk repair: a line of a chunk is wider than the 31 bits the digit planes
  carry, so that (output, chunk) is summed separately and added in;
* whole-output fix-up: the integer outer sum would leave the int64 range, or
  a line holds inf/NaN or is wider than 62 bits;
* split chunk ranges: few output tiles, the chunk range is cut into pieces
  whose integer sums add exactly;
* bias alignment: a bias far finer or far coarser than the output grain.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as inputs
from tests.gpu_util import bits, dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import deterministic_invariant_gemm_fwd_gb300 as cg  # noqa: E402


def run(pass_, A, B, bias, M, K, N, f64):
    shape = oracle.out_shape(pass_, M, K, N)
    tA, tB = dev(A), dev(B)
    tb = dev(bias) if bias is not None else None
    if f64:
        out = torch.empty(shape, dtype=torch.float64, device="cuda")
        cg.carbon_debug_exact_y64(pass_, out, tA, tB, tb, M, K, N, "bf16")
    else:
        out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        {"fwd": lambda: cg.carbon_gemm_fwd(out, tA, tB, tb, M, K, N, "bf16", "exact"),
         "dx": lambda: cg.carbon_gemm_dx(out, tA, tB, M, K, N, "bf16", "exact"),
         "dw": lambda: cg.carbon_gemm_dw(out, tA, tB, M, K, N, "bf16", "exact")}[pass_]()
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    return host_bits(out)


def check(pass_, A, B, bias, M, K, N):
    """Bit-exact against the oracle; returns (chunk repairs, fix-ups) of the
    bf16 output call."""
    ref, ref64 = oracle.gemm(pass_, "bf16", A, B, bias, M, K, N)
    got64 = run(pass_, A, B, bias, M, K, N, True)
    cg.carbon_debug_kernel_timing(True)
    try:
        got = run(pass_, A, B, bias, M, K, N, False)
        counts = cg.carbon_debug_exact_path_counts()
    finally:
        cg.carbon_debug_kernel_timing(False)
    assert np.array_equal(got64, bits(ref64)), \
        f"{pass_} {M}x{K}x{N}: {np.count_nonzero(got64 != bits(ref64))} float64 mismatches"
    assert np.array_equal(got, bits(ref)), \
        f"{pass_} {M}x{K}x{N}: {np.count_nonzero(got != bits(ref))} output mismatches"
    return counts


def bf16(a):
    return inputs.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def spread(rng, shape, lo, hi, sign=True):
    """bf16 values m * 2^e, e uniform in [lo, hi], random 8-bit significands."""
    v = np.ldexp(1.0 + rng.integers(0, 128, shape) / 128.0, rng.integers(lo, hi + 1, shape))
    if sign:
        v = v * rng.choice([-1.0, 1.0], shape)
    return v


def test_rounded_chunk_values():
    """Same-sign operands of width ~30: chunk sums far above 2^53 units of the
    chunk grain, so KBN's partial sums round; the chunk value must be the exact
    sum rounded once."""
    rng = np.random.default_rng(11)
    M, K, N = 140, 600, 70
    X = bf16(spread(rng, (M, K), -11, 11, sign=False))
    W = bf16(spread(rng, (K, N), -11, 11, sign=False))
    b = bf16(rng.standard_normal(N))
    check("fwd", X, W, b, M, K, N)


def test_chunk_repair_wide_lines():
    """A few rows and columns hold one tiny entry each (width ~45 bits in that
    chunk): only those (output, chunk) pairs leave the tensor cores."""
    rng = np.random.default_rng(12)
    M, K, N = 200, 520, 100
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-3)
    X = inputs.bf16_bits_to_f32(L["X"]).copy()
    W = inputs.bf16_bits_to_f32(L["W"]).copy()
    X[[3, 77, 150], [10, 300, 511]] = np.float32(2.0 ** -40)
    W[[5, 260], [7, 64]] = np.float32(-(2.0 ** -50))
    X, W = bf16(X), bf16(W)
    repairs, fixups = check("fwd", X, W, L["b"], M, K, N)
    assert repairs > 0
    repairs, fixups = check("dw", X, L["dY"], None, M, K, N)
    assert repairs > 0


def test_fixup_outer_sum_out_of_range():
    """Row 0's first chunk holds tiny entries and its second huge ones: in the
    output grain the running sum needs far more than 62 bits, so those outputs
    are recomputed whole."""
    rng = np.random.default_rng(13)
    M, K, N = 130, 512, 65
    X = rng.standard_normal((M, K))
    X[0, :256] = np.ldexp(1.0, -90) * (1 + rng.integers(0, 128, 256) / 128.0)
    X[0, 256:] = np.ldexp(1.0, 60) * (1 + rng.integers(0, 128, 256) / 128.0)
    W = rng.standard_normal((K, N)) * 0.02
    repairs, fixups = check("fwd", bf16(X), bf16(W), bf16(rng.standard_normal(N) * 0.02), M, K, N)
    assert fixups > 0


def test_fixup_non_finite_and_extreme_widths():
    """inf in one row, entries 2^-120 and 2^120 in another (width > 62): whole
    fix-up with the literal float64 loop for those chunks."""
    rng = np.random.default_rng(14)
    M, K, N = 66, 300, 33
    X = rng.standard_normal((M, K))
    X[5, 17] = np.inf
    X[9, 3] = 2.0 ** -120
    X[9, 200] = 2.0 ** 120
    W = rng.standard_normal((K, N)) * 0.02
    ref, ref64 = oracle.gemm("fwd", "bf16", bf16(X), bf16(W), None, M, K, N)
    got64 = run("fwd", bf16(X), bf16(W), None, M, K, N, True)
    got = run("fwd", bf16(X), bf16(W), None, M, K, N, False)
    finite = np.isfinite(ref64)
    assert np.array_equal(got64[finite], bits(ref64)[finite])
    assert np.array_equal(np.isnan(got64.view(np.float64)), np.isnan(ref64))
    assert np.array_equal(got[finite], bits(ref)[finite])


@pytest.mark.parametrize("M", [4096, 4000])
def test_split_chunk_ranges_dw(M):
    """dW with one row tile and two column tiles over 16 chunks of tokens: the
    chunk range is cut into pieces whose integer sums must add to the
    one-piece result."""
    rng = np.random.default_rng(M)
    K, N = 128, 100
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-4)
    check("dw", L["X"], L["dY"], None, M, K, N)


def test_bias_far_from_the_grain():
    """Bias entries far finer than the output grain (2^-110) and far coarser
    (2^50): the bias is added through float64 there."""
    rng = np.random.default_rng(15)
    M, K, N = 130, 300, 66
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N)) * 0.02
    b = rng.standard_normal(N) * 0.02
    b[:10] = np.ldexp(1.0, -110) * (1 + rng.integers(0, 128, 10) / 128.0)
    b[10:20] = np.ldexp(1.0, 50) * (1 + rng.integers(0, 128, 10) / 128.0)
    b[20] = 0.0
    b[21] = -0.0
    check("fwd", bf16(X), bf16(W), bf16(b), M, K, N)


@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_gpt2_shape_tail_and_zero_lines(pass_):
    """A GPT-2-like layer with ragged sizes, zero rows and zero columns, and
    whole zero chunks."""
    rng = np.random.default_rng(16)
    M, K, N = 300, 700, 190
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-4)
    X = inputs.bf16_bits_to_f32(L["X"]).copy()
    X[7, :] = 0.0
    X[:, 256:512] = 0.0
    W = inputs.bf16_bits_to_f32(L["W"]).copy()
    W[:, 3] = 0.0
    dY = inputs.bf16_bits_to_f32(L["dY"]).copy()
    dY[:, 11] = -0.0
    ops = {"fwd": (bf16(X), bf16(W), L["b"]), "dx": (bf16(dY), bf16(W), None),
           "dw": (bf16(X), bf16(dY), None)}[pass_]
    check(pass_, *ops, M, K, N)


@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_plane_counts_per_tile_and_trailing_zeros(pass_):
    """Operand lines of every digit count: the B side's lines (columns of W,
    rows of W for dX, columns of dY for dW) come in groups of 64, each group
    of a different width, so the column tiles of one chunk need 1, 2, 3 and 4
    digit planes (the tensor-core kernel then runs MMAs of
    N = 64, 128, 192 and 256); the A side mixes the same spans by row.  Half
    of the values have significands with trailing zero bits (a line's base
    sits above its smallest exponent), and one chunk of every B line is all
    zero, or holds a single power of two."""
    rng = np.random.default_rng(31)
    M, K, N = 260, 580, 264            # 3 chunks (the last one short), ragged tiles

    def lines(n, length, seed_off):
        r = np.random.default_rng(100 + seed_off)
        v = np.empty((n, length))
        for li in range(n):
            kind = (li // 64) % 4                # line width about 6, 12, 20, 28 bits
            e0 = int(r.integers(-20, 4))
            if kind == 0:                        # integers below 2^6 times 2^e0: one digit
                v[li] = np.ldexp(r.integers(-63, 64, length).astype(np.float64), e0)
            else:                                # 8 + 8 (kind - 1) + 3 bits: kind + 1 digits
                v[li] = spread(r, length, e0 - (8 * kind - 5), e0)
            coarse = (r.random(length) < 0.5) & (v[li] != 0)   # 4-bit significands
            a = np.abs(v[li, coarse])
            ex = np.floor(np.log2(a)).astype(np.int64)
            v[li, coarse] = np.sign(v[li, coarse]) * np.ldexp(np.round(np.ldexp(a, 3 - ex)), ex - 3)
            q = int(r.integers(0, (length + 255) // 256))
            lo, hi = 256 * q, min(length, 256 * q + 256)
            if li % 3 == 0:
                v[li, lo:hi] = 0.0
            elif li % 3 == 1:
                v[li, lo:hi] = 0.0
                v[li, lo + int(r.integers(0, hi - lo))] = np.ldexp(1.0, int(r.integers(-30, 10)))
        return v

    if pass_ == "fwd":
        X = bf16(lines(M, K, 0))
        W = bf16(lines(N, K, 1).T)
        b = bf16(rng.standard_normal(N))
        check("fwd", X, W, b, M, K, N)
    elif pass_ == "dx":
        dY = bf16(lines(M, N, 2))
        W = bf16(lines(K, N, 3))           # rows of W are the B lines of dX
        check("dx", dY, W, None, M, K, N)
    else:
        Mt, Kd, Nd = 600, 200, 264         # dW: reduction over 600 tokens
        X = bf16(lines(Kd, Mt, 4).T)
        dY = bf16(lines(Nd, Mt, 5).T)
        check("dw", X, dY, None, Mt, Kd, Nd)


def test_outer_sum_wraps_within_a_piece():
    """Two chunks of one piece whose shifted chunk sums each fit 63 bits but
    whose running sum passes 2^63 (the int64 sum wraps): rows of integers
    8..504 in chunks 0 and 1 and one entry near 2^-25 in chunk 2 (so the row's
    grain is 28 bits below those chunks), columns whose chunk sums give about
    2^61 and 2^62 in grain units, scaled per column across the boundary.  The
    kernel must notice the wrap and send the output to the fix-up, never keep
    the wrapped sum (a signed range test that overflowed once let it through).
    With 2 x 2 output tiles and 3 chunks the chunk range is cut in two pieces,
    chunks 0 and 1 together."""
    rng = np.random.default_rng(7)
    M, K, N = 130, 768, 70
    X = np.zeros((M, K))
    W = np.zeros((K, N))
    for i in range(M):
        X[i, :512] = np.ldexp(rng.integers(1, 64, 512).astype(np.float64), 3)
        X[i, 512 + int(rng.integers(0, 256))] = np.ldexp(1.0, int(rng.integers(-26, -24)))
    for j in range(N):
        c = 0.6 + 0.9 * j / N
        for q, target in ((0, 700.0), (1, 1500.0), (2, 1.0)):
            w = rng.random(256) + 0.5
            w = w / w.sum() * target * c / 256.0
            w[int(rng.integers(0, 256))] = np.ldexp(1.0 + rng.integers(0, 128) / 128.0, -20)
            W[256 * q:256 * q + 256, j] = w
    _, fixups = check("fwd", bf16(X), bf16(W), None, M, K, N)
    assert fixups > 0


def _tie_operands(rng, exps, ks, cs, hs, K, main_at, tie_at, tiny_at, sigma):
    """Rows of m * 2^E (m of 8 bits, random sign) at reduction index main_at
    (against W = 1), 2^(E-8+sigma) at tie_at (against c * 2^-sigma: c times
    half a bf16 ulp of the main value) and +-2^(E-8-k) at tiny_at (against h),
    for every E in exps and k in ks (k None: no tiny entry), 6 rows each, the
    first with the largest m; columns for every (c, h) pair, three times.
    The tie entries make the exact sums land on bf16 midpoints or near them,
    the tiny ones decide them or vanish in the float64 rounding."""
    rows = [(E, k, r) for E in exps for k in ks for r in range(6)]
    cols = [(c, h) for c in cs for h in hs] * 3
    M, N = len(rows), len(cols)
    X = np.zeros((M, K))
    W = np.zeros((K, N))
    for i, (E, k, r) in enumerate(rows):
        a = 127 if r == 0 else rng.integers(0, 128)              # 127: a midpoint rounds up a binade
        a &= -(1 << max(0, -126 - E))                            # bf16 subnormals hold fewer bits
        X[i, main_at] = rng.choice([-1.0, 1.0]) * np.ldexp(1.0 + a / 128.0, E)
        X[i, tie_at] = np.ldexp(1.0, E - 8 + sigma)
        if k is not None:
            X[i, tiny_at] = rng.choice([-1.0, 1.0]) * np.ldexp(1.0, E - 8 - k)
    for j, (c, h) in enumerate(cols):
        W[main_at, j] = 1.0
        W[tie_at, j] = np.ldexp(c, -sigma)
        W[tiny_at, j] = h
    return X, W, M, N


def test_output_rounding_midpoints_and_double_rounding():
    """The finalize rounds the exact sum on the conversion units (float32
    truncation with a sticky bit, then one rounding to bf16): exact sums on
    bf16 midpoints, just off them, and wider than 53 bits (where the float64
    rounding of the literal algorithm comes first and may leave a midpoint),
    in four chunks taken as four pieces, with biases that join the integer
    sum, tie with it, or stay too far from its grain."""
    rng = np.random.default_rng(21)
    c = [0.0, 1.0, -1.0, 3.0, -3.0, 1.5, -1.5, 0.5]
    X, W, M, N = _tie_operands(rng, exps=[0, 5, -9, 30, -40], ks=[None, 12, 37, 45, 50], cs=c,
                               hs=[0.0, 1.0, -1.0], K=1024, main_at=0, tie_at=300, tiny_at=900,
                               sigma=0)
    b = np.array([[0.0, 2.0 ** -8, -(2.0 ** -8), 3 * 2.0 ** -9, 2.0 ** -100, 1.0, -1.0][j % 7]
                  for j in range(N)])
    repairs, fixups = check("fwd", bf16(X), bf16(W), bf16(b), M, 1024, N)
    assert repairs == 0 and fixups == 0
    check("fwd", bf16(X), bf16(W), None, M, 1024, N)


def test_output_rounding_at_the_ends_of_the_range():
    """Midpoints at the top of the bf16 range (rounding to inf goes the float64
    way), at the smallest normal exponent, and below it (subnormal results)."""
    rng = np.random.default_rng(22)
    c = [0.0, 1.0, -1.0, 3.0, 1.5]
    X, W, M, N = _tie_operands(rng, exps=[127, 126, -125, -126, -127, -130], ks=[None], cs=c,
                               hs=[0.0], K=40, main_at=0, tie_at=1, tiny_at=2, sigma=6)
    check("fwd", bf16(X), bf16(W), None, M, 40, N)
    b = np.array([[0.0, 1.5 * 2.0 ** 126, -(2.0 ** 127), 2.0 ** -126, -(2.0 ** -133)][j % 5]
                  for j in range(N)])
    check("fwd", bf16(X), bf16(W), bf16(b), M, 40, N)
