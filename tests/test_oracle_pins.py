"""Pins for the CPU oracle against values fixed outside its own code.

Every check compares the oracle with something it does not compute itself:
hand-worked fixtures, closed forms (identity, all-ones, exact row sums), exact
integer arithmetic done by numpy's int64 matmul, exactly rounded sums
(math.fsum), numpy's float64 matmul on tiny shapes, and the classical
error bound of a recursive FMA summation.  A plausible mistake in the oracle
(dropped term, wrong index or leading dimension, transposed operand, unfused
or reordered accumulation, -0 start) fails at least one of them; the
"planted mistake" tests at the end show that for the main ones.
"""
import math
import os

import numpy as np
import pytest

from async_copy_pipelined_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    return rows


def _f32_from_bits(vals):
    return np.array([int(v, 16) for v in vals], dtype=np.uint32).view(np.float32)


# ---------------------------------------------------------------- fixtures

@pytest.mark.parametrize("name", ["int_2x3x2.txt", "int_3x4x2_padded.txt"])
def test_hand_worked_integer_fixtures(orc, name):
    fx = _read_fixture(name)
    M, N, K = (int(fx[k][0][0]) for k in ("M", "N", "K"))
    A = np.array([[float(v) for v in r] for r in fx["A"]], dtype=np.float32)
    B = np.array([[float(v) for v in r] for r in fx["B"]], dtype=np.float32)
    want = np.array([[float(v) for v in r] for r in fx["C"]])
    assert A.shape == (M, int(fx["lda"][0][0]))
    np.testing.assert_array_equal(orc.gemm_f64(A, B, M, N, K), want)
    np.testing.assert_array_equal(orc.gemm_fmaf_chain(A, B, M, N, K), want.astype(np.float32))
    Ab = inputs.f32_to_bf16_bits(A)
    Bb = inputs.f32_to_bf16_bits(B)
    np.testing.assert_array_equal(orc.gemm_bf16_f64(Ab, Bb, M, N, K), want)


@pytest.mark.parametrize("name", ["fma_fused.txt", "fma_order.txt"])
def test_fp32_chain_fixtures(orc, name):
    fx = _read_fixture(name)
    M, N, K = (int(fx[k][0][0]) for k in ("M", "N", "K"))
    A = _f32_from_bits(fx["A_bits"][0]).reshape(M, K)
    B = np.stack([_f32_from_bits(r) for r in fx["B_bits"]]).reshape(K, N)
    got = orc.gemm_fmaf_chain(A, B, M, N, K)
    want_bits = int(fx["C_fmaf_bits"][0][0], 16)
    assert int(got.view(np.uint32)[0, 0]) == want_bits
    got64 = orc.gemm_f64(A, B, M, N, K)
    assert got64[0, 0] == float(fx["C_f64"][0][0])


def test_page4_pattern_golden(orc):
    """Cross-machine pin: the oracle's bits for the day-74 input pattern."""
    import hashlib
    fx = _read_fixture("page4_pattern.txt")
    n = int(fx["N"][0][0])
    a = inputs.matrix_f32("page4a", n, n, 0, 0)
    b = inputs.matrix_f32("page4b", n, n, 0, 0)
    assert hashlib.sha256(a.tobytes()).hexdigest() == fx["a_sha256"][0][0]
    assert hashlib.sha256(b.tobytes()).hexdigest() == fx["b_sha256"][0][0]
    c32 = orc.gemm_fmaf_chain(a, b, n, n, n)
    c64 = orc.gemm_f64(a, b, n, n, n)
    assert hashlib.sha256(c32.tobytes()).hexdigest() == fx["fmaf_sha256"][0][0]
    assert math.fsum(c64.ravel().tolist()) == float(fx["f64_fsum"][0][0])
    for i, j, _, bits, _, f64 in fx["sample"]:
        i, j = int(i), int(j)
        assert int(c32[i, j].view(np.uint32)) == int(bits, 16)
        assert c64[i, j] == float(f64)


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 7, 5), (33, 17, 33), (64, 96, 64)])
def test_identity_left(orc, M, N, K):
    K = M
    A = inputs.matrix_f32("identity", M, K, 0, 0)
    B = inputs.matrix_f32("uniform", K, N, 11, inputs.TAG_B)
    np.testing.assert_array_equal(orc.gemm_f64(A, B, M, N, K), B.astype(np.float64))
    np.testing.assert_array_equal(orc.gemm_fmaf_chain(A, B, M, N, K), B)


@pytest.mark.parametrize("M,N", [(1, 1), (9, 4), (40, 40), (70, 33)])
def test_identity_right(orc, M, N):
    K = N
    A = inputs.matrix_f32("uniform", M, K, 12, inputs.TAG_A, ld=K + 3)
    B = inputs.matrix_f32("identity", K, N, 0, 0)
    np.testing.assert_array_equal(orc.gemm_f64(A, B, M, N, K), A[:, :K].astype(np.float64))
    np.testing.assert_array_equal(orc.gemm_fmaf_chain(A, B, M, N, K), A[:, :K])


@pytest.mark.parametrize("K", [1, 16, 256, 1000])
def test_all_ones(orc, K):
    M, N = 7, 9
    A = inputs.matrix_f32("ones", M, K, 0, 0)
    B = inputs.matrix_f32("ones", K, N, 0, 0)
    np.testing.assert_array_equal(orc.gemm_f64(A, B, M, N, K), np.full((M, N), float(K)))
    np.testing.assert_array_equal(orc.gemm_fmaf_chain(A, B, M, N, K), np.full((M, N), K, np.float32))
    ones16 = inputs.f32_to_bf16_bits(A)
    np.testing.assert_array_equal(
        orc.gemm_bf16_f64(ones16, inputs.f32_to_bf16_bits(B), M, N, K), np.full((M, N), float(K)))


@pytest.mark.parametrize("K", [3, 256, 1000, 4099])
def test_row_sums_exact(orc, K):
    """B = ones: C[i][j] is the exact row sum of A for every j.

    Uniform draws are multiples of 2^-23 in [-1, 1), so every partial sum is a
    multiple of 2^-23 below K in magnitude and exact in float64: the oracle
    must equal math.fsum of the row (an exactly rounded sum) bit for bit.
    """
    M, N = 6, 5
    A = inputs.matrix_f32("uniform", M, K, 3, inputs.TAG_A, ld=K + 1)
    B = inputs.matrix_f32("ones", K, N, 0, 0)
    got = orc.gemm_f64(A, B, M, N, K)
    for i in range(M):
        want = math.fsum(A[i, :K].astype(np.float64).tolist())
        assert np.all(got[i] == want)


def test_column_sums_exact(orc):
    """A = ones: C[i][j] is the exact column sum of B (catches a transposed B)."""
    M, N, K = 4, 37, 300
    A = inputs.matrix_f32("ones", M, K, 0, 0)
    B = inputs.matrix_f32("uniform", K, N, 5, inputs.TAG_B, ld=N + 2)
    got = orc.gemm_f64(A, B, M, N, K)
    for j in range(N):
        want = math.fsum(B[:K, j].astype(np.float64).tolist())
        assert np.all(got[:, j] == want)


# ---------------------------------------------------- exact integer arithmetic

SHAPES = [(1, 1, 1), (2, 3, 5), (15, 16, 17), (31, 33, 63), (64, 65, 127), (129, 63, 16), (3, 5, 1000)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("pad", [0, 1, 3, 4])
def test_smallint_exact_vs_integer_matmul(orc, M, N, K, pad):
    """Entries in {-2..2}: every partial sum is an integer below 2^24, exact in
    float32, float64 and bfloat16 products, in any order; numpy's int64 matmul
    gives the unique right answer."""
    A = inputs.matrix_f32("smallint", M, K, 21, inputs.TAG_A, ld=K + pad)
    B = inputs.matrix_f32("smallint", K, N, 21, inputs.TAG_B, ld=N + pad)
    want = A[:, :K].astype(np.int64) @ B[:, :N].astype(np.int64)
    np.testing.assert_array_equal(orc.gemm_f64(A, B, M, N, K), want.astype(np.float64))
    np.testing.assert_array_equal(orc.gemm_fmaf_chain(A, B, M, N, K), want.astype(np.float32))
    Ab, Bb = inputs.f32_to_bf16_bits(A), inputs.f32_to_bf16_bits(B)
    np.testing.assert_array_equal(orc.gemm_bf16_f64(Ab, Bb, M, N, K), want.astype(np.float64))


# ------------------------------------------------------ floating point pins

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 31, 65), (64, 64, 128)])
def test_f64_exact_for_short_k(orc, M, N, K):
    """For K <= 128 and uniform inputs the float64 sum is exact (products are
    multiples of 2^-46 below 1, sums below 128 need < 53 bits), so the oracle
    equals the exactly rounded sum of the products (math.fsum)."""
    A = inputs.matrix_f32("uniform", M, K, 7, inputs.TAG_A)
    B = inputs.matrix_f32("uniform", K, N, 7, inputs.TAG_B)
    got = orc.gemm_f64(A, B, M, N, K)
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    for i in range(M):
        for j in range(N):
            assert got[i, j] == math.fsum((A64[i, :K] * B64[:K, j]).tolist())


@pytest.mark.parametrize("M,N,K", [(2, 3, 4), (16, 16, 16), (33, 7, 129), (50, 70, 300)])
def test_f64_vs_numpy_matmul(orc, M, N, K):
    A = inputs.matrix_f32("normal", M, K, 8, inputs.TAG_A)
    B = inputs.matrix_f32("normal", K, N, 8, inputs.TAG_B)
    want = A.astype(np.float64) @ B.astype(np.float64)
    got = orc.gemm_f64(A, B, M, N, K)
    scale = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.all(np.abs(got - want) <= 4 * K * 2.0 ** -53 * scale + 1e-300)


@pytest.mark.parametrize("K", [16, 256, 1000, 4096])
def test_fmaf_chain_within_recursive_summation_bound(orc, K):
    """|fl(chain) - exact| <= gamma_K * sum|a_k b_k|, gamma_K = K u / (1 - K u),
    u = 2^-24 (Higham, Accuracy and Stability of Numerical Algorithms, 2nd ed.,
    section 3.1, recursive summation with FMA).  The exact value is the float64
    oracle, itself exact to well below this bound."""
    M, N = 8, 40
    A = inputs.matrix_f32("uniform", M, K, 9, inputs.TAG_A)
    B = inputs.matrix_f32("uniform", K, N, 9, inputs.TAG_B)
    chain = orc.gemm_fmaf_chain(A, B, M, N, K).astype(np.float64)
    exact = orc.gemm_f64(A, B, M, N, K)
    absum = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    assert np.all(np.abs(chain - exact) <= gamma * absum)
    # The library's acceptance bound for FP32, max|C - C_ref| <= 1e-5 * K, holds too.
    assert np.max(np.abs(chain - exact)) <= 1e-5 * K


def test_fmaf_chain_starts_from_plus_zero(orc):
    """(-0) * 1 added to a +0 start gives +0; a -0 start would give -0."""
    A = np.array([[-0.0]], dtype=np.float32)
    B = np.array([[1.0]], dtype=np.float32)
    got = orc.gemm_fmaf_chain(A, B, 1, 1, 1)
    assert int(got.view(np.uint32)[0, 0]) == 0x00000000


def test_fmaf_chain_is_float32_accumulation(orc):
    """The chain rounds to float32 at every step: 1 + 2^-30 (per step) vanishes."""
    K = 5
    A = np.array([[1.0] + [2.0 ** -30] * (K - 1)], dtype=np.float32)
    B = np.ones((K, 1), dtype=np.float32)
    assert orc.gemm_fmaf_chain(A, B, 1, 1, K)[0, 0] == np.float32(1.0)
    assert orc.gemm_f64(A, B, 1, 1, K)[0, 0] == 1.0 + (K - 1) * 2.0 ** -30


# ---------------------------------------------------------------- bfloat16

def test_bf16_widening_exact(orc):
    """bf16 bits 0x3F80 = 1, 0xC000 = -2, 0x3EAB ~ 0.333984375, 0x0001 = 2^-133."""
    vals = np.array([[0x3F80, 0xC000, 0x3EAB, 0x0001]], dtype=np.uint16)
    ident = inputs.f32_to_bf16_bits(np.eye(4, dtype=np.float32))
    got = orc.gemm_bf16_f64(vals, ident, 1, 4, 4)
    np.testing.assert_array_equal(got[0], [1.0, -2.0, 0.333984375, 2.0 ** -133])


@pytest.mark.parametrize("M,N,K", [(3, 4, 5), (32, 48, 64), (17, 9, 300)])
def test_bf16_vs_numpy_on_widened_values(orc, M, N, K):
    A = inputs.matrix_bf16("normal", M, K, 4, inputs.TAG_A, sigma=0.5)
    B = inputs.matrix_bf16("normal", K, N, 4, inputs.TAG_B, sigma=0.5)
    A32, B32 = inputs.bf16_bits_to_f32(A), inputs.bf16_bits_to_f32(B)
    want = A32.astype(np.float64) @ B32.astype(np.float64)
    got = orc.gemm_bf16_f64(A, B, M, N, K)
    scale = np.abs(A32.astype(np.float64)) @ np.abs(B32.astype(np.float64))
    assert np.all(np.abs(got - want) <= 4 * K * 2.0 ** -53 * scale)


# ------------------------------------------------------------- generators

def test_generator_uniform_exact_grid_and_range():
    v = inputs.uniform_values(2, inputs.TAG_A, 1 << 16)
    assert v.min() >= -1.0 and v.max() < 1.0
    scaled = v.astype(np.float64) * 2.0 ** 23
    assert np.all(scaled == np.round(scaled))
    assert abs(float(v.mean())) < 0.02


def test_generator_counter_based_and_chunk_independent():
    a = inputs.draws(5, 1, 0, 1000)
    b = inputs.draws(5, 1, 400, 600)
    np.testing.assert_array_equal(a[400:], b)
    assert not np.array_equal(inputs.draws(5, 2, 0, 10), a[:10])


def test_generator_splitmix64_reference_value():
    """SplitMix64 finaliser on gamma (the first output of the seed-0 stream in
    the published algorithm) is 0xE220A8397B1DCDAF."""
    z = inputs._mix64_int(0x9E3779B97F4A7C15)
    assert z == 0xE220A8397B1DCDAF


def test_generator_padding_is_nan():
    a = inputs.matrix_f32("uniform", 4, 10, 1, 1, ld=13)
    assert np.all(np.isnan(a[:, 10:])) and not np.any(np.isnan(a[:, :10]))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = inputs.normal_values(4, inputs.TAG_A, 1 << 15, 0.5)
    x = np.concatenate([x, np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 65504.0], np.float32)])
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_normal_moments():
    v = inputs.normal_values(3, inputs.TAG_A, 1 << 18, 1.0).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


# ----------------------------------------------------- planted mistakes

# Each mutation plants one plausible mistake in a copy of the oracle's C
# source; the copy is compiled on the CPU and must fail the pin battery.
MUTATIONS = {
    "dropped_last_term": ("for (p = 0; p < K; ++p)", "for (p = 0; p < K - 1; ++p)"),
    "lda_ignored": ("A[i * lda + p]", "A[i * K + p]"),
    "ldb_ignored": ("B + p * ldb;", "B + p * N;"),
    "transposed_b_f64": ("c[j] += a * (double)b[j];", "c[j] += a * (double)B[j * ldb + p];"),
    "unfused_chain": ("c[j] = fmaf(a, b[j], c[j]);", "c[j] = a * b[j] + c[j];"),
    "minus_zero_start": ("c[j] = 0.0f;", "c[j] = -0.0f;"),
    "float_accumulation_f64": ("c[j] += a * (double)b[j];", "c[j] = (float)(c[j] + a * (double)b[j]);"),
    "bf16_wrong_widening": ("(uint32_t)h << 16", "(uint32_t)h << 15"),
    "bf16_dropped_term": ("c[j] += a * (double)bf16_to_float(b[j]);",
                          "if (p + 1 < K) c[j] += a * (double)bf16_to_float(b[j]);"),
}


def _pin_battery(orc, lib):
    """Run the fixture, closed-form and exact-integer pins against ``lib``.
    Returns the names of the pins that fail."""
    failed = []

    def check(name, ok):
        if not ok:
            failed.append(name)

    for fname in ("int_2x3x2.txt", "int_3x4x2_padded.txt"):
        fx = _read_fixture(fname)
        M, N, K = (int(fx[k][0][0]) for k in ("M", "N", "K"))
        A = np.array([[float(v) for v in r] for r in fx["A"]], dtype=np.float32)
        B = np.array([[float(v) for v in r] for r in fx["B"]], dtype=np.float32)
        want = np.array([[float(v) for v in r] for r in fx["C"]])
        check(fname + ":f64", np.array_equal(orc.gemm_f64(A, B, M, N, K, lib=lib), want))
        check(fname + ":fmaf", np.array_equal(orc.gemm_fmaf_chain(A, B, M, N, K, lib=lib), want))
        Ab, Bb = inputs.f32_to_bf16_bits(A), inputs.f32_to_bf16_bits(B)
        check(fname + ":bf16", np.array_equal(orc.gemm_bf16_f64(Ab, Bb, M, N, K, lib=lib), want))
    for fname in ("fma_fused.txt", "fma_order.txt"):
        fx = _read_fixture(fname)
        M, N, K = (int(fx[k][0][0]) for k in ("M", "N", "K"))
        A = _f32_from_bits(fx["A_bits"][0]).reshape(M, K)
        B = np.stack([_f32_from_bits(r) for r in fx["B_bits"]]).reshape(K, N)
        got = orc.gemm_fmaf_chain(A, B, M, N, K, lib=lib)
        check(fname + ":fmaf", int(got.view(np.uint32)[0, 0]) == int(fx["C_fmaf_bits"][0][0], 16))
        check(fname + ":f64", orc.gemm_f64(A, B, M, N, K, lib=lib)[0, 0] == float(fx["C_f64"][0][0]))
    got = orc.gemm_fmaf_chain(np.array([[-0.0]], np.float32), np.array([[1.0]], np.float32), 1, 1, 1, lib=lib)
    check("plus_zero_start", int(got.view(np.uint32)[0, 0]) == 0)
    M, N, K, pad = 15, 17, 33, 3
    A = inputs.matrix_f32("smallint", M, K, 21, inputs.TAG_A, ld=K + pad)
    B = inputs.matrix_f32("smallint", K, N, 21, inputs.TAG_B, ld=N + pad)
    want = (A[:, :K].astype(np.int64) @ B[:, :N].astype(np.int64)).astype(np.float64)
    with np.errstate(invalid="ignore"):
        check("smallint:f64", np.array_equal(orc.gemm_f64(A, B, M, N, K, lib=lib), want))
        check("smallint:fmaf", np.array_equal(orc.gemm_fmaf_chain(A, B, M, N, K, lib=lib), want))
        check("smallint:bf16", np.array_equal(orc.gemm_bf16_f64(
            inputs.f32_to_bf16_bits(A), inputs.f32_to_bf16_bits(B), M, N, K, lib=lib), want))
    K = 300
    A = inputs.matrix_f32("uniform", 3, K, 3, inputs.TAG_A)
    B = inputs.matrix_f32("ones", K, 2, 0, 0)
    got = orc.gemm_f64(A, B, 3, 2, K, lib=lib)
    check("row_sums", all(np.all(got[i] == math.fsum(A[i].astype(np.float64).tolist())) for i in range(3)))
    vals = np.array([[0x3F80, 0xC000, 0x3EAB, 0x0001]], dtype=np.uint16)
    ident = inputs.f32_to_bf16_bits(np.eye(4, dtype=np.float32))
    check("bf16_widening", np.array_equal(orc.gemm_bf16_f64(vals, ident, 1, 4, 4, lib=lib)[0],
                                          [1.0, -2.0, 0.333984375, 2.0 ** -133]))
    return failed


def test_pin_battery_passes_on_the_real_oracle(orc):
    assert _pin_battery(orc, orc._load()) == []


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_pins_catch_planted_mistakes(orc, tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(orc._SRC).read()
    assert old in src, f"mutation anchor for {name} not found in the oracle source"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = orc.load_variant(orc.compile_source(str(mutant), str(tmp_path / f"libmutant_{name}.so")))
    assert _pin_battery(orc, lib), f"planted mistake {name} passed every pin"
