"""Pins for the CPU oracle (no GPU).

The oracle computes the AllReduce-sum of "Every Microsecond Matters", Sec.
III-A: every rank receives the element-wise sum of all ranks' inputs, added in
rank order in the binary32 (binary32/bfloat16 inputs) or binary64 (binary64
inputs) running type, bfloat16 results rounded to nearest-even.

None of these checks re-types the oracle's loop.  Each one fixes the answer by
something else: a closed form, exact integer arithmetic, IEEE rounding worked
by hand, ``math.fsum`` (the correctly rounded sum) with the textbook
recursive-summation error bound, or torch's bfloat16 conversion.  A dropped
term, a wrong sign, a wrong rank order, a wrong running precision or a wrong
tie rule each fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from latency_barrier_free_gb300 import inputs

U32 = 2.0 ** -24  # unit roundoff, binary32
U64 = 2.0 ** -53  # unit roundoff, binary64


def _as_f32(bits_u16):
    return (bits_u16.astype(np.uint32) << 16).view(np.float32)


def _int_round_to_sig_bits(k: int, bits: int) -> int:
    """Round a positive integer to `bits` significant bits, ties to even,
    using integer arithmetic only (independent of any float conversion)."""
    if k == 0:
        return 0
    n = k.bit_length()
    if n <= bits:
        return k
    drop = n - bits
    q, rem = divmod(k, 1 << drop)
    half = 1 << (drop - 1)
    if rem > half or (rem == half and q % 2 == 1):
        q += 1
    return q << drop


@pytest.mark.parametrize("dtype", ["fp32", "fp64"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16, 61, 64])
def test_closed_form_rank_plus_one(n, dtype):
    # sum_{r=0}^{N-1} (r + 1) = N(N+1)/2; every partial sum is an integer
    # below 2^24, so the binary32/binary64 result is exact in any order.
    sends = inputs.rank_plus_one(n, 37, dtype)
    outs = oracle.allreduce(sends, dtype)
    for o in outs:
        assert np.all(o == n * (n + 1) // 2)


@pytest.mark.parametrize("n", [2, 4, 8, 16, 61, 64])
def test_closed_form_bf16(n):
    # Accumulated exactly in binary32, then one rounding to 8 significant bits.
    # N in {2, 4, 8} gives 3, 10, 36 (exact); N = 61 gives 1891 -> 1888.
    sends = inputs.rank_plus_one(n, 19, "bf16")
    outs = oracle.allreduce(sends, "bf16")
    expect = _int_round_to_sig_bits(n * (n + 1) // 2, 8)
    for o in outs:
        assert np.all(_as_f32(o) == expect)
    if n == 61:
        assert expect == 1888


@pytest.mark.parametrize("iteration", [0, 1, 2, 999])
def test_integer_inputs_are_exact(iteration):
    # Workload 1: 32 binary32 integers in [-8, 8] on 2 ranks: sums are exact.
    sends = inputs.workload1(iteration)
    outs = oracle.allreduce(sends, "fp32")
    exact = [int(a) + int(b) for a, b in zip(sends[0].tolist(), sends[1].tolist())]
    for o in outs:
        assert o.tolist() == [float(v) for v in exact]


def test_integer_inputs_many_ranks_exact():
    g = inputs.rng(99, 0)
    sends = inputs.small_integers(g, 64, 1000, "fp32", lo=-1000, hi=1000)
    outs = oracle.allreduce(sends, "fp32")
    exact = np.sum(np.stack([s.astype(np.int64) for s in sends]), axis=0)
    assert np.array_equal(outs[0].astype(np.int64), exact)


def test_rank_order_binary32():
    # 2^24 + 1 is a tie between 2^24 (even significand) and 2^24 + 2, so
    # left-to-right ((2^24 + 1) + 1) stays at 2^24, while (1 + 1) + 2^24
    # reaches 2^24 + 2 exactly.  Fixes the left-to-right rank order.
    big = np.float32(2.0 ** 24)
    one = np.float32(1.0)
    fwd = [np.array([big], np.float32), np.array([one], np.float32), np.array([one], np.float32)]
    rev = [np.array([one], np.float32), np.array([one], np.float32), np.array([big], np.float32)]
    assert oracle.allreduce(fwd, "fp32")[0][0] == 2.0 ** 24
    assert oracle.allreduce(rev, "fp32")[0][0] == 2.0 ** 24 + 2


def test_bf16_accumulates_in_binary32():
    # bfloat16 inputs 256, 1, 1: a binary32 running sum gives 258 (exact in
    # bfloat16, whose spacing at 2^8 is 2); a bfloat16 running sum would
    # round 257 to 256 (tie to even) and end at 256.
    to_bf = lambda v: inputs._bf16_bits_from_f32(np.array([v], np.float32))
    sends = [to_bf(256.0), to_bf(1.0), to_bf(1.0)]
    out = oracle.allreduce(sends, "bf16")[0]
    assert _as_f32(out)[0] == 258.0
    # bfloat16 inputs 2^24, 1, 2^16, 1.  binary32 running sum: 2^24 + 1 ties
    # to 2^24; + 2^16 is exact; + 1 ties to 2^24 + 2^16 (even).  That value is
    # itself a bfloat16 tie (spacing 2^17 at 2^24) and rounds to 2^24.  A
    # binary64 running sum would reach 2^24 + 2^16 + 2, above the tie, and
    # round up to 2^24 + 2^17 instead.
    sends = [to_bf(2.0 ** 24), to_bf(1.0), to_bf(2.0 ** 16), to_bf(1.0)]
    out = oracle.allreduce(sends, "bf16")[0]
    assert _as_f32(out)[0] == 2.0 ** 24


def test_negative_zero():
    # IEEE: (-0) + (-0) = -0 under round-to-nearest.
    for dtype, dt in (("fp32", np.float32), ("fp64", np.float64)):
        sends = [np.array([-0.0, 0.0], dt) for _ in range(3)]
        out = oracle.allreduce(sends, dtype)[0]
        assert np.signbit(out[0]) and not np.signbit(out[1])


@pytest.mark.parametrize("n", [2, 4, 8, 64])
def test_fsum_error_bound_fp32(n):
    # Recursive summation: |computed - exact| <= (N-1) u sum|x| (+ O(u^2)).
    # A dropped term or a sign error is off by |x_p|, far above this bound.
    sends = inputs.normal(inputs.rng(98, n), n, 2000, "fp32")
    got = oracle.allreduce(sends, "fp32")[0].astype(np.float64)
    cols = np.stack([s.astype(np.float64) for s in sends], axis=1)
    exact = np.array([math.fsum(row) for row in cols])
    bound = (n - 1) * U32 * np.abs(cols).sum(axis=1) * (1 + 1e-6)
    assert np.all(np.abs(got - exact) <= bound)
    if n >= 8:
        # the running type really is binary32: some results differ from the
        # correctly rounded binary32 value of the exact sum
        assert np.any(got != exact.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("n", [2, 8, 64])
def test_fsum_error_bound_fp64(n):
    sends = inputs.uniform(inputs.rng(97, n), n, 2000, "fp64")
    got = oracle.allreduce(sends, "fp64")[0]
    cols = np.stack(sends, axis=1)
    exact = np.array([math.fsum(row) for row in cols])
    bound = (n - 1) * U64 * np.abs(cols).sum(axis=1) * (1 + 1e-9)
    assert np.all(np.abs(got - exact) <= bound)


@pytest.mark.parametrize("n", [2, 8, 64])
def test_bf16_one_rounding_of_binary32_sum(n):
    # The binary32 running sum of bf16 values is within (N-1) u32 sum|x| of the
    # exact sum; one final rounding to bfloat16 adds at most half a bf16 ulp.
    sends = inputs.normal(inputs.rng(96, n), n, 3000, "bf16")
    got = _as_f32(oracle.allreduce(sends, "bf16")[0]).astype(np.float64)
    cols = np.stack([_as_f32(s).astype(np.float64) for s in sends], axis=1)
    exact = np.array([math.fsum(row) for row in cols])
    absum = np.abs(cols).sum(axis=1)
    ulp = np.array([2.0 ** (math.frexp(abs(v))[1] - 8) if v != 0 else 0.0 for v in got])
    assert np.all(np.abs(got - exact) <= (n - 1) * U32 * absum + ulp)


def test_reference_sum_against_fsum():
    for dtype in ("fp32", "bf16", "fp64"):
        sends = inputs.normal(inputs.rng(95, 1), 16, 500, dtype)
        s, a = oracle.reference_sum(sends, dtype)
        vals = [(_as_f32(x).astype(np.float64) if dtype == "bf16" else x.astype(np.float64)) for x in sends]
        cols = np.stack(vals, axis=1)
        exact = np.array([math.fsum(row) for row in cols])
        # long double carries at least binary64 precision
        assert np.all(np.abs(s - exact) <= 16 * U64 * np.abs(cols).sum(axis=1))
        assert np.allclose(a, np.abs(cols).sum(axis=1), rtol=1e-15, atol=0)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.Generator(np.random.PCG64(1234))
    bits = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    special = np.array([
        0x00000000, 0x80000000, 0x3F808000, 0x3F818000, 0x3F80FFFF, 0x3F807FFF,  # ties, near-ties
        0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0xFF7FFFFF,                            # overflow edge
        0x7F800000, 0xFF800000, 0x00000001, 0x80000001, 0x00008000, 0x00018000,    # inf, subnormals
        0x007FFFFF, 0x00800000,
    ], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    f = bits.view(np.float32)
    ours = oracle.f32_to_bf16(f)
    theirs = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], theirs[~nan])
    # NaN stays NaN (quiet bit set), sign kept
    o = ours[nan].astype(np.uint32)
    assert np.all((o & 0x7F80) == 0x7F80) and np.all((o & 0x007F) != 0)
    assert np.array_equal(o >> 15, (bits[nan] >> 31))


def test_all_ranks_identical_and_in_place():
    sends = inputs.normal(inputs.rng(94, 0), 8, 1001, "fp32")
    outs = oracle.allreduce(sends, "fp32")
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    inplace = [s.copy() for s in sends]
    oracle.allreduce(inplace, "fp32", recvs=inplace)
    for o in inplace:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_scaling_by_two_is_exact():
    # Multiplying every input by 2 scales every partial sum by 2 exactly.
    sends = inputs.normal(inputs.rng(93, 0), 16, 3000, "fp32")
    a = oracle.allreduce(sends, "fp32")[0]
    b = oracle.allreduce([(s * np.float32(2)).astype(np.float32) for s in sends], "fp32")[0]
    assert np.array_equal(b, a * np.float32(2))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_threaded_equals_single(dtype):
    sends = inputs.normal(inputs.rng(92, 0), 8, 10007, dtype)
    a = oracle.allreduce(sends, dtype)
    for nt in (1, 3, 8, 64):
        b = oracle.allreduce_mt(sends, dtype, nt)
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_empty_and_ragged():
    assert [o.size for o in oracle.allreduce([np.zeros(0, np.float32)] * 3, "fp32")] == [0, 0, 0]
    with pytest.raises(ValueError):
        oracle.allreduce([np.zeros(3, np.float32), np.zeros(4, np.float32)], "fp32")


# ------------------------------------------------ the other collectives ----
# Definitions (paper text, Sec. III-A opening; review summary): ReduceScatter
# leaves block r of the rank-order sum in rank r; AllGather concatenates the
# inputs in rank order; Broadcast copies the root's input; Reduce leaves the
# sum in the root only.
def _blocked(n, count, dtype):
    """send[p][r*count + i] = 32 r + 4 p + (i mod 4): integers up to 255, exact
    in bfloat16 too, so every binary32 sum below is exact, and a swapped
    block/rank index changes the result (N <= 8)."""
    np_dt = oracle.DTYPES[dtype][1]
    i = np.arange(count)
    out = []
    for p in range(n):
        v = np.concatenate([32.0 * r + 4.0 * p + (i % 4) for r in range(n)])
        out.append(oracle.f32_to_bf16(v) if dtype == "bf16" else v.astype(np_dt))
    return out


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_reduce_scatter_closed_form(n, dtype):
    count = 11
    outs = oracle.reduce_scatter(_blocked(n, count, dtype), dtype)
    i = np.arange(count)
    for r in range(n):
        expect = n * 32.0 * r + 4.0 * n * (n - 1) / 2 + n * (i % 4)
        got = _as_f32(outs[r]) if dtype == "bf16" else outs[r]
        if dtype == "bf16":  # one rounding of the exact integer to 8 significant bits
            expect = np.array([_int_round_to_sig_bits(int(e), 8) for e in expect], dtype=np.float64)
        assert np.array_equal(got.astype(np.float64), expect), r


def test_reduce_scatter_rank_order():
    # block 1 of three ranks holds 2^24, 1, 1: adding in rank order gives 2^24
    # (each +1 is a tie that rounds to even), the reverse order 2^24 + 2.
    big = np.float32(2.0 ** 24)
    sends = [np.array([0, big], np.float32), np.array([0, 1], np.float32), np.array([0, 1], np.float32)]
    sends = [np.concatenate([s, s, s])[:6] for s in sends]  # N*count = 6, count = 2
    outs = oracle.reduce_scatter(sends, "fp32")
    assert outs[0][1] == big  # rank order; the reverse order would give 2^24 + 2
    rev = oracle.reduce_scatter(sends[::-1], "fp32")
    assert rev[0][1] == big + 2


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
@pytest.mark.parametrize("n", [1, 2, 5])
def test_all_gather_layout(n, dtype):
    count = 9
    np_dt = oracle.DTYPES[dtype][1]
    sends = [(100 * p + np.arange(count)).astype(np_dt) for p in range(n)]
    outs = oracle.all_gather(sends, dtype)
    k = np.arange(n * count)
    for r in range(n):
        assert np.array_equal(outs[r], (100 * (k // count) + k % count).astype(np_dt))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_broadcast_copies_root_only(dtype):
    n, count = 4, 13
    np_dt = oracle.DTYPES[dtype][1]
    sends = [(1000 * p + np.arange(count)).astype(np_dt) for p in range(n)]
    for root in range(n):
        outs = oracle.broadcast(sends, dtype, root)
        for r in range(n):
            assert np.array_equal(outs[r], (1000 * root + np.arange(count)).astype(np_dt))


@pytest.mark.parametrize("dtype", ["fp32", "fp64"])
def test_reduce_to_root_leaves_others(dtype):
    n, count = 6, 17
    np_dt = oracle.DTYPES[dtype][1]
    sends = inputs.rank_plus_one(n, count, dtype)
    for root in (0, 3, 5):
        recvs = [np.full(count, -7, dtype=np_dt) for _ in range(n)]
        oracle.reduce(sends, dtype, root, recvs)
        for r in range(n):
            expect = n * (n + 1) // 2 if r == root else -7
            assert np.all(recvs[r] == expect)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_allgather_of_reducescatter_is_allreduce(dtype):
    # Element by element both sides are the same rank-order sum, so the
    # identity holds bit for bit; an index slip in either function breaks it.
    # The AllReduce side is pinned by the tests above.
    n, count = 5, 23
    g = inputs.rng(90, 0)
    sends = inputs.normal(g, n, n * count, dtype)
    ag = oracle.all_gather(oracle.reduce_scatter(sends, dtype), dtype)
    ar = oracle.allreduce(sends, dtype)
    for r in range(n):
        assert np.array_equal(ag[r].view(np.uint8), ar[r].view(np.uint8))
    red = oracle.reduce(sends, dtype, 2)
    assert np.array_equal(red[2].view(np.uint8), ar[0].view(np.uint8))


# ------------------------------------------- AllReduce + residual add ----
# recv[r] = round(sum_p x_p + res[r]): the residual joins the running value
# after the rank-order sum, and bfloat16 is rounded once at the end.
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_residual_closed_form(dtype):
    n, count = 6, 19
    sends = inputs.rank_plus_one(n, count, dtype)
    np_dt = oracle.DTYPES[dtype][1]
    res = []
    for r in range(n):
        v = np.full(count, 2.0 * r, dtype=np.float64)
        res.append(oracle.f32_to_bf16(v) if dtype == "bf16" else v.astype(np_dt))
    outs = oracle.allreduce_residual(sends, res, dtype)
    for r in range(n):
        got = _as_f32(outs[r]) if dtype == "bf16" else outs[r]
        assert np.all(got == n * (n + 1) // 2 + 2 * r), r  # integers below 256: exact


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_residual_zero_is_allreduce(dtype):
    n, count = 5, 31
    sends = inputs.normal(inputs.rng(91, 0), n, count, dtype)
    zeros = [np.zeros(count, dtype=oracle.DTYPES[dtype][1]) for _ in range(n)]
    outs = oracle.allreduce_residual(sends, zeros, dtype)
    ar = oracle.allreduce(sends, dtype)
    for a, b in zip(outs, ar):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_residual_added_after_the_sum():
    # x = (2^24, 1), res = 1: the sum rounds 2^24 + 1 to 2^24 (tie to even),
    # then + 1 rounds again to 2^24; adding the residual first would give
    # 2^24 + 2.
    big = np.float32(2.0 ** 24)
    sends = [np.array([big], np.float32), np.array([1], np.float32)]
    res = [np.array([1], np.float32)] * 2
    outs = oracle.allreduce_residual(sends, res, "fp32")
    assert outs[0][0] == big and outs[1][0] == big


def test_residual_bf16_rounds_once():
    # 256 + 1 + residual 1 = 258 exactly in binary32, one rounding -> 258.
    # Rounding the AllReduce to bfloat16 first (257 -> 256, ties to even)
    # and adding the residual after (257 -> 256) would give 256.
    sends = [oracle.f32_to_bf16(np.array([256.0])), oracle.f32_to_bf16(np.array([1.0]))]
    res = [oracle.f32_to_bf16(np.array([1.0]))] * 2
    outs = oracle.allreduce_residual(sends, res, "bf16")
    assert _as_f32(outs[0])[0] == 258.0 and _as_f32(outs[1])[0] == 258.0
