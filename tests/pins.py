"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an oracle instance (``oracle.Oracle``) and raises
``AssertionError`` on a mismatch.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutations.py`` runs them on copies of the oracle
with a planted mistake and requires that at least one fails.

What the pins rest on (none of it is the oracle's own code):
  * the storage formats' definitions, through numpy's float16 / float32 casts,
    torch's bfloat16 decode, and exact rational rounding (``fractions``);
  * closed forms of the normalisation (constant row, unit weight, scale
    invariance at eps = 0, one-element rows);
  * a worked example of the fixed binary32 summation order;
  * exact integer sums;
  * brute force on tiny rows in exact rational / 50-digit decimal arithmetic;
  * for the 8-bit output, torch's float8 decoders and casts and a brute-force
    nearest search over the code table;
  * for the GEMM producer, numpy's binary64 matrix product, the identity
    weight (reduces to the fused form), a constructed single-rounding case and
    exact rational brute force;
  * for the 8-bit partials, the pinned reduce over the same values (power-of-
    two scales, torch's float8 decoders) and exact rational brute force;
  * for the tensor-parallel form, the pinned reduce over the ranks' stacked
    partials, a worked example of the rank order, and the properties a
    partition of the rows into contiguous rank blocks must have.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

# ---------------------------------------------------------------------------
# Storage formats, from the library decoders
# ---------------------------------------------------------------------------

FORMATS = {  # precision p, emin, emax
    "f32": (24, -126, 127),
    "f16": (11, -14, 15),
    "bf16": (8, -126, 127),
}


def lib_decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode storage bits with numpy / torch (not the oracle)."""
    if dtype == "f32":
        return np.asarray(bits, np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)
    import torch
    t = torch.from_numpy(np.asarray(bits, np.uint16).astype(np.int16).copy())
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def rn_exact(v: Fraction, dtype: str) -> float:
    """Round an exact rational to the storage format: nearest, ties to even,
    overflow to infinity.  Exact rational arithmetic throughout; Python's
    ``round`` on a Fraction rounds half to even."""
    p, emin, emax = FORMATS[dtype]
    if v == 0:
        return 0.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    q = e - (p - 1)
    n = round(a / Fraction(2) ** q)
    r = Fraction(n) * Fraction(2) ** q
    max_finite = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    out = math.inf if r > max_finite else float(r)
    return out if v > 0 else -out


def bits_of(values: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bits of values that are exactly representable (library casts)."""
    values = np.asarray(values, np.float64)
    if dtype == "f32":
        return values.astype(np.float32)
    if dtype == "f16":
        return values.astype(np.float16).view(np.uint16)
    import torch
    t = torch.from_numpy(values.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def ulp_dist(a_bits: np.ndarray, b_bits: np.ndarray, dtype: str) -> np.ndarray:
    """Distance in units in the last place between two arrays of storage bits."""
    if dtype == "f32":
        a = np.asarray(a_bits, np.float32).view(np.int32).astype(np.int64)
        b = np.asarray(b_bits, np.float32).view(np.int32).astype(np.int64)
        sign = 1 << 31
    else:
        a = np.asarray(a_bits, np.uint16).astype(np.int64)
        b = np.asarray(b_bits, np.uint16).astype(np.int64)
        sign = 1 << 15
    a = np.where(a & sign, -(a & (sign - 1)), a & (sign - 1))
    b = np.where(b & sign, -(b & (sign - 1)), b & (sign - 1))
    return np.abs(a - b)


# ---------------------------------------------------------------------------
# Pins on the format code
# ---------------------------------------------------------------------------

def pin_decode_all_patterns(O):
    """Every f16 / bf16 bit pattern decodes as numpy / torch decode it."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in ("f16", "bf16"):
        got = O.decode(allbits, dt)
        want = lib_decode(allbits, dt)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), dt
        assert np.array_equal(got[~nan], want[~nan]), dt
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan])), dt


def _rounding_probe(dtype, rng, n=20000):
    """Doubles that stress rounding: random magnitudes across the whole range
    of the format (subnormals and overflow included) plus exact midpoints."""
    p, emin, emax = FORMATS[dtype]
    e = rng.integers(emin - p - 2, emax + 2, size=n)
    m = rng.random(n) + 1.0
    v = np.ldexp(m, e) * np.where(rng.random(n) < 0.5, -1.0, 1.0)
    # exact midpoints between neighbours: (2k + 1) * 2^(q-1)
    k = rng.integers(1 << (p - 1), 1 << p, size=n // 4)
    q = rng.integers(emin - (p - 1), emax - (p - 1) + 1, size=n // 4)
    mids = np.ldexp(2.0 * k + 1.0, q - 1)
    # midpoints in the subnormal range and at the overflow threshold
    sub = np.ldexp(2.0 * rng.integers(0, 1 << (p - 1), size=64) + 1.0, emin - (p - 1) - 1)
    maxf = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    edge = np.array([maxf, maxf + 2.0 ** (emax - p), maxf + 2.0 ** (emax - p) * 0.999,
                     np.nextafter(maxf + 2.0 ** (emax - p), 0), 2.0 ** (emin - p),
                     2.0 ** (emin - p) * 1.0001, 2.0 ** (emin - p) * 0.9999, 0.0, -0.0])
    return np.concatenate([v, mids, -mids, sub, edge, -edge])


def pin_round_matches_library(O):
    """One rounding double -> f16 / f32 equals numpy's cast (both round once,
    to nearest, ties to even)."""
    rng = np.random.default_rng(1)
    for dt, np_t in (("f16", np.float16), ("f32", np.float32)):
        v = _rounding_probe(dt, rng)
        with np.errstate(over="ignore"):
            want = v.astype(np_t)
        got = O.round_to(v, dt)
        if dt == "f16":
            assert np.array_equal(got, want.view(np.uint16)), dt
        else:
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), dt


def pin_round_bf16_nearest(O):
    """One rounding double -> bf16 picks the nearest bf16 value, ties to the
    even pattern, overflow to infinity: brute force over the table of every
    finite bf16 value, decoded by torch."""
    allbits = np.arange(0, 0x7F80, dtype=np.uint16)  # +0 .. largest finite
    table = lib_decode(allbits, "bf16")
    rng = np.random.default_rng(2)
    v = _rounding_probe("bf16", rng, n=8000)
    got = O.round_to(v, "bf16")
    a = np.abs(v)
    i = np.clip(np.searchsorted(table, a), 1, len(table) - 1)
    lo, hi = table[i - 1], table[i]
    below = a - lo
    above = hi - a
    pick = np.where(below < above, i - 1, i)
    tie = below == above
    pick = np.where(tie & ((i - 1) % 2 == 0), i - 1, pick)
    res = allbits[pick].astype(np.uint32)
    maxf = table[-1]
    half_ulp = (table[-1] - table[-2]) / 2
    res = np.where(a > maxf, 0x7F7F, res)               # between max and the midpoint
    res = np.where(a >= maxf + half_ulp, 0x7F80, res)  # at or past it: infinity
    res = np.where(np.signbit(v), res | 0x8000, res).astype(np.uint16)
    assert np.array_equal(got, res)


def pin_round_exact_rationals(O):
    """Hand-checked ties: the exact midpoint between two neighbours goes to
    the even one."""
    cases = {
        # bf16 has 8 significant bits: neighbours of 1 are 1 and 1 + 2^-7
        "bf16": [(1 + 2.0 ** -8, 1.0), (1 + 3 * 2.0 ** -8, 1 + 2.0 ** -6),
                 (1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -7)],
        # f16 has 11 significant bits
        "f16": [(1 + 2.0 ** -11, 1.0), (1 + 3 * 2.0 ** -11, 1 + 2.0 ** -9),
                (65520.0, math.inf), (65519.99, 65504.0), (2.0 ** -25, 0.0),
                (3 * 2.0 ** -26, 2.0 ** -24)],
        "f32": [(1 + 2.0 ** -24, 1.0), (1 + 3 * 2.0 ** -24, 1 + 2.0 ** -22)],
    }
    for dt, pairs in cases.items():
        v = np.array([a for a, _ in pairs])
        got = O.decode(O.round_to(v, dt), dt)
        want = np.array([b for _, b in pairs])
        assert np.array_equal(got, want), (dt, got, want)
        for a, b in pairs:
            assert rn_exact(Fraction(a), dt) == b, (dt, a)


# ---------------------------------------------------------------------------
# Pins on the residual (step 1)
# ---------------------------------------------------------------------------

def _rand_bits(rng, shape, dtype, scale=1.0):
    v = rng.standard_normal(shape) * scale
    return bits_of(v.astype(np.float32).astype(np.float64), dtype)


def pin_fused_residual_is_exact_rounded_sum(O):
    """R = 1: the stored residual is the exact sum x + r rounded once
    (for f16 / bf16 the binary32 add of two such values never double-rounds)."""
    rng = np.random.default_rng(3)
    for dt in ("bf16", "f16", "f32"):
        T, H = 4, 257
        x = _rand_bits(rng, (T, H), dt)
        r = _rand_bits(rng, (T, H), dt, scale=3.0)
        g = bits_of(np.ones(H), dt)
        res = O.fused_add_rms_norm(x, r, g, 1e-6, dt)
        xv, rv = lib_decode(x, dt).ravel(), lib_decode(r, dt).ravel()
        want = np.array([rn_exact(Fraction(a) + Fraction(b), dt) for a, b in zip(xv, rv)])
        got = lib_decode(res.residual, dt).ravel()
        assert np.array_equal(got, want), dt


def pin_reduce_order_worked_example(O):
    """Worked example of the fixed order: partials (2^24, 1, -2^24) and
    residual 0.  In binary32, 2^24 + 1 rounds back to 2^24 (tie to even), so
    the sequential sum is exactly 0; the exact sum is 1, and any other order
    that adds 1 last, or a wider accumulator, gives 1."""
    for dt in ("bf16", "f32"):  # 2^24 overflows binary16
        H = 3
        p = np.stack([bits_of(np.full((1, H), v), dt) for v in (2.0 ** 24, 1.0, -(2.0 ** 24))])
        r = bits_of(np.zeros((1, H)), dt)
        g = bits_of(np.ones(H), dt)
        res = O.reduce_add_rms_norm(p, r, g, 1e-6, dt)
        assert np.all(lib_decode(res.residual, dt) == 0.0), dt
    # One final rounding, not one per add: partials (2^11, 1, 1) in f16 and
    # (2^8, 1, 1) in bf16.  binary32 holds 2^k + 2 exactly and it is
    # representable in the storage type; rounding after every add would
    # lose each 1 to a tie-to-even and give 2^k.
    for dt, big in (("f16", 2048.0), ("bf16", 256.0)):
        p = np.stack([bits_of(np.full((1, 2), v), dt) for v in (big, 1.0, 1.0)])
        r = bits_of(np.zeros((1, 2)), dt)
        res = O.reduce_add_rms_norm(p, r, bits_of(np.ones(2), dt), 1e-6, dt)
        assert np.all(lib_decode(res.residual, dt) == big + 2.0), dt
        # and the final rounding itself ties to even: 2^k + 1 -> 2^k
        p1 = np.stack([bits_of(np.full((1, 2), v), dt) for v in (big, 1.0)])
        res1 = O.reduce_add_rms_norm(p1, r, bits_of(np.ones(2), dt), 1e-6, dt)
        assert np.all(lib_decode(res1.residual, dt) == big), dt


def pin_reduce_integer_sums(O):
    """Small integers add exactly in every order: the residual is the plain
    integer sum of all partials and the residual, per element."""
    rng = np.random.default_rng(4)
    for dt in ("bf16", "f16", "f32"):
        R, T, H = 8, 3, 67
        pi = rng.integers(-12, 13, size=(R, T, H))
        ri = rng.integers(-12, 13, size=(T, H))
        p = bits_of(pi.astype(np.float64), dt).reshape(R, T, H)
        r = bits_of(ri.astype(np.float64), dt)
        res = O.reduce_add_rms_norm(p, r, bits_of(np.ones(H), dt), 1e-6, dt)
        want = (pi.sum(0) + ri).astype(np.float64)
        assert np.array_equal(lib_decode(res.residual, dt), want), dt


def pin_reduce_brute_force_binary32(O):
    """Tiny random reduce problems: the residual equals the sequential
    binary32 sum p0 + p1 + ... + p{R-1} + r, each add rounded to binary32 in
    exact rational arithmetic, then one rounding to the storage type."""
    rng = np.random.default_rng(5)
    for dt in ("bf16", "f16", "f32"):
        for R in (2, 3, 8):
            T, H = 2, 9
            scales = rng.choice([1e-3, 1.0, 300.0], size=R)
            p = np.stack([_rand_bits(rng, (T, H), dt, s) for s in scales])
            r = _rand_bits(rng, (T, H), dt)
            res = O.reduce_add_rms_norm(p, r, bits_of(np.ones(H), dt), 1e-6, dt)
            pv = lib_decode(p, dt)
            rv = lib_decode(r, dt)
            want = np.empty((T, H))
            for t in range(T):
                for i in range(H):
                    acc = Fraction(pv[0, t, i])
                    for k in range(1, R):
                        acc = Fraction(rn_exact(acc + Fraction(pv[k, t, i]), "f32"))
                    acc = Fraction(rn_exact(acc + Fraction(rv[t, i]), "f32"))
                    want[t, i] = rn_exact(acc, dt)
            assert np.array_equal(lib_decode(res.residual, dt), want), (dt, R)


def pin_reduce_special_cases(O):
    """reduce with partials (x, 0, ..., 0) equals fused(x); reduce with R = 1
    equals fused; fused with a zero residual equals plain."""
    rng = np.random.default_rng(6)
    for dt in ("bf16", "f16", "f32"):
        T, H = 5, 130
        x = _rand_bits(rng, (T, H), dt)
        r = _rand_bits(rng, (T, H), dt)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        zero = bits_of(np.zeros((T, H)), dt)
        f = O.fused_add_rms_norm(x, r, g, 1e-5, dt)
        red = O.reduce_add_rms_norm(np.stack([x] + [zero] * 3), r, g, 1e-5, dt)
        red1 = O.reduce_add_rms_norm(x[None], r, g, 1e-5, dt)
        for other in (red, red1):
            assert np.array_equal(other.y, f.y), dt
            assert np.array_equal(other.residual, f.residual), dt
        plain = O.rms_norm(x, g, 1e-5, dt)
        fz = O.fused_add_rms_norm(x, zero, g, 1e-5, dt)
        assert np.array_equal(plain.y, fz.y), dt
        assert np.array_equal(fz.residual, x), dt


# ---------------------------------------------------------------------------
# Pins on the normalisation (steps 2-4)
# ---------------------------------------------------------------------------

def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-300))


def pin_constant_row(O):
    """A row of constant c gives y_i = c / sqrt(c^2 + eps) * gamma_i."""
    getcontext().prec = 50
    for dt in ("f32", "f16", "bf16"):
        for c, eps in ((3.0, 1e-6), (0.015625, 0.25), (-2.5, 1e-5), (1.0, 1.0), (0.0078125, 0.0)):
            H = 96
            x = bits_of(np.full((1, H), c), dt)
            gv = np.linspace(0.5, 1.5, H)
            g = bits_of(gv, dt)
            gd = lib_decode(g, dt)
            e32 = float(np.float32(eps))
            res = O.rms_norm(x, g, eps, dt, want_y64=True)
            k = Decimal(c) / (Decimal(c) * Decimal(c) + Decimal(e32)).sqrt()
            want = np.array([float(k * Decimal(gi)) for gi in gd])
            assert _rel(res.y64[0], want) < 1e-14, (dt, c, eps)
            inv = 1 / (Decimal(c) * Decimal(c) + Decimal(e32)).sqrt()
            assert abs(res.inv[0] - float(inv)) <= 1e-15 * float(inv), (dt, c, eps)


def pin_unit_gamma_rms(O):
    """With gamma = 1 the output's mean square is ms / (ms + eps), ms being the
    input's mean square (exact rational)."""
    rng = np.random.default_rng(7)
    for dt in ("f32", "f16", "bf16"):
        for eps in (1e-6, 0.5):
            T, H = 3, 200
            x = _rand_bits(rng, (T, H), dt, scale=0.7)
            g = bits_of(np.ones(H), dt)
            res = O.rms_norm(x, g, eps, dt, want_y64=True)
            xv = lib_decode(x, dt)
            e32 = Fraction(float(np.float32(eps)))
            for t in range(T):
                ms = sum(Fraction(v) ** 2 for v in xv[t]) / H
                want = float(ms / (ms + e32))
                got = float(np.mean(res.y64[t] ** 2))
                assert abs(got - want) <= 1e-13 * want, (dt, eps, t)


def pin_scale_invariance(O):
    """eps = 0: scaling the row by a power of two changes nothing; scaling an
    f32 row by 3 changes y only by binary64 rounding."""
    rng = np.random.default_rng(8)
    for dt, k in (("f32", 2.0 ** 10), ("f16", 4.0), ("bf16", 2.0 ** -20), ("bf16", 2.0 ** 30)):
        T, H = 4, 123
        xv = lib_decode(_rand_bits(rng, (T, H), dt), dt)
        x = bits_of(xv, dt)
        xk = bits_of(xv * k, dt)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        a = O.rms_norm(x, g, 0.0, dt, want_y64=True)
        b = O.rms_norm(xk, g, 0.0, dt, want_y64=True)
        assert np.array_equal(a.y, b.y), (dt, k)
        assert np.allclose(a.inv, b.inv * k, rtol=1e-15, atol=0), (dt, k)
    # values with 8 significant bits, so that 3x is exact in binary32
    xv = lib_decode(_rand_bits(rng, (2, 50), "bf16"), "bf16")
    g = bits_of(np.ones(50), "f32")
    a = O.rms_norm(bits_of(xv, "f32"), g, 0.0, "f32", want_y64=True)
    b = O.rms_norm(bits_of(xv * 3.0, "f32"), g, 0.0, "f32", want_y64=True)
    assert _rel(a.y64, b.y64) < 1e-14


def pin_single_element_rows(O):
    """H = 1: y = x / sqrt(x^2 + eps) * gamma."""
    getcontext().prec = 50
    rng = np.random.default_rng(9)
    for dt in ("f32", "f16", "bf16"):
        x = _rand_bits(rng, (32, 1), dt, scale=2.0)
        g = bits_of(np.array([1.25]), dt)
        res = O.rms_norm(x, g, 1e-3, dt, want_y64=True)
        xv = lib_decode(x, dt)[:, 0]
        e32 = Decimal(float(np.float32(1e-3)))
        want = np.array([float(Decimal(v) / (Decimal(v) ** 2 + e32).sqrt() * Decimal(1.25))
                         for v in xv])
        assert _rel(res.y64[:, 0], want) < 1e-14, dt


def pin_brute_force_tiny(O):
    """Tiny fused problems against a from-scratch computation: exact rational
    residual and sum of squares, 50-digit square root, exact rounding of y."""
    getcontext().prec = 50
    rng = np.random.default_rng(10)
    for dt in ("f32", "f16", "bf16"):
        T, H = 3, 11
        x = _rand_bits(rng, (T, H), dt)
        r = _rand_bits(rng, (T, H), dt, scale=0.5)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        eps = 1e-2
        res = O.fused_add_rms_norm(x, r, g, eps, dt, want_y64=True)
        xv, rv, gv = lib_decode(x, dt), lib_decode(r, dt), lib_decode(g, dt)
        e32 = Fraction(float(np.float32(eps)))
        for t in range(T):
            h = [Fraction(rn_exact(Fraction(xv[t, i]) + Fraction(rv[t, i]), dt)) for i in range(H)]
            ss = sum(v * v for v in h)
            m = ss / H + e32
            inv = 1 / (Decimal(m.numerator) / Decimal(m.denominator)).sqrt()
            assert abs(res.inv[t] - float(inv)) <= 1e-15 * float(inv), (dt, t)
            yd = [Decimal(h[i].numerator) / Decimal(h[i].denominator) * inv * Decimal(gv[i])
                  for i in range(H)]
            want64 = np.array([float(v) for v in yd])
            assert _rel(res.y64[t], want64) < 1e-14, (dt, t)
            # the stored output is the one rounding of that value (away from
            # exact ties, which random data does not hit)
            want_bits = np.array([rn_exact(Fraction(v), dt) for v in want64])
            assert np.array_equal(lib_decode(res.y[t], dt), want_bits), (dt, t)


# ---------------------------------------------------------------------------
# Pins on the general form: row strides and an fp32 residual
# ---------------------------------------------------------------------------

GARBAGE = {"f32": np.float32(-1234.5), "f16": np.uint16(0x7BFF), "bf16": np.uint16(0x4B4B)}


def _strided(dense, ld, dtype, extra=0):
    """Copy [T, H] storage into a flat buffer with row stride ld, the padding
    (and `extra` trailing elements) filled with a garbage pattern."""
    T, H = dense.shape
    buf = np.full(T * ld + extra, GARBAGE[dtype], dtype=dense.dtype)
    view = buf[:T * ld].reshape(T, ld)
    view[:, :H] = dense
    return buf


def _rows(buf, T, ld, H):
    return buf[:T * ld].reshape(T, ld)[:, :H]


def pin_strided_equals_dense(O):
    """Rows with a stride larger than H (padding holding garbage) give the
    dense results, and nothing outside the first H elements of each row of y
    or of the residual is written."""
    rng = np.random.default_rng(11)
    for dt in ("f32", "bf16", "f16"):
        for R in (0, 1, 3):
            T, H, ldx, ldr, ldy = 5, 37, 45, 41, 50
            n = max(R, 1)
            parts = np.stack([_rand_bits(rng, (T, H), dt) for _ in range(n)])
            res = _rand_bits(rng, (T, H), dt)
            g = bits_of(rng.uniform(0.5, 1.5, H), dt)
            slice_ = T * ldx + 3
            X = np.concatenate([_strided(parts[r], ldx, dt, extra=3) for r in range(n)])
            Rb = _strided(res, ldr, dt)
            Y = np.full(T * ldy, GARBAGE[dt], dtype=parts.dtype)
            r_ex = O.rows_ex(dt, dt, T, H, R, X, ldx, slice_, Rb if R else None, ldr, g, 1e-5,
                             Y, ldy)
            if R == 0:
                want = O.rms_norm(parts[0], g, 1e-5, dt)
            elif R == 1:
                want = O.fused_add_rms_norm(parts[0], res, g, 1e-5, dt)
            else:
                want = O.reduce_add_rms_norm(parts, res, g, 1e-5, dt)
            assert np.array_equal(_rows(Y, T, ldy, H), want.y), (dt, R)
            pad_y = Y[:T * ldy].reshape(T, ldy)[:, H:]
            assert np.array_equal(pad_y, np.full_like(pad_y, GARBAGE[dt])), (dt, R)
            if R:
                assert np.array_equal(_rows(Rb, T, ldr, H), want.residual), (dt, R)
                pad_r = Rb.reshape(T, ldr)[:, H:]
                assert np.array_equal(pad_r, np.full_like(pad_r, GARBAGE[dt])), (dt, R)


def pin_fp32_residual_sum(O):
    """An fp32 residual with 16-bit inputs: the stored residual is the binary32
    sequential sum itself, with no rounding to 16 bits (exact rational
    emulation of every add), and inv / y64 follow from that binary32 row."""
    getcontext().prec = 50
    rng = np.random.default_rng(12)
    for dt in ("bf16", "f16"):
        for R in (1, 3):
            T, H = 3, 17
            parts = np.stack([_rand_bits(rng, (T, H), dt) for _ in range(R)])
            res = (rng.standard_normal((T, H)) * 0.37).astype(np.float32)  # not 16-bit values
            g = bits_of(rng.uniform(0.5, 1.5, H), dt)
            X = parts.reshape(-1).copy()
            Rb = res.reshape(-1).copy()
            Y = np.zeros(T * H, parts.dtype)
            out = O.rows_ex(dt, "f32", T, H, R, X, H, T * H, Rb, H, g, 1e-3, Y, H, want_y64=True)
            pv = lib_decode(parts, dt)
            gv = lib_decode(g, dt)
            e32 = Fraction(float(np.float32(1e-3)))
            for t in range(T):
                h = []
                for i in range(H):
                    acc = Fraction(pv[0, t, i])
                    for k in range(1, R):
                        acc = Fraction(rn_exact(acc + Fraction(pv[k, t, i]), "f32"))
                    acc = Fraction(rn_exact(acc + Fraction(float(res[t, i])), "f32"))
                    h.append(acc)
                got = out.residual.reshape(T, H)[t].astype(np.float64)
                assert np.array_equal(got, np.array([float(v) for v in h])), (dt, R, t)
                m = sum(v * v for v in h) / H + e32
                inv = 1 / (Decimal(m.numerator) / Decimal(m.denominator)).sqrt()
                assert abs(out.inv[t] - float(inv)) <= 1e-15 * float(inv), (dt, R, t)
                want = np.array([float(Decimal(v.numerator) / Decimal(v.denominator) * inv *
                                       Decimal(gv[i])) for i, v in enumerate(h)])
                assert _rel(out.y64[t], want) < 1e-14, (dt, R, t)


def pin_fp32_residual_matches_16bit_when_exact(O):
    """Integer data whose sums stay exactly representable in 16 bits: an fp32
    residual and a 16-bit residual give identical y and identical residual
    values."""
    rng = np.random.default_rng(13)
    for dt in ("bf16", "f16"):
        R, T, H = 4, 3, 29
        pi = rng.integers(-8, 9, size=(R, T, H)).astype(np.float64)
        ri = rng.integers(-8, 9, size=(T, H)).astype(np.float64)
        parts = bits_of(pi, dt).reshape(R, T, H)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        same = O.reduce_add_rms_norm(parts, bits_of(ri, dt), g, 1e-6, dt)
        Rb = ri.astype(np.float32).reshape(-1).copy()
        Y = np.zeros(T * H, parts.dtype)
        mixed = O.rows_ex(dt, "f32", T, H, R, parts.reshape(-1).copy(), H, T * H, Rb, H, g, 1e-6,
                          Y, H)
        assert np.array_equal(mixed.y.reshape(T, H), same.y), dt
        assert np.array_equal(mixed.residual.reshape(T, H).astype(np.float64),
                              lib_decode(same.residual, dt)), dt


# ---------------------------------------------------------------------------
# Pins on the 8-bit output (e4m3 / e5m2 codes with a per-tensor or per-row
# scale)
# ---------------------------------------------------------------------------

FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def lib_decode_fp8(codes, fmt: str) -> np.ndarray:
    """Decode 8-bit codes with torch's float8 types (not the oracle)."""
    import torch
    td = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8).copy())
    return c.view(td).to(torch.float64).numpy()


def _fp8_table(fmt):
    """Values and codes of the non-negative finite codes, ascending."""
    codes = np.arange(128, dtype=np.uint8)
    vals = lib_decode_fp8(codes, fmt)
    ok = np.isfinite(vals)
    return vals[ok], codes[ok]


def fp8_nearest(u, fmt: str) -> np.ndarray:
    """Brute force: the code of the finite value nearest to each u (exact
    rational distances, ties to the even code), so values beyond the largest
    finite value saturate to it; the sign bit is u's."""
    vals, codes = _fp8_table(fmt)
    u = np.asarray(u, np.float64)
    out = np.empty(u.size, np.uint8)
    for n, x in enumerate(u.ravel()):
        a = abs(float(x))
        k = int(np.searchsorted(vals, a))
        if k >= len(vals):
            c = codes[-1]
        elif vals[k] == a or k == 0:
            c = codes[k]
        else:
            fa = Fraction(a)
            dl, dh = fa - Fraction(vals[k - 1]), Fraction(vals[k]) - fa
            c = codes[k - 1] if dl < dh or (dl == dh and codes[k - 1] % 2 == 0) else codes[k]
        out[n] = c | (0x80 if np.signbit(x) else 0)
    return out.reshape(u.shape)


def pin_fp8_decode_all_codes(O):
    """Every code of both formats decodes as torch's float8 types decode it."""
    codes = np.arange(256, dtype=np.uint8)
    for fmt in ("e4m3", "e5m2"):
        a = O.decode_fp8(codes, fmt)
        b = lib_decode_fp8(codes, fmt)
        assert np.array_equal(np.isnan(a), np.isnan(b)), fmt
        ok = ~np.isnan(b)
        assert np.array_equal(a[ok], b[ok]), fmt


def _fp8_probe(fmt, rng):
    vals, _ = _fp8_table(fmt)
    mid = (vals[1:] + vals[:-1]) / 2  # exact in binary64
    top = FP8_MAX[fmt]
    step = vals[-1] - vals[-2]
    probe = [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), vals,
             np.exp2(rng.uniform(np.log2(vals[1]) - 2, np.log2(top) + 1, 3000)),
             np.array([0.0, vals[1] / 2, vals[1] / 4, top + step / 2, top + step,
                       top * 1.01, top * 4, 1e30])]
    p = np.concatenate(probe)
    return np.concatenate([p, -p])


def pin_fp8_round_nearest(O):
    """Rounding to 8 bits is nearest-even with saturation (brute force over the
    code table), and agrees with torch's float32 -> float8 cast inside the
    finite range."""
    import torch
    rng = np.random.default_rng(21)
    for fmt in ("e4m3", "e5m2"):
        p = _fp8_probe(fmt, rng)
        got = O.round_fp8(p, fmt)
        assert np.array_equal(got, fp8_nearest(p, fmt)), fmt
        td = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
        p32 = p[np.abs(p) <= FP8_MAX[fmt]].astype(np.float32)
        lib = torch.from_numpy(p32).to(td).view(torch.uint8).numpy()
        assert np.array_equal(O.round_fp8(p32.astype(np.float64), fmt), lib), fmt


def pin_fp8_tensor_scale_closed_form(O):
    """A constant row c with weights gamma_i and a per-tensor scale s:
    u_i = c / sqrt(c^2 + eps) * gamma_i / s (50-digit decimal), and each code
    is the nearest-even 8-bit value of u_i."""
    getcontext().prec = 50
    for dt in ("f32", "bf16", "f16"):
        for fmt, s in (("e4m3", 0.0078125), ("e4m3", 0.3), ("e5m2", 2.0 ** -10)):
            T, H, c, eps = 2, 64, 1.5, 1e-3
            x = bits_of(np.full((T, H), c), dt)
            gd = lib_decode(bits_of(np.linspace(-2.0, 2.0, H), dt), dt)
            g = bits_of(gd, dt)
            codes, _, u = O.rows_fp8(dt, fmt, T, H, 0, x.reshape(-1), H, T * H, None, H, g,
                                     eps, "tensor", s, want_u64=True)
            e32 = Decimal(float(np.float32(eps)))
            s32 = Decimal(float(np.float32(s)))
            k = Decimal(c) / (Decimal(c) * Decimal(c) + e32).sqrt()
            want = np.array([float(k * Decimal(gi) / s32) for gi in gd])
            for t in range(T):
                assert _rel(u[t], want) < 1e-14, (dt, fmt, s)
            assert np.array_equal(codes, fp8_nearest(u, fmt)), (dt, fmt, s)


def pin_fp8_row_scale(O):
    """Per-row scale: s_t = max_i |v_i| / maxf with v the normalised row of the
    16-bit-output path (whose pins fix it), u = v / s_t, codes nearest-even of
    u; the largest element becomes +-maxf; a row of zeros has s = 1 and zero
    codes; the residual is the one of the 16-bit-output path."""
    rng = np.random.default_rng(22)
    for dt in ("f32", "bf16", "f16"):
        for R in (0, 1, 3):
            T, H = 5, 77
            n = max(R, 1)
            parts = np.stack([_rand_bits(rng, (T, H), dt) for _ in range(n)])
            parts[:, 2] = bits_of(np.zeros((n, H)), dt)
            res = _rand_bits(rng, (T, H), dt)
            if R:
                res[2] = bits_of(np.zeros(H), dt)
            g = bits_of(rng.uniform(-1.5, 1.5, H), dt)
            if R == 0:
                ref = O.rms_norm(parts[0], g, 1e-5, dt, want_y64=True)
            elif R == 1:
                ref = O.fused_add_rms_norm(parts[0], res, g, 1e-5, dt, want_y64=True)
            else:
                ref = O.reduce_add_rms_norm(parts, res, g, 1e-5, dt, want_y64=True)
            for fmt in ("e4m3", "e5m2"):
                rb = res.reshape(-1).copy() if R else None
                codes, rs, u = O.rows_fp8(dt, fmt, T, H, R, parts.reshape(-1).copy(), H, T * H,
                                          rb, H, g, 1e-5, "row", want_u64=True)
                amax = np.max(np.abs(ref.y64), axis=1)
                s = np.where(amax > 0, amax / FP8_MAX[fmt], 1.0)
                assert np.array_equal(rs, s.astype(np.float32)), (dt, R, fmt)
                assert _rel(u, ref.y64 / s[:, None]) < 1e-15, (dt, R, fmt)
                assert np.array_equal(codes, fp8_nearest(u, fmt)), (dt, R, fmt)
                vals = lib_decode_fp8(codes, fmt)
                top = np.max(np.abs(vals), axis=1)
                assert np.array_equal(top[amax > 0], np.full((amax > 0).sum(), FP8_MAX[fmt]))
                assert rs[2] == 1.0 and np.all(vals[2] == 0), (dt, R, fmt)
                if R:
                    assert np.array_equal(rb.reshape(T, H), ref.residual), (dt, R, fmt)


def pin_fp8_strides(O):
    """Strided inputs and a code row stride larger than H: the dense result in
    the first H bytes of each row, the padding untouched."""
    rng = np.random.default_rng(23)
    for dt in ("bf16", "f32"):
        for R in (0, 1, 3):
            T, H, ldx, ldr, ldq = 4, 45, 51, 47, 64
            n = max(R, 1)
            parts = np.stack([_rand_bits(rng, (T, H), dt) for _ in range(n)])
            res = _rand_bits(rng, (T, H), dt)
            g = bits_of(rng.uniform(0.5, 1.5, H), dt)
            slice_ = T * ldx + 5
            X = np.concatenate([_strided(parts[r], ldx, dt, extra=5) for r in range(n)])
            Rs = _strided(res, ldr, dt) if R else None
            Rd = res.reshape(-1).copy() if R else None
            for mode in ("tensor", "row"):
                a = O.rows_fp8(dt, "e4m3", T, H, R, X, ldx, slice_, Rs, ldr, g, 1e-5, mode, 0.05,
                               ldq, fill=0x5A)
                b = O.rows_fp8(dt, "e4m3", T, H, R, parts.reshape(-1).copy(), H, T * H, Rd, H, g,
                               1e-5, mode, 0.05)
                assert np.array_equal(a[0][:, :H], b[0]), (dt, R, mode)
                assert np.all(a[0][:, H:] == 0x5A), (dt, R, mode)
                assert np.array_equal(a[1], b[1]), (dt, R, mode)
                if R:
                    assert np.array_equal(_rows(Rs, T, ldr, H), Rd.reshape(T, H)), (dt, R, mode)
                    pad = Rs.reshape(T, ldr)[:, H:]
                    assert np.array_equal(pad, np.full_like(pad, GARBAGE[dt])), (dt, R, mode)
                    # second call on updated residuals: restore for the next mode
                    Rs = _strided(res, ldr, dt)
                    Rd = res.reshape(-1).copy()


# ---------------------------------------------------------------------------
# Pins on the GEMM producer with the fused epilogue
# ---------------------------------------------------------------------------

def _gemm(O, dt, A, W, r, g, eps, lda=None, ldw=None, ldr=None, ldy=None, T=None, H=None,
          K=None):
    T = T or A.shape[0]
    H = H or W.shape[0]
    K = K or A.shape[-1]
    return O.gemm_add_rms_norm(dt, A.reshape(-1), W.reshape(-1), r, g, eps, T, H, K, lda, ldw,
                               ldr, ldy, want_p64=True)


def pin_gemm_product_library(O):
    """P and sum |A W| against numpy's binary64 matrix product of the
    library-decoded operands, with magnitudes spread over 2^+-20 so that the
    sums are not all exact."""
    rng = np.random.default_rng(31)
    for dt in ("bf16", "f16", "f32"):
        T, H, K = 5, 7, 300
        av = rng.standard_normal((T, K)) * np.exp2(rng.integers(-20, 21, (T, K)) * (dt != "f16"))
        wv = rng.standard_normal((H, K)) * 0.1
        A, W = bits_of(av, dt), bits_of(wv, dt)
        r = bits_of(rng.standard_normal((T, H)), dt).reshape(-1).copy()
        res = _gemm(O, dt, A, W, r, bits_of(np.ones(H), dt), 1e-6)
        ad, wd = lib_decode(A, dt), lib_decode(W, dt)
        P = ad @ wd.T
        S = np.abs(ad) @ np.abs(wd).T
        tol = 4 * K * 2.0 ** -53
        assert np.all(np.abs(res.p64 - P) <= tol * S), dt
        assert np.all(np.abs(res.abs64 - S) <= tol * S), dt


def pin_gemm_identity_is_fused(O):
    """W = I (H = K): P = A exactly, and the GEMM form equals the fused form
    with x = A bit for bit (y, residual; the fused form's binary32 sum of two
    storage values rounds like the exact sum)."""
    rng = np.random.default_rng(32)
    for dt in ("bf16", "f16", "f32"):
        T, H = 6, 96
        A = _rand_bits(rng, (T, H), dt)
        r = _rand_bits(rng, (T, H), dt)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        W = bits_of(np.eye(H), dt)
        got = _gemm(O, dt, A, W, r.reshape(-1).copy(), g, 1e-5)
        want = O.fused_add_rms_norm(A, r, g, 1e-5, dt)
        assert np.array_equal(got.y.reshape(T, H), want.y), dt
        assert np.array_equal(got.residual.reshape(T, H), want.residual), dt


def pin_gemm_one_rounding(O):
    """The residual is the exact P + r rounded once: with A = [1, 1],
    W = [1, 3 * 2^-10], r = 2^-8 (bf16), P + r = 1 + 7 * 2^-10 rounds to
    1 + 2^-7, whereas rounding P first (to 1) would give the tie 1 + 2^-8 and
    round it to 1."""
    A = bits_of(np.array([[1.0, 1.0]]), "bf16")
    W = bits_of(np.array([[1.0, 3 * 2.0 ** -10]]), "bf16")
    r = bits_of(np.array([2.0 ** -8]), "bf16").copy()
    got = _gemm(O, "bf16", A, W, r, bits_of(np.array([1.0]), "bf16"), 1e-6)
    assert lib_decode(got.residual, "bf16")[0] == 1 + 2.0 ** -7
    assert got.p64[0, 0] == 1 + 3 * 2.0 ** -10


def pin_gemm_brute_force_tiny(O):
    """Tiny problems from scratch: exact rational P and residual rounding,
    exact sum of squares, 50-digit root, exact rounding of y."""
    getcontext().prec = 50
    rng = np.random.default_rng(33)
    for dt in ("bf16", "f16", "f32"):
        T, H, K = 3, 9, 11
        A = _rand_bits(rng, (T, K), dt)
        W = _rand_bits(rng, (H, K), dt, scale=0.3)
        r = _rand_bits(rng, (T, H), dt)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        got = _gemm(O, dt, A, W, r.reshape(-1).copy(), g, 1e-2)
        ad, wd, rd, gd = (lib_decode(A, dt), lib_decode(W, dt), lib_decode(r, dt),
                          lib_decode(g, dt))
        e32 = Fraction(float(np.float32(1e-2)))
        for t in range(T):
            P = [sum(Fraction(ad[t, k]) * Fraction(wd[i, k]) for k in range(K)) for i in range(H)]
            h = [Fraction(rn_exact(P[i] + Fraction(rd[t, i]), dt)) for i in range(H)]
            got_h = lib_decode(got.residual.reshape(T, H)[t], dt)
            assert np.array_equal(got_h, np.array([float(v) for v in h])), (dt, t)
            m = sum(v * v for v in h) / H + e32
            inv = 1 / (Decimal(m.numerator) / Decimal(m.denominator)).sqrt()
            assert abs(got.inv[t] - float(inv)) <= 1e-15 * float(inv), (dt, t)
            want = [rn_exact(Fraction(Decimal(v.numerator) / Decimal(v.denominator) * inv *
                                      Decimal(gd[i])), dt) for i, v in enumerate(h)]
            assert np.array_equal(lib_decode(got.y.reshape(T, H)[t], dt), np.array(want)), (dt, t)


def pin_gemm_strides(O):
    """Row strides for A, W, the residual and y (padding holding garbage):
    the dense results, the padding of the residual untouched."""
    rng = np.random.default_rng(34)
    for dt in ("bf16", "f32"):
        T, H, K = 4, 10, 24
        lda, ldw, ldr, ldy = 30, 27, 13, 16
        A = _rand_bits(rng, (T, K), dt)
        W = _rand_bits(rng, (H, K), dt, scale=0.2)
        r = _rand_bits(rng, (T, H), dt)
        g = bits_of(rng.uniform(0.5, 1.5, H), dt)
        dense = _gemm(O, dt, A, W, r.reshape(-1).copy(), g, 1e-5)
        Rs = _strided(r, ldr, dt)
        got = O.gemm_add_rms_norm(dt, _strided(A, lda, dt), _strided(W, ldw, dt), Rs, g, 1e-5,
                                  T, H, K, lda, ldw, ldr, ldy)
        assert np.array_equal(got.y.reshape(T, ldy)[:, :H], dense.y.reshape(T, H)), dt
        assert np.array_equal(_rows(Rs, T, ldr, H), dense.residual.reshape(T, H)), dt
        pad = Rs.reshape(T, ldr)[:, H:]
        assert np.array_equal(pad, np.full_like(pad, GARBAGE[dt])), dt


# ---------------------------------------------------------------------------
# Pins on the 8-bit partials (reduce over e4m3 / e5m2 codes with a scale each)
# ---------------------------------------------------------------------------

def _finite_codes(rng, fmt, shape, top=None):
    """Random codes of finite values (optionally |value| <= top), both signs."""
    vals, codes = _fp8_table(fmt)
    pick = codes if top is None else codes[vals <= top]
    c = rng.choice(pick, size=shape).astype(np.uint8)
    return c | (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7)


def pin_fp8in_power_of_two_scales_are_reduce(O):
    """With power-of-two scales every dequantised partial code * 2^k is exact,
    so the 8-bit form must equal the (pinned) 16-bit / binary32 reduce over
    partials holding those values, bit for bit, residual and y; the values
    come from torch's float8 decoders, not the oracle's."""
    rng = np.random.default_rng(21)
    for dt in ("bf16", "f16", "f32"):
        for fmt in ("e4m3", "e5m2"):
            R, T, H = 5, 3, 70
            top = 448.0 if fmt == "e4m3" else (4096.0 if dt == "f16" else None)
            codes = _finite_codes(rng, fmt, (R, T, H), top)
            ks = rng.integers(-3, 4, size=R) if dt != "f16" else rng.integers(-3, 1, size=R)
            scales = np.exp2(ks).astype(np.float32)
            r = _rand_bits(rng, (T, H), dt)
            g = bits_of(rng.uniform(0.5, 1.5, H), dt)
            vals = lib_decode_fp8(codes, fmt) * scales[:, None, None].astype(np.float64)
            p16 = bits_of(vals, dt).reshape(R, T, H)
            assert np.array_equal(lib_decode(p16, dt), vals), (dt, fmt)  # exact in dt
            got = O.reduce_fp8in(codes, scales, r, g, 1e-6, dt, fmt)
            want = O.reduce_add_rms_norm(p16, r, g, 1e-6, dt)
            assert np.array_equal(got.residual, want.residual), (dt, fmt)
            assert np.array_equal(got.y, want.y), (dt, fmt)


def pin_fp8in_brute_force(O):
    """Arbitrary scales: each partial enters as code * scale rounded once to
    binary32, summed in order p0 .. p{R-1}, then the residual, each add in
    binary32, one rounding to the storage type -- in exact rationals."""
    rng = np.random.default_rng(22)
    for dt in ("bf16", "f16", "f32"):
        for fmt in ("e4m3", "e5m2"):
            R, T, H = 4, 2, 11
            codes = _finite_codes(rng, fmt, (R, T, H), 448.0)
            scales = rng.uniform(1e-3, 3.0, size=R).astype(np.float32)
            r = _rand_bits(rng, (T, H), dt)
            res = O.reduce_fp8in(codes, scales, r, bits_of(np.ones(H), dt), 1e-6, dt, fmt)
            dec = lib_decode_fp8(codes, fmt)
            rv = lib_decode(r, dt)
            want = np.empty((T, H))
            for t in range(T):
                for i in range(H):
                    v = [Fraction(rn_exact(Fraction(dec[k, t, i]) * Fraction(float(scales[k])),
                                           "f32")) for k in range(R)]
                    acc = v[0]
                    for k in range(1, R):
                        acc = Fraction(rn_exact(acc + v[k], "f32"))
                    acc = Fraction(rn_exact(acc + Fraction(rv[t, i]), "f32"))
                    want[t, i] = rn_exact(acc, dt)
            assert np.array_equal(lib_decode(res.residual, dt), want), (dt, fmt)


# ---------------------------------------------------------------------------
# Tensor-parallel form (reduce-scatter, residual + norm, all-gather)
# ---------------------------------------------------------------------------

def pin_tp_partition(O):
    """Rank r's rows: contiguous blocks in rank order that cover 0 .. T-1
    exactly once, sizes differing by at most one (T = qN + m: m blocks of
    q + 1 rows, N - m of q), for every N up to 9 and T up to 40."""
    for N in range(1, 10):
        for T in range(0, 41):
            blocks = [O.tp_rows(T, N, r) for r in range(N)]
            assert blocks[0][0] == 0 and blocks[-1][1] == T, (T, N, blocks)
            for (a0, a1), (b0, b1) in zip(blocks, blocks[1:]):
                assert a1 == b0, (T, N, blocks)
            sizes = sorted(b - a for a, b in blocks)
            q, m = divmod(T, N)
            assert sizes == [q] * (N - m) + [q + 1] * m, (T, N, blocks)


def pin_tp_is_reduce_over_ranks(O):
    """The N ranks' partials give, in every rank's buffer, the y of the
    (pinned) reduce over those partials stacked in rank order, and the same
    updated residual: the reduce-scatter, norm and all-gather compute the
    reduce form with R = N, row by row whoever owns the row."""
    rng = np.random.default_rng(31)
    for dt in ("bf16", "f16", "f32"):
        for N, T, H in ((1, 5, 24), (2, 7, 40), (3, 10, 33), (5, 4, 16), (8, 19, 64)):
            bufs = [_rand_bits(rng, (T, H), dt, 1.0 / math.sqrt(N)) for _ in range(N)]
            r = _rand_bits(rng, (T, H), dt)
            g = bits_of(rng.uniform(0.5, 1.5, H), dt)
            got = O.tp_reduce_add_rms_norm(bufs, r, g, 1e-6, dt)
            want = O.reduce_add_rms_norm(np.stack(bufs), r, g, 1e-6, dt)
            assert np.array_equal(got.residual, want.residual), (dt, N)
            assert len(got.ys) == N
            for q, y in enumerate(got.ys):
                assert np.array_equal(y, want.y), (dt, N, q)


def pin_tp_rank_order_worked_example(O):
    """Three ranks hold 2^24, 1 and -2^24 (binary32): in rank order
    fl32(fl32(2^24 + 1) - 2^24) = 0, while the exact sum, and the reverse
    order, give 1.  With a zero residual the stored residual is 0 and y is 0
    in every rank's buffer."""
    T, H = 4, 8
    vals = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    bufs = [np.full((T, H), v, np.float32) for v in vals]
    r = np.zeros((T, H), np.float32)
    g = np.ones(H, np.float32)
    got = O.tp_reduce_add_rms_norm(bufs, r, g, 1e-6, "f32")
    assert np.array_equal(got.residual, np.zeros((T, H), np.float32)), got.residual
    for y in got.ys:
        assert np.array_equal(y, np.zeros((T, H), np.float32))
    # the residual joins after the last rank: (2^24 + 1) + 1 = 2^24 + 2 in one
    # rounding would give 2^24 + 2; in order it is fl32(2^24 + 1) + 1 = 2^24
    bufs = [np.full((T, H), 2.0 ** 24, np.float32), np.ones((T, H), np.float32)]
    got = O.tp_reduce_add_rms_norm(bufs, np.ones((T, H), np.float32), g, 1e-6, "f32")
    assert np.all(got.residual == np.float32(2.0 ** 24)), got.residual


ALL_PINS = [
    pin_decode_all_patterns,
    pin_round_matches_library,
    pin_round_bf16_nearest,
    pin_round_exact_rationals,
    pin_fused_residual_is_exact_rounded_sum,
    pin_reduce_order_worked_example,
    pin_reduce_integer_sums,
    pin_reduce_brute_force_binary32,
    pin_reduce_special_cases,
    pin_constant_row,
    pin_unit_gamma_rms,
    pin_scale_invariance,
    pin_single_element_rows,
    pin_brute_force_tiny,
    pin_strided_equals_dense,
    pin_fp32_residual_sum,
    pin_fp32_residual_matches_16bit_when_exact,
    pin_fp8_decode_all_codes,
    pin_fp8_round_nearest,
    pin_fp8_tensor_scale_closed_form,
    pin_fp8_row_scale,
    pin_fp8_strides,
    pin_gemm_product_library,
    pin_gemm_identity_is_fused,
    pin_gemm_one_rounding,
    pin_gemm_brute_force_tiny,
    pin_gemm_strides,
    pin_fp8in_power_of_two_scales_are_reduce,
    pin_fp8in_brute_force,
    pin_tp_partition,
    pin_tp_is_reduce_over_ranks,
    pin_tp_rank_order_worked_example,
]
