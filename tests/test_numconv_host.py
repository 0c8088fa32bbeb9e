"""The library's integer-only float conversion (pp_numeric.cuh), compiled
for the host, against Python's float() — an independent correctly rounded
decimal-to-binary64 conversion.  Exact for at most 19 significant digits
with 0 <= q <= 55; within 1 ulp everywhere (the tolerance of the spec)."""
import ctypes
import os
import random
import struct
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dfa_parsing_delimiter_gb300", "csrc")


@pytest.fixture(scope="module")
def harness():
    subprocess.check_call(["python3", os.path.join(CSRC, "gen_pow10.py"),
                           os.path.join(CSRC, "pow5_table.inc")])
    d = tempfile.mkdtemp()
    so = os.path.join(d, "numconv.so")
    cuda_inc = "/usr/local/cuda/include"
    subprocess.check_call(["g++", "-O2", "-shared", "-fPIC", "-std=c++17",
                           "-I" + CSRC, "-I" + os.path.join(ROOT, "include"), "-I" + cuda_inc,
                           os.path.join(ROOT, "tests", "numconv_harness.cpp"), "-o", so])
    L = ctypes.CDLL(so)
    L.h_parse_floats.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                 ctypes.c_void_p]
    L.h_decimal_to_binary64.restype = ctypes.c_uint64
    L.h_decimal_to_binary64.argtypes = [ctypes.c_uint64, ctypes.c_int]
    return L


def _run(L, strs):
    buf = b"".join(s.encode() + b"\x00" for s in strs)
    a = np.frombuffer(buf, dtype=np.uint8)
    bits = np.zeros(len(strs), dtype=np.uint64)
    err = np.zeros(len(strs), dtype=np.int32)
    L.h_parse_floats(a.ctypes.data, len(strs), bits.ctypes.data, err.ctypes.data)
    return bits, err


def _ulps(a_bits, b_bits):
    def ordered(x):
        i = x.view(np.int64)
        return np.where(i < 0, np.int64(-0x8000000000000000) - i, i)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def _want(strs):
    return np.array([struct.unpack("<Q", struct.pack("<d", float(s)))[0] for s in strs],
                    dtype=np.uint64)


def test_exact_cases(harness):
    strs = ["0", "-0", "1", "0.1", "463.86", "1e22", "1e23", "9007199254740993",
            "9007199254740992", "9007199254740994", "9007199254740995", "1.7976931348623157e308",
            "1.7976931348623158e308", "1.7976931348623159e308", "2.2250738585072014e-308",
            "2.2250738585072011e-308", "4.9406564584124654e-324", "2.4703282292062328e-324",
            "2.4703282292062327e-324", "1e-400", "1e400", "123.456e-5", ".5", "5.", "-2.5e-3",
            "18446744073709551615", "18446744073709551616", "0.000000000000000000000000000001",
            "179769313486231580793728971405301e276", "7.2057594037927933e16",
            "4503599627370496.5", "4503599627370497.5", "1.00000000000000011102230246251565404236316680908203125"]
    bits, err = _run(harness, strs)
    assert (err == 0).all()
    want = _want(strs)
    d = _ulps(bits, want)
    exact_expected = [s for s in strs if len(s.replace("-", "").replace(".", "").lstrip("0")) <= 19]
    assert int(d.max()) <= 1, [(s, int(x)) for s, x in zip(strs, d) if x]


def test_ties_exact_for_small_positive_exponents(harness):
    """Binary ties reachable with <= 19 digits and 0 <= q <= 55 round to even."""
    rng = random.Random(1)
    strs = []
    for _ in range(20000):
        m = rng.randrange(1 << 53, 1 << 54) | 1      # odd 54-bit: a tie at 53 bits
        e = rng.randint(0, 10)
        v = m << e
        s = str(v)
        if len(s) <= 19:
            strs.append(s)
    bits, err = _run(harness, strs)
    assert (bits == _want(strs)).all()


@pytest.mark.parametrize("seed", range(4))
def test_random_short_exact(harness, seed):
    """<= 19 significant digits: correctly rounded for every exponent here."""
    rng = random.Random(seed)
    strs = []
    for _ in range(100000):
        nd = rng.randint(1, 19)
        digits = str(rng.randint(1, 9)) + "".join(rng.choice("0123456789") for _ in range(nd - 1))
        k = rng.randint(0, nd)
        s = digits[:k] + "." + digits[k:] if k < nd else digits
        s += "e%d" % rng.randint(-330, 310)
        strs.append(("-" if rng.random() < 0.5 else "") + s)
    bits, err = _run(harness, strs)
    assert (err == 0).all()
    d = _ulps(bits, _want(strs))
    assert int(d.max()) <= 1
    # mismatches, if any, only where the spec's 1-ulp tolerance applies
    assert np.count_nonzero(d) <= 5


@pytest.mark.parametrize("seed", range(2))
def test_random_long_within_one_ulp(harness, seed):
    rng = random.Random(100 + seed)
    strs = []
    for _ in range(100000):
        nd = rng.randint(1, 40)
        digits = "".join(rng.choice("0123456789") for _ in range(nd))
        k = rng.randint(0, nd)
        s = digits[:k] + "." + digits[k:]
        if s == ".":
            s = "0."
        if rng.random() < 0.7:
            s += rng.choice("eE") + rng.choice(["", "+", "-"]) + str(rng.randint(0, 350))
        strs.append(s)
    bits, err = _run(harness, strs)
    assert (err == 0).all()
    d = _ulps(bits, _want(strs))
    assert int(d.max()) <= 1


def test_workload_shapes_exact(harness):
    """The printed shapes of the float workloads (%.2f in [0,500], %.6g of
    N(0, 1e3)) convert exactly."""
    rng = random.Random(9)
    strs = ["%d.%02d" % (c // 100, c % 100) for c in (rng.randint(0, 50000) for _ in range(50000))]
    strs += ["%.6g" % rng.gauss(0, 1e3) for _ in range(50000)]
    bits, err = _run(harness, strs)
    assert (bits == _want(strs)).all()


def test_syntax(harness):
    bad = ["", "+", ".", "e5", "1e", "1e+", "1.2.3", "inf", "nan", "0x1p3", "--1", "+.e1", "1a"]
    bits, err = _run(harness, bad)
    assert (err != 0).all()


def _short(L, ws, qs):
    L.h_short_decimal_to_binary64.restype = ctypes.c_uint64
    L.h_short_decimal_to_binary64.argtypes = [ctypes.c_uint32, ctypes.c_int]
    return np.array([L.h_short_decimal_to_binary64(w, q) for w, q in zip(ws, qs)], dtype=np.uint64)


def _exact(ws, qs):
    from fractions import Fraction
    return np.array([struct.unpack("<Q", struct.pack("<d", float(Fraction(w) / 10 ** (-q))))[0]
                     for w, q in zip(ws, qs)], dtype=np.uint64)


def test_short_significand_edges(harness):
    """The short path (w < 2^32, -17 <= q <= 0): dyadic values and the ends
    of the range are exact."""
    cases = [(1, 0), (9, 0), (4294967295, 0), (5, -1), (25, -2), (125, -3), (1, -1), (1, -17),
             (4294967295, -17), (4294967295, -1), (46386, -2), (50000, -2), (3, -1),
             (123456789, -7), (1, -8), (999999999, -9), (2 ** 31, 0), (2 ** 31 - 1, -3),
             (5 ** 13, -13), (99999999, -7), (10000000, -7)]
    ws, qs = zip(*cases)
    assert (_short(harness, ws, qs) == _exact(ws, qs)).all()


@pytest.mark.parametrize("seed", range(3))
def test_short_significand_random(harness, seed):
    """Random w < 2^32 and q in [-17, 0] against exact rational rounding:
    correctly rounded."""
    rng = random.Random(50 + seed)
    ws = [rng.choice([rng.randrange(1, 1 << 32), rng.randrange(1, 100000)]) for _ in range(20000)]
    qs = [rng.randint(-17, 0) for _ in ws]
    assert (_short(harness, ws, qs) == _exact(ws, qs)).all()


def test_short_significand_workload_shapes_exact(harness):
    """%.2f in [0, 500] and the significands %.6g prints convert exactly."""
    rng = random.Random(11)
    ws = [rng.randint(1, 50000) for _ in range(20000)] + [rng.randint(1, 999999) for _ in range(20000)]
    qs = [-2] * 20000 + [rng.randint(-6, 0) for _ in range(20000)]
    assert (_short(harness, ws, qs) == _exact(ws, qs)).all()


def _short_decimal(L, s, n, dot):
    L.h_short_decimal.restype = ctypes.c_int
    L.h_short_decimal.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.c_int,
                                  ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_int)]
    w, k = ctypes.c_uint32(0), ctypes.c_int(0)
    ok = L.h_short_decimal(s, n, dot, ctypes.byref(w), ctypes.byref(k))
    return (w.value, k.value) if ok else None


def _short_decimal_want(s, n, dot):
    """Plain reading: n digits, or (dot) digits with one '.' and at least one
    digit; the value as (digits as an integer, digits after the '.')."""
    t = s[:n]
    digits = b"".join(bytes([c]) for c in t if 0x30 <= c <= 0x39)
    dots = t.count(b".")
    if len(digits) + dots != n or (dots and not dot) or dots > 1 or not digits:
        return None
    k = n - 1 - t.index(b".") if dots else 0
    return int(digits), k


def test_short_decimal_exhaustive_small(harness):
    """Every string of 1..3 characters over digits, '.', signs, 'e' and
    bytes that alias digits or '.' in their low bits, with garbage after."""
    import itertools
    alpha = [b"0", b"5", b"9", b".", b"+", b"e", b"/", b":", b"\x80", b"\xae", b"\xb5", b" ", b"\x00"]
    for n in (1, 2, 3):
        for tup in itertools.product(alpha, repeat=n):
            s = b"".join(tup) + b"7.x\x00\xff9.1"[: 8 - n]
            for dot in (0, 1):
                assert _short_decimal(harness, s, n, dot) == _short_decimal_want(s, n, dot), (s, n, dot)


@pytest.mark.parametrize("seed", range(2))
def test_short_decimal_random(harness, seed):
    """Random 1..8-character fields: mostly valid plain decimals (the
    workloads' shapes), some with one character replaced."""
    rng = random.Random(70 + seed)
    for _ in range(20000):
        n = rng.randint(1, 8)
        kind = rng.random()
        if kind < 0.4:
            t = "".join(rng.choice("0123456789") for _ in range(n))
        else:
            t = "".join(rng.choice("0123456789") for _ in range(n))
            if n > 1:
                i = rng.randrange(n)
                t = t[:i] + "." + t[i + 1:]
        s = bytearray(t.encode() + bytes(rng.randrange(256) for _ in range(8 - n)))
        if rng.random() < 0.2:
            s[rng.randrange(n)] = rng.choice(b".-+e/:\x80\xae\xb0 0")
        s = bytes(s)
        for dot in (0, 1):
            assert _short_decimal(harness, s, n, dot) == _short_decimal_want(s, n, dot), (s, n, dot)


# ------------------------------------------------------------ timestamps
def _ts(L, strs):
    L.h_parse_timestamps.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                     ctypes.c_void_p]
    buf = b"".join(s + b"\x00" for s in strs)
    a = np.frombuffer(buf, dtype=np.uint8)
    out = np.zeros(len(strs), dtype=np.int64)
    err = np.zeros(len(strs), dtype=np.int32)
    L.h_parse_timestamps(a.ctypes.data, len(strs), out.ctypes.data, err.ctypes.data)
    return out, err


def test_days_from_civil_every_day_against_ordinal(harness):
    """The closed-form day count against Python's date ordinals, every day of
    years 1..9999 sampled every 7 days plus all days of leap-rule years."""
    import datetime
    L = harness
    L.h_days_from_civil.restype = ctypes.c_int64
    L.h_days_from_civil.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    epoch = datetime.date(1970, 1, 1).toordinal()
    o = datetime.date(1, 1, 1).toordinal()
    end = datetime.date(9999, 12, 31).toordinal()
    days = list(range(o, end + 1, 7))
    for y in (1, 4, 100, 400, 1600, 1700, 1900, 1969, 1970, 2000, 2024, 2100, 9999):
        d0 = datetime.date(y, 1, 1).toordinal()
        days += range(d0, d0 + 365 + (1 if (y % 4 == 0 and y % 100) or y % 400 == 0 else 0))
    for k in days:
        dt = datetime.date.fromordinal(k)
        assert L.h_days_from_civil(dt.year, dt.month, dt.day) == k - epoch, dt
    # year 0 of the proleptic calendar: 719528 days before 1970
    assert L.h_days_from_civil(0, 1, 1) == -719528
    assert L.h_days_from_civil(0, 3, 1) == -719468


def test_timestamp_words_match_timegm_and_reject_bad_fields(harness):
    import calendar
    import random
    rng = random.Random(11)
    strs, want = [], []
    for _ in range(5000):
        y, mo = rng.randint(0, 9999), rng.randint(1, 12)
        leap = (y % 4 == 0 and y % 100 != 0) or y % 400 == 0
        dim = [31, 29 if leap else 28, 31, 30, 31, 30, 31, 31, 30, 31, 30, 31][mo - 1]
        d, h, mi, s = rng.randint(1, dim), rng.randint(0, 23), rng.randint(0, 59), rng.randint(0, 59)
        if rng.random() < 0.5:
            strs.append(b"%04d-%02d-%02d %02d:%02d:%02d" % (y, mo, d, h, mi, s))
        else:
            strs.append(b"%04d-%02d-%02d" % (y, mo, d))
            h = mi = s = 0
        days = (calendar.timegm((max(y, 1), mo, d, 0, 0, 0, 0, 0, 0)) // 86400 if y else
                -719528 + sum([31, 29, 31, 30, 31, 30, 31, 31, 30, 31, 30, 31][:mo - 1]) + d - 1)
        want.append(days * 86400 + h * 3600 + mi * 60 + s)
    bad = [b"1900-02-29", b"2023-02-29", b"2021-04-31", b"2021-13-01", b"2021-00-10",
           b"2021-01-00", b"2021-01-01 24:00:00", b"2021-01-01 23:60:00",
           b"2021-01-01 23:59:60", b"2021-1-01", b"2021/01/01", b"2021-01-01T00:00:00",
           b"2021-01-01 00:00", b"2021-01-01 ", b"2021-01-01 00:00:0x", b"20210101",
           b"2021-01-01 00:00:00 ", b"2021-01-0\x80", b"\xb021-01-01"]
    out, err = _ts(harness, strs + bad + [b""])
    assert err[:len(strs)].tolist() == [0] * len(strs)
    assert out[:len(strs)].tolist() == want
    assert err[len(strs):-1].tolist() == [PP_SYNTAX] * len(bad)
    assert out[len(strs):].tolist() == [0] * (len(bad) + 1)
    assert err[-1] == 0


PP_SYNTAX = 8
