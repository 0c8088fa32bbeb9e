"""Pins for the oracle on long numeric fields (hundreds to tens of
thousands of bytes), the inputs that the library converts with a whole warp
(ParPaRaw Section 3.3, collaboration on long fields).  Expected values come
from Python's float() and int() on the same text, not from the oracle."""
import random
import struct

import pytest

import oracle as O


def _bits(x):
    return struct.unpack("<Q", struct.pack("<d", x))[0]


def long_numbers(rng):
    z = "0" * rng.randint(300, 3000)
    d = "".join(rng.choice("0123456789") for _ in range(rng.randint(300, 2000)))
    return [
        z + "1.5",
        "-" + z + "." + z + "25e-3",
        "1" + d + "e-" + "0" * 400 + str(len(d)),
        "." + z + "7",
        d + "." + d,
        "+" + d[:25] + "e" + "0" * 500 + "5",
        "1e" + "9" * 400,          # overflows to inf
        "1e-" + "9" * 400,         # underflows to 0
        "-0." + z,
        z,
    ]


@pytest.mark.parametrize("seed", range(3))
def test_long_floats_match_python(seed):
    rng = random.Random(seed)
    vals = long_numbers(rng)
    data = "".join(v + "\n" for v in vals).encode()
    cols, st = O.csv_parse(data, ["f64"])
    assert st["error"] == 0 and st["n_records"] == len(vals)
    for got, v in zip(cols[0].tolist(), vals):
        assert _bits(got) == _bits(float(v)), v[:40]


def test_long_integers_match_python():
    z = "0" * 3000
    vals = [(z + "127", "i8"), ("-" + z + "128", "i8"), (z + "128", "i8"),
            (z + "9223372036854775807", "i64"), ("-" + z + "9223372036854775808", "i64"),
            (z + "9223372036854775808", "i64"), ("1" + "0" * 19, "i64"),
            (z + "2147483647", "i32"), ("-" + z + "2147483649", "i32")]
    lim = {"i8": 7, "i32": 31, "i64": 63}
    for text, ty in vals:
        cols, st = O.csv_parse((text + "\n").encode(), [ty])
        x = int(text)
        if -(1 << lim[ty]) <= x < (1 << lim[ty]):
            assert st["error"] == 0 and cols[0].tolist() == [x], text[-30:]
        else:
            assert st["error"] == O.E_NUM_OVERFLOW and cols[0].tolist() == [0], text[-30:]


@pytest.mark.parametrize("text", ["1" * 500 + "..5", "-" * 2 + "1" * 500, "1" * 500 + "e",
                                  "1" * 500 + "e+", "1" * 500 + "x", "." * 300,
                                  "1" * 400 + "e5.5", "1" * 300 + "e-" + "2" * 300 + "-"])
def test_long_syntax_errors(text):
    cols, st = O.csv_parse(("7\n" + text + "\n").encode(), ["f64"])
    assert st["error"] == O.E_NUM_SYNTAX and st["first_error_offset"] == 2
    assert cols[0].tolist() == [7.0, 0.0]


def test_long_integer_rejects_float_syntax():
    cols, st = O.csv_parse(("1" * 400 + ".0\n").encode(), ["i64"])
    assert st["error"] == O.E_NUM_SYNTAX and cols[0].tolist() == [0]
