"""Long numeric fields (ParPaRaw Section 3.3, collaboration on long fields):
fields longer than the per-lane limit (256 bytes) are queued by the tile pass
and converted by a warp each.  Every case is compared with the oracle
element by element (floats within 1 ulp, integers, error bits and the first
error offset exact): multi-KB fields mixed with short ones, fields spanning
several tiles or starting at a tile boundary, quoted fields, CRLF inputs with
carriage returns inside numbers, syntax and overflow errors at any depth,
more long fields than the queue holds, and the options that drop records."""
import random

import numpy as np
import pytest
import torch

import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import compare_csv, to_dev
from test_gpu_options import compare_ex

pytestmark = pytest.mark.gpu
TILE = 16384


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _digits(rng, n, lead_zero=False):
    s = "".join(rng.choice("0123456789") for _ in range(n))
    return ("0" * rng.randint(0, n) + s) if lead_zero else s


def long_float(rng):
    k = rng.randint(0, 7)
    n = rng.randint(260, 3000)
    if k == 0:
        return "0" * n + "1.5"
    if k == 1:
        return "-" + "0" * n + "." + "0" * rng.randint(0, 300) + _digits(rng, 30) + "e-" + "0" * 50 + "7"
    if k == 2:
        return _digits(rng, n) + "." + _digits(rng, rng.randint(0, 400))
    if k == 3:
        return "." + "0" * n + "123456789012345678901234567"
    if k == 4:
        return "+" + _digits(rng, 30) + "e" + "0" * n + str(rng.randint(0, 300))
    if k == 5:
        return '"' + _digits(rng, n, True) + "." + _digits(rng, 40) + '"'
    if k == 6:
        return "1e" + "9" * n if rng.random() < 0.5 else "1e-" + "9" * n
    return "-0." + "0" * n


def long_int(rng, bits):
    n = rng.randint(260, 3000)
    v = rng.randint(-(1 << (bits - 1)), (1 << (bits - 1)) - 1)
    if rng.random() < 0.2:
        v = (1 << (bits - 1)) if rng.random() < 0.5 else -(1 << (bits - 1)) - 1  # out of range
    s = ("-" if v < 0 else rng.choice(["", "+"])) + "0" * n + str(abs(v))
    return '"' + s + '"' if rng.random() < 0.2 else s


def short_value(rng, ty):
    if ty == "f64":
        return f"{rng.uniform(-1e3, 1e3):.6g}"
    if ty == "str":
        return "".join(rng.choice("abc") for _ in range(rng.randint(0, 8)))
    return str(rng.randint(-100, 100))


def table(rng, n_rows, types, p_long):
    bits = {"i8": 8, "i32": 32, "i64": 64}
    rows = []
    for _ in range(n_rows):
        f = []
        for ty in types:
            if ty != "str" and rng.random() < p_long:
                f.append(long_float(rng) if ty == "f64" else long_int(rng, bits[ty]))
            else:
                f.append(short_value(rng, ty))
        rows.append(",".join(f))
    return ("\n".join(rows) + "\n").encode()


@pytest.mark.parametrize("seed", range(4))
def test_long_fields_mixed(seed):
    rng = random.Random(700 + seed)
    types = ["f64", "i64", "str", "i32", "f64", "i8"]
    data = table(rng, 300, types, 0.25)
    assert len(data) > 8 * TILE
    pp.debug_long_fields(reset=True)
    compare_csv(data, types)
    # the long fields went through the warp pass (the oracle counts them)
    n_long = sum(1 for row in data.split(b"\n") for f, t in zip(row.split(b","), types)
                 if t != "str" and len(f) > 256)
    assert pp.debug_long_fields() == n_long > 0


def test_long_fields_spanning_tiles():
    """Fields of 20-60 KB: each spans several tiles; one starts exactly at a
    tile boundary, one ends exactly at one."""
    pre = "1,2\n"
    a = "0" * 50000 + "12345.678e-2"
    b = "0" * 40000 + "9223372036854775807"
    data = (pre + a + "," + b + "\n").encode()
    compare_csv(data, ["f64", "i64"])
    # a field starting at a tile boundary
    head = "x" * (TILE - 3) + ",1\n"
    assert len(head) == TILE
    data = (head + "0" * 30000 + "7.25,-" + "0" * 20000 + "5\n").encode()
    compare_csv(data, ["f64", "i64"])
    # a field ending at a tile boundary
    body = "0" * (2 * TILE - 6) + "1.5"
    data = ("3," + body + "\n").encode()
    assert data.index(b"\n") in (2 * TILE - 1, 2 * TILE, 2 * TILE + 1)
    compare_csv(data, ["i32", "f64"])


@pytest.mark.parametrize("where", [0, 100, 1000, 5000])
def test_long_field_errors(where):
    """A bad byte at several depths of a 6 KB field: a syntax error at the
    field's first byte; integers of 20 significant digits overflow."""
    rng = random.Random(where)
    good = _digits(rng, 6000)
    for bad in ("x", ".", "e", "-", '"'):
        s = good[:where] + bad + good[where:]
        text = "1.5," + ('"' + s + '"' if bad == '"' else s) + "\n7,8\n"
        compare_csv(text.encode(), ["f64", "f64"])
    compare_csv(("1," + "0" * 3000 + "1" + "0" * 19 + "\n").encode(), ["i64", "i64"])
    compare_csv(("1," + "1" * 3000 + "e" + "\n").encode(), ["i64", "f64"])
    compare_csv(("1," + "1" * 3000 + ".5" + "\n").encode(), ["i64", "i32"])


def test_more_long_fields_than_the_queue():
    """Over 4096 long fields in one call: those beyond the queue are
    converted by their lanes, with the same values."""
    rng = random.Random(5)
    rows = []
    for i in range(4400):
        r = rng.randint(-50, 50)
        rows.append("0" * 300 + str(rng.randint(0, 10 ** 6)) + "." + str(i) + "," +
                    ("-" if r < 0 else "") + "0" * 280 + str(abs(r)))
    data = ("\n".join(rows) + "\n").encode()
    pp.debug_long_fields(reset=True)
    compare_csv(data, ["f64", "i8"])
    assert pp.debug_long_fields() == 4096


def test_long_fields_crlf():
    """With CRLF line ends a carriage return outside quotes is a control
    symbol: inside a long unquoted number it is dropped."""
    rng = random.Random(9)
    rows = []
    for _ in range(40):
        d = list(_digits(rng, rng.randint(300, 900)))
        for _ in range(5):
            d.insert(rng.randint(0, len(d)), "\r")
        rows.append("".join(d) + "," + "".join(d[:50]).replace("\r", "") + ".5")
    data = ("\r\n".join(rows) + "\r\n").encode()
    compare_csv(data, ["f64", "f64"], crlf=True)


def test_long_fields_with_dropped_records():
    """Skipped and rejected records shift the output rows of the long
    fields queued after them."""
    rng = random.Random(21)
    rows = []
    for i in range(200):
        nf = 2 if rng.random() < 0.8 else 3
        rows.append(",".join("0" * rng.randint(250, 700) + str(i * 7 + k) for k in range(nf)))
    data = ("\n".join(rows) + "\n").encode()
    compare_ex(data, ["i64", "f64"], skip_records=sorted(rng.sample(range(200), 30)))
    compare_ex(data, ["i64", "f64"], reject=True)


def test_long_field_last_record_without_newline():
    """The input ends inside a long field of a record with no record
    delimiter: the field still closes (the virtual delimiter at the end),
    also when it spans tiles."""
    for n in (300, 3 * TILE):
        compare_csv(("1,2\n3," + "0" * n + "4.5").encode(), ["i32", "f64"])
        compare_csv(("1,2\n3," + "0" * n + "-77").encode(), ["i32", "i64"])


def test_long_fields_fixed_scratch():
    """pp_parse_noalloc queues long fields in its fixed buffer too."""
    rng = random.Random(31)
    rows = ["0" * rng.randint(300, 2000) + str(i) + ".25," + str(i) for i in range(300)]
    data = ("\n".join(rows) + "\n").encode()
    n = len(data)
    out = pp.CsvOutputs(["f64", "i32"], n + 1, [0, 0])
    pp.debug_long_fields(reset=True)
    out.run_noalloc(to_dev(data), n, pp.desc_csv())
    st = pp.read_status(out.status, 2)
    ref, rst = O.csv_parse(data, ["f64", "i32"])
    assert st["error"] == rst["error"] == 0 and st["n_records"] == rst["n_records"] == 300
    got = out.results(st)
    assert np.array_equal(got[0].cpu().numpy(), ref[0]) and np.array_equal(got[1].cpu().numpy(), ref[1])
    assert pp.debug_long_fields() == 300
