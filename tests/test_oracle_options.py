"""Pins for the oracle's parse options (ParPaRaw Section 4): default values
for empty and missing numeric fields, rejecting records whose field count
differs from the schema's, skipping records and skipping rows.  The
expected values come from the page's own example, from hand cases, and from
Python's csv module (an independent RFC-4180 reader) with plain list
filtering, never from the oracle itself."""
import csv
import io
import random
import struct

import numpy as np
import pytest

import oracle as O


def _bits(x):
    return struct.unpack("<Q", struct.pack("<d", x))[0]


def _fields(cols, st, k):
    out = []
    for r in range(st["n_records"]):
        row = []
        for c in range(k):
            offs, chars = cols[c]
            row.append(bytes(chars[offs[r]:offs[r + 1]]).decode())
        out.append(row)
    return out


def _csv_rows(rng, n_rows, max_fields, alpha="ab,\"\n x1"):
    rows = []
    for _ in range(n_rows):
        k = rng.randint(1, max_fields)
        rows.append(["".join(rng.choice(alpha) for _ in range(rng.randint(0, 5)))
                     for _ in range(k)])
    return rows


def _write(rows):
    buf = io.StringIO()
    csv.writer(buf, lineterminator="\n").writerows(rows)
    return buf.getvalue().encode()


# ------------------------------------------------------------ defaults
def test_defaults_for_empty_and_missing_fields():
    """Section 4, "Default values for empty strings": an empty field, and a
    field missing from a short record, take the column's default."""
    data = b'1,,2.5\n4\n,"",\n'
    types = ["i64", "i32", "f64"]
    d = [7, -3 & 0xFFFFFFFFFFFFFFFF, _bits(1.5)]
    cols, st = O.csv_parse(data, types, defaults=d)
    assert st["n_records"] == 3
    assert st["error"] == O.E_COLCOUNT and st["first_error_offset"] == 8  # "4\n" has 1 field
    assert cols[0].tolist() == [1, 4, 7]
    assert cols[1].tolist() == [-3, -3, -3]      # empty, missing, quoted empty
    assert cols[2].tolist() == [2.5, 1.5, 1.5]
    # without defaults the default is 0
    cols, st = O.csv_parse(data, types)
    assert cols[0].tolist() == [1, 4, 0] and cols[1].tolist() == [0, 0, 0]
    assert cols[2].tolist() == [2.5, 0.0, 0.0]


def test_defaults_truncate_to_the_column_width():
    cols, _ = O.csv_parse(b",\n", ["i8", "i32"], defaults=[0x1FF, 0x1_0000_0005])
    assert cols[0].tolist() == [-1] and cols[1].tolist() == [5]


def test_defaults_do_not_touch_strings_or_values():
    cols, st = O.csv_parse(b"a,1\n,2\n", ["str", "i64"], defaults=[99, 42])
    assert st["error"] == 0
    offs, chars = cols[0]
    assert offs.tolist() == [0, 1, 1] and bytes(chars) == b"a"
    assert cols[1].tolist() == [1, 2]


# ------------------------------------------------------------ reject
def test_reject_on_the_pages_example(golden):
    """The page's example of a record with fewer fields ("1,Apples\\n2\\n"):
    with two columns and rejection, only the first record is emitted."""
    data = b"1,Apples\n2\n"
    cols, st = O.csv_parse(data, ["i64", "str"], reject=True)
    assert st["n_records"] == 1 and st["n_dropped"] == 1
    assert st["error"] == O.E_COLCOUNT and st["first_error_offset"] == 10
    assert cols[0].tolist() == [1]
    offs, chars = cols[1]
    assert offs.tolist() == [0, 6] and bytes(chars) == b"Apples"


@pytest.mark.parametrize("seed", range(5))
def test_reject_matches_csv_module_filter(seed):
    rng = random.Random(seed)
    k = rng.randint(1, 4)
    rows = _csv_rows(rng, 500, k + 1)
    data = _write(rows)
    ref = list(csv.reader(io.StringIO(data.decode(), newline="")))
    keep = [r for r in ref if len(r) == k]
    cols, st = O.csv_parse(data, ["str"] * k, reject=True)
    assert st["n_records"] == len(keep) and st["n_dropped"] == len(ref) - len(keep)
    assert _fields(cols, st, k) == keep
    assert bool(st["error"] & O.E_COLCOUNT) == (len(keep) != len(ref))


# ------------------------------------------------------------ skip records
@pytest.mark.parametrize("seed", range(5))
def test_skip_records_matches_csv_module_filter(seed):
    rng = random.Random(50 + seed)
    k = rng.randint(1, 4)
    rows = [r[:k] + [""] * (k - len(r[:k])) for r in _csv_rows(rng, 400, k)]
    data = _write(rows)
    ref = list(csv.reader(io.StringIO(data.decode(), newline="")))
    skip = sorted(rng.sample(range(len(ref)), 40)) + [len(ref) + 5]   # one past the end
    cols, st = O.csv_parse(data, ["str"] * k, skip_records=skip)
    keep = [r for i, r in enumerate(ref) if i not in set(skip)]
    assert st["error"] == 0
    assert st["n_records"] == len(keep) and st["n_dropped"] == 40
    assert _fields(cols, st, k) == keep


def test_skipped_records_report_no_errors():
    """A skipped record's fields are irrelevant: no conversion, no column
    count check; the DFA still checks the input."""
    data = b"h1,h2\n1,2\n3\nx,4\n"
    cols, st = O.csv_parse(data, ["i32", "i32"], skip_records=[0, 2])
    assert st["n_records"] == 2 and st["n_dropped"] == 2
    assert st["error"] == O.E_NUM_SYNTAX and st["first_error_offset"] == 12
    assert cols[0].tolist() == [1, 0] and cols[1].tolist() == [2, 4]


# ------------------------------------------------------------ skip rows
def test_skip_rows_are_lines_not_records():
    """Rows are lines: a quoted newline splits a record into two rows, and
    skipping a row removes its bytes before the DFA runs (Section 4)."""
    data = b'a,"x\ny"\nb,z\nc,w'
    assert bytes(O.skip_rows(data, [1])) == b'a,"x\nb,z\nc,w'
    assert bytes(O.skip_rows(data, [0, 3])) == b'y"\nb,z\n'
    assert bytes(O.skip_rows(data, [])) == data
    assert bytes(O.skip_rows(data, [7, 9])) == data


@pytest.mark.parametrize("seed", range(4))
def test_skip_rows_matches_line_filter(seed):
    rng = random.Random(90 + seed)
    lines = [("".join(rng.choice("abc,1") for _ in range(rng.randint(0, 8)))).encode()
             for _ in range(300)]
    data = b"\n".join(lines)                       # no final newline
    skip = sorted(rng.sample(range(len(lines)), 30))
    kept = [ln for i, ln in enumerate(lines) if i not in set(skip)]
    want = b"".join(ln + b"\n" for ln in kept[:-1]) + (kept[-1] if 299 not in skip else kept[-1] + b"\n")
    if 299 in skip:
        want = b"".join(ln + b"\n" for ln in kept)
    assert bytes(O.skip_rows(data, skip)) == want
    # and the parse of the filtered input is the parse of the kept lines
    cols, st = O.csv_parse(data, ["str"] * 3, skip_rows_=skip)
    ref_cols, ref_st = O.csv_parse(want, ["str"] * 3)
    assert st == ref_st


# ------------------------------------------------------------ type inference
@pytest.mark.parametrize("text,want", [
    (b"0", "i8"), (b"127", "i8"), (b"-128", "i8"), (b"+5", "i8"),
    (b"128", "i32"), (b"-129", "i32"), (b"2147483647", "i32"), (b"-2147483648", "i32"),
    (b"2147483648", "i64"), (b"-2147483649", "i64"), (b"9223372036854775807", "i64"),
    (b"-9223372036854775808", "i64"),
    (b"9223372036854775808", "f64"), (b"-9223372036854775809", "f64"),
    (b"1.0", "f64"), (b".5", "f64"), (b"7.", "f64"), (b"1e5", "f64"), (b"-2.5E-3", "f64"),
    (b"abc", "str"), (b"1,5", None), (b"1.2.3", "str"), (b"--1", "str"), (b"1e", "str"),
    (b"0x10", "str"), (b"inf", "str"), (b"", "i8"), (b'"12"', "i8"), (b'"1""2"', "str"),
])
def test_infer_single_values(text, want):
    """The smallest type backing one value (ParPaRaw Section 4, "Type
    inference"): integer ranges at their exact edges, the float grammar,
    quoted values read without their quotes."""
    if want is None:  # a field delimiter: two one-digit columns
        assert O.infer_types(text + b"\n", 2)[0] == ["i8", "i8"]
        return
    types, st = O.infer_types(text + b"\n", 1)
    assert st["error"] == 0 and types == [want]


def test_infer_takes_the_largest_per_column():
    data = b"1,2.5,x,,\n-200,3,,\n99999999999,1e5,\"\"\n"
    types, st = O.infer_types(data, 5)
    assert types == ["i64", "f64", "str", "i8", "i8"] and st["n_records"] == 3


@pytest.mark.parametrize("seed", range(4))
def test_infer_of_concatenation_is_the_maximum(seed):
    """Inference is a reduction with the maximum over a total order: the
    type of a column over two inputs is the larger of the two types."""
    rng = random.Random(300 + seed)
    order = ["i8", "i32", "i64", "f64", "str"]
    pool = [b"1", b"-7", b"300", b"-40000", b"5000000000", b"2.5", b"1e9", b"", b"ab", b'"9"']

    def part():
        return b"".join(b",".join(rng.choice(pool) for _ in range(3)) + b"\n"
                        for _ in range(rng.randint(1, 20)))
    a, b = part(), part()
    ta, _ = O.infer_types(a, 3)
    tb, _ = O.infer_types(b, 3)
    tab, _ = O.infer_types(a + b, 3)
    assert tab == [max(x, y, key=order.index) for x, y in zip(ta, tb)]
