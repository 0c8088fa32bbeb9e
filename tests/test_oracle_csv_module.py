"""The oracle against Python's csv module, an independent RFC-4180 reader
and writer: rows written by csv.writer (minimal quoting, doubled quotes,
delimiters and line breaks inside quoted fields) parse back to the same
fields, with LF and with CRLF line ends, and the column-count inference
agrees with the rows' lengths."""
import csv
import io
import random

import pytest

import oracle as O

ALPHA = "ab,\"\n\r x1"


def _rows(rng, n_rows, max_fields):
    rows = []
    for _ in range(n_rows):
        k = rng.randint(1, max_fields)
        rows.append(["".join(rng.choice(ALPHA) for _ in range(rng.randint(0, 6)))
                     for _ in range(k)])
    return rows


def _fields(cols, st, k):
    out = []
    for r in range(st["n_records"]):
        row = []
        for c in range(k):
            offs, chars = cols[c]
            row.append(bytes(chars[offs[r]:offs[r + 1]]).decode())
        out.append(row)
    return out


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("crlf", [False, True])
def test_csv_writer_round_trip(seed, crlf):
    rng = random.Random(seed)
    k = rng.randint(1, 5)
    rows = [_rows(rng, k, 1) for _ in range(300)]  # k one-field rows, as one row of k fields
    rows = [[f[0] for f in r] for r in rows]
    buf = io.StringIO()
    csv.writer(buf, lineterminator="\r\n" if crlf else "\n").writerows(rows)
    data = buf.getvalue().encode()
    cols, st = O.csv_parse(data, ["str"] * k, crlf=crlf)
    assert st["error"] == 0 and st["n_records"] == len(rows)
    assert _fields(cols, st, k) == rows
    # and the csv module reads the oracle's input the same way
    assert list(csv.reader(io.StringIO(data.decode(), newline=""))) == rows


@pytest.mark.parametrize("seed", range(6))
def test_count_fields_matches_csv_module(seed):
    rng = random.Random(100 + seed)
    rows = _rows(rng, 400, 9)
    buf = io.StringIO()
    csv.writer(buf, lineterminator="\n").writerows(rows)
    data = buf.getvalue().encode()
    (mn, mx), st = O.count_fields(data)
    lens = [len(r) for r in csv.reader(io.StringIO(data.decode(), newline=""))]
    assert st["error"] == 0 and st["n_records"] == len(rows)
    assert (mn, mx) == (min(lens), max(lens))
