"""Pins of the CPU oracle against what the pages and mathematics fix.

Nothing here uses the GPU library's arithmetic: expected values come from
the pages' worked examples (tests/golden), exhaustive enumeration, closed
forms, independent library routines (Python's float() and int()), and the
generator's record of what it wrote.
"""
import itertools
import random

import numpy as np
import pytest

import datagen
import oracle as O

BITS = {"INVALID_INPUT": O.E_INVALID_INPUT, "BAD_END_STATE": O.E_BAD_END_STATE,
        "COLCOUNT": O.E_COLCOUNT, "NUM_SYNTAX": O.E_NUM_SYNTAX,
        "NUM_OVERFLOW": O.E_NUM_OVERFLOW}


def _records(cols, col_types, st):
    """Reassemble per-record field texts from oracle columns."""
    R = st["n_records"]
    out = []
    for r in range(R):
        row = []
        for c, t in enumerate(col_types):
            if t == "str":
                off, ch = cols[c]
                row.append(bytes(ch[off[r]:off[r + 1]]).decode("latin-1"))
            else:
                row.append(cols[c][r])
        out.append(row)
    return out


# --------------------------------------------------------------- golden
def test_golden_csv_cases(golden):
    for case in golden["csv_cases"]:
        data = case["input"].encode("latin-1")
        cols, st = O.csv_parse(data, case["col_types"])
        want_err = 0
        for b in case.get("error_bits", []):
            want_err |= BITS[b]
        assert st["error"] == want_err, case["cite"]
        if "first_error_offset" in case:
            assert st["first_error_offset"] == case["first_error_offset"], case["cite"]
        if "records" in case:
            assert st["n_records"] == len(case["records"])
            got = _records(cols, case["col_types"], st)
            for r, rec in enumerate(case["records"]):
                for c, v in enumerate(rec):
                    t = case["col_types"][c]
                    if t == "str":
                        assert got[r][c] == v, case["cite"]
                    else:
                        assert int(got[r][c]) == int(v), case["cite"]
                # missing fields take the default
                for c in range(len(rec), len(case["col_types"])):
                    t = case["col_types"][c]
                    assert (got[r][c] == "") if t == "str" else (got[r][c] == 0)
        if "fields_per_record" in case:
            _, tg, _ = O.tags(data)
            nf = []
            k = 0
            for t in tg:
                if t == O.TAG_FD:
                    k += 1
                elif t == O.TAG_RD:
                    nf.append(k + 1)
                    k = 0
            assert nf == case["fields_per_record"], case["cite"]


def test_golden_column_offsets(golden):
    for case in golden["column_offset_cases"]:
        chunk = case["chunk"].encode()
        _, tg, _ = O.tags(chunk)   # the chunk starts at a record boundary
        is_abs, o = False, 0
        for t in tg:
            if t == O.TAG_RD:
                is_abs, o = True, 0
            elif t == O.TAG_FD:
                o += 1
        assert (is_abs, o) == (case["is_abs"], case["offset"]), case["cite"]


def test_golden_lexer_cases(golden):
    kinds = datagen.TOKEN_KINDS
    for case in golden["lexer_cases"]:
        data = bytes.fromhex(case["input_hex"]) if "input_hex" in case else case["input"].encode()
        (ids, starts, lens), st = O.tokenize(data)
        assert st["error"] == 0, case["cite"]
        got = [[kinds[i], int(n)] for i, n in zip(ids, lens)]
        assert got == case["tokens"], case["cite"]


def test_golden_arrow_layout(golden):
    for case in golden["arrow_cases"]:
        data = ("\n".join(case["strings"]) + "\n").encode()
        cols, st = O.csv_parse(data, ["str"])
        off, ch = cols[0]
        assert off.tolist() == case["offsets"], case["cite"]
        assert bytes(ch) == case["chars"].encode(), case["cite"]


# ---------------------------------------------------------- brute force
def test_bruteforce_csv_len8():
    """Every string of length 1..8 over one byte per symbol group: the
    scan-derived chunk start states and column offsets equal the sequential
    walk for every chunk size 1..8 (ParPaRaw Sections 3.1-3.2)."""
    bad, checked = O.bruteforce(O.KIND_CSV, b'",\na', 8)
    assert checked == sum(4 ** k for k in range(1, 9))
    assert bad == 0


def test_bruteforce_lexer_len6():
    alpha = b' {"\\-+01.ex'   # one byte per lexer symbol group (11 groups)
    assert len(alpha) == 11
    bad, checked = O.bruteforce(O.KIND_LEX, alpha, 6)
    assert checked == sum(11 ** k for k in range(1, 7))
    assert bad == 0


def test_bruteforce_detects_wrong_composition_order():
    """The brute force is not vacuous: composing in the wrong order (b o a)
    breaks the scan-vs-sequential equality on some input."""
    def chunk_starts_wrong(data, chunk):
        pre = np.arange(5, dtype=np.uint8)
        out = []
        for off in range(0, len(data), chunk):
            out.append(int(pre[0]))
            stv = O.stv(data[off:off + chunk])
            pre = O.compose(stv, pre)     # wrong order
        return out
    found = False
    for s in itertools.product(b'",\na', repeat=4):
        data = bytes(s)
        sb, _, _ = O.tags(data)
        for ch in (1, 2):
            seq = [int(sb[i]) for i in range(0, len(data), ch)]
            if chunk_starts_wrong(data, ch) != seq:
                found = True
                break
        if found:
            break
    assert found


def _closure(gens, cap):
    seen = {bytes(g) for g in gens}
    frontier = list(seen)
    while frontier and len(seen) < cap:
        nxt = []
        for a in frontier:
            for g in gens:
                c = bytes(O.compose(np.frombuffer(a, np.uint8), g))
                if c not in seen:
                    seen.add(c)
                    nxt.append(c)
        frontier = nxt
    return [np.frombuffer(x, np.uint8) for x in seen]


def test_composite_associative_csv_closure():
    """The composite operation is associative with the identity vector as
    unit on the whole monoid the CSV symbol groups generate."""
    gens = [O.stv(bytes([b])) for b in b'",\na']
    M = _closure(gens, 10_000)
    assert len(M) < 10_000
    ident = np.arange(5, dtype=np.uint8)
    for a in M:
        assert np.array_equal(O.compose(ident, a), a)
        assert np.array_equal(O.compose(a, ident), a)
    for a, b, c in itertools.product(M, repeat=3):
        assert np.array_equal(O.compose(O.compose(a, b), c), O.compose(a, O.compose(b, c)))


def test_composite_matches_concatenation_lexer():
    """STV(xy) = STV(x) o STV(y) on random lexer chunks (|S| = 16)."""
    rng = random.Random(7)
    alpha = b' {"\\-+01.exa]:,E'
    for _ in range(3000):
        x = bytes(rng.choice(alpha) for _ in range(rng.randint(0, 12)))
        y = bytes(rng.choice(alpha) for _ in range(rng.randint(0, 12)))
        a, b = O.stv(x, kind=O.KIND_LEX), O.stv(y, kind=O.KIND_LEX)
        assert np.array_equal(O.stv(x + y, kind=O.KIND_LEX), O.compose(a, b))


def test_composite_associative_lexer_sample():
    gens = [O.stv(bytes([b]), kind=O.KIND_LEX) for b in b' {"\\-+01.ex']
    M = _closure(gens, 3000)
    rng = random.Random(3)
    for _ in range(20000):
        a, b, c = (M[rng.randrange(len(M))] for _ in range(3))
        assert np.array_equal(O.compose(O.compose(a, b), c), O.compose(a, O.compose(b, c)))


# ------------------------------------------------------------- numerics
INT_CASES = [
    ("i8", b"127", 127, 0), ("i8", b"-128", -128, 0), ("i8", b"128", 0, O.E_NUM_OVERFLOW),
    ("i8", b"-129", 0, O.E_NUM_OVERFLOW), ("i8", b"+5", 5, 0), ("i8", b"007", 7, 0),
    ("i32", b"2147483647", 2**31 - 1, 0), ("i32", b"-2147483648", -2**31, 0),
    ("i32", b"2147483648", 0, O.E_NUM_OVERFLOW),
    ("i64", b"9223372036854775807", 2**63 - 1, 0),
    ("i64", b"-9223372036854775808", -2**63, 0),
    ("i64", b"9223372036854775808", 0, O.E_NUM_OVERFLOW),
    ("i64", b"99999999999999999999999", 0, O.E_NUM_OVERFLOW),
    ("i32", b"", 0, 0), ("i32", b"+", 0, O.E_NUM_SYNTAX), ("i32", b"-", 0, O.E_NUM_SYNTAX),
    ("i32", b"1.5", 0, O.E_NUM_SYNTAX), ("i32", b"1e3", 0, O.E_NUM_SYNTAX),
    ("i32", b" 1", 0, O.E_NUM_SYNTAX), ("i32", b"--1", 0, O.E_NUM_SYNTAX),
    ("i64", b"99999999999999999999999x", 0, O.E_NUM_SYNTAX),
    ("i32", b'"42"', 42, 0),
]


@pytest.mark.parametrize("ty,text,val,err", INT_CASES)
def test_int_conversion(ty, text, val, err):
    cols, st = O.csv_parse(text + b"\n", [ty])
    assert st["error"] == err
    assert int(cols[0][0]) == val


FLOAT_OK = [b"0", b"-0", b"1.5", b".5", b"5.", b"1e5", b"1E+05", b"-2.5e-3", b"123456789012345678901234567890",
            b"0.1", b"1e308", b"1e309", b"-1e400", b"1e-320", b"2.2250738585072014e-308",
            b"4.9406564584124654e-324", b"2.4703282292062327e-324", b"2.4703282292062328e-324",
            b"9007199254740993", b"0.000000000000000000000000000001", b"179769313486231580793728971405301e276",
            b"1.7976931348623157e308", b"1.7976931348623159e308", b'"3.25"', b"00001.000"]
FLOAT_BAD = [b"+", b".", b"e5", b"1e", b"1e+", b"1.2.3", b"inf", b"nan", b"0x1p3", b"1,0", b" 1", b"1 ", b"--1",
             b"+.e1"]


@pytest.mark.parametrize("text", FLOAT_OK)
def test_float_conversion_matches_python(text):
    """Python's float() is an independent correctly rounded conversion."""
    field = text + b"\n"
    cols, st = O.csv_parse(field, ["f64"]) if b"," not in text else O.csv_parse(field, ["f64"])
    assert st["error"] == 0
    want = float(text.strip(b'"').decode())
    got = float(cols[0][0])
    assert got == want or (np.isnan(got) and np.isnan(want))
    assert np.signbit(got) == np.signbit(want)


@pytest.mark.parametrize("text", FLOAT_BAD)
def test_float_syntax_errors(text):
    if b"," in text:
        cols, st = O.csv_parse(b'"' + text + b'"\n', ["f64"])
    else:
        cols, st = O.csv_parse(text + b"\n", ["f64"])
    assert st["error"] == O.E_NUM_SYNTAX
    assert st["first_error_offset"] == 0
    assert float(cols[0][0]) == 0.0


def test_float_random_strings_match_python():
    rng = random.Random(11)
    lines = []
    vals = []
    for _ in range(20000):
        mant = "".join(rng.choice("0123456789") for _ in range(rng.randint(1, 25)))
        if rng.random() < 0.5:
            k = rng.randint(0, len(mant))
            mant = mant[:k] + "." + mant[k:]
            if mant == ".":
                mant = "0."
        s = ("-" if rng.random() < 0.3 else "") + mant
        if rng.random() < 0.5:
            s += rng.choice("eE") + rng.choice(["", "+", "-"]) + str(rng.randint(0, 340))
        lines.append(s)
        vals.append(float(s))
    data = ("\n".join(lines) + "\n").encode()
    cols, st = O.csv_parse(data, ["f64"])
    assert st["error"] == 0
    assert np.array_equal(cols[0].view(np.uint64), np.array(vals).view(np.uint64))


# --------------------------------------------------- generator round trip
@pytest.mark.parametrize("name", ["csv4_1mib", "csv16_256mib", "csv3_1gib", "csv18_2gib"])
def test_generator_roundtrip_csv(name):
    w = datagen.WORKLOADS[name]
    data, info, side = datagen.generate(name, target=300_000, sidecar=True)
    truth = datagen.sidecar_fields(side)
    cols, st = O.csv_parse(data, w["cols"])
    assert st["error"] == 0
    assert st["n_records"] == info["n_records"]
    nc = len(w["cols"])
    assert len(truth) == info["n_records"] * nc == info["n_fields"]
    for c, t in enumerate(w["cols"]):
        col_truth = truth[c::nc]
        if t == "str":
            off, ch = cols[c]
            got = [bytes(ch[off[r]:off[r + 1]]) for r in range(info["n_records"])]
            assert got == col_truth
            assert st["chars_len"][c] == info["col_value_bytes"][c]
        elif t == "f64":
            want = np.array([float(x) for x in col_truth])
            assert np.array_equal(cols[c].view(np.uint64), want.view(np.uint64))
        else:
            assert cols[c].tolist() == [int(x) for x in col_truth]


def test_generator_roundtrip_tokens():
    data, info, side = datagen.generate("json_2gib", target=300_000, sidecar=True)
    truth = datagen.sidecar_tokens(side)
    (ids, starts, lens), st = O.tokenize(data)
    assert st["error"] == 0
    assert st["n_tokens"] == info["n_tokens"] == len(truth)
    # the generator emits each whitespace run as one token, but a run at a
    # token boundary may touch the next run only through non-ws tokens
    assert [(int(i), int(n)) for i, n in zip(ids, lens)] == truth


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("name", ["csv4_1mib", "csv16_256mib", "csv3_1gib", "csv18_2gib"])
def test_invariants_csv(name):
    w = datagen.WORKLOADS[name]
    data, info, _ = datagen.generate(name, target=200_000)
    sb, tg, end = O.tags(data)
    nfd = int(np.count_nonzero(tg == O.TAG_FD))
    nrd = int(np.count_nonzero(tg == O.TAG_RD))
    nctrl = int(np.count_nonzero(tg == O.TAG_CTRL))
    ndata = int(np.count_nonzero(tg == O.TAG_DATA))
    assert nfd + nrd + nctrl + ndata == data.size          # byte conservation
    assert nfd + nrd == info["n_fields"]                    # fields = #FD + #RD
    cols, st = O.csv_parse(data, w["cols"])
    assert st["n_records"] == nrd                           # input ends with '\n'
    total_value = 0
    for c, t in enumerate(w["cols"]):
        if t == "str":
            off, ch = cols[c]
            assert off[0] == 0 and np.all(np.diff(off) >= 0) and off[-1] == ch.size
            total_value += ch.size
    if all(t == "str" for t in w["cols"]):
        assert total_value == ndata


def test_invariants_tokens():
    data, info, _ = datagen.generate("json_2gib", target=200_000)
    (ids, starts, lens), st = O.tokenize(data)
    assert st["error"] == 0
    assert starts[0] == 0 and np.all(np.diff(starts.astype(np.int64)) > 0)
    assert int(lens.astype(np.int64).sum()) == data.size
    ws = ids == 9
    assert not np.any(ws[1:] & ws[:-1])                    # no two adjacent ws tokens
    assert np.array_equal(starts[1:], starts[:-1] + lens[:-1])


def test_generator_workload3_quoted_fraction():
    data, info, _ = datagen.generate("csv3_1gib", target=32 << 20)
    frac = info["quoted_bytes"] / info["n_bytes"]
    assert 0.80 <= frac <= 0.90


def test_edge_inputs():
    cols, st = O.csv_parse(b"", ["str"])
    assert st["n_records"] == 0 and st["error"] == 0 and cols[0][0].tolist() == [0]
    cols, st = O.csv_parse(b"abc", ["str"])          # unterminated tail is a record
    assert st["n_records"] == 1 and bytes(cols[0][1]) == b"abc"
    cols, st = O.csv_parse(b"\n\n", ["str"])         # empty lines: one empty field each
    assert st["n_records"] == 2 and cols[0][0].tolist() == [0, 0, 0]
    cols, st = O.csv_parse(b"a,b,c\n", ["str", "str"])   # extra field dropped
    assert st["error"] == O.E_COLCOUNT and st["first_error_offset"] == 5
    assert bytes(cols[1][1]) == b"b"
    cols, st = O.csv_parse(b'"a"', ["str"])          # ends in ESC: accepting
    assert st["error"] == 0 and bytes(cols[0][1]) == b"a"
    cols, st = O.csv_parse(b'"a"x\n', ["str"])       # other after closing quote
    assert st["error"] == O.E_INVALID_INPUT and st["first_error_offset"] == 3


# ------------------------------------------------------------ timestamps
# Python's calendar.timegm (proleptic Gregorian, seconds since 1970-01-01
# 00:00:00) is an independent implementation of the same day count.
def _timegm(y, mo, d, h=0, mi=0, s=0):
    import calendar
    return calendar.timegm((y, mo, d, h, mi, s, 0, 0, 0))


TS_OK = [
    (b"1970-01-01 00:00:00", 0), (b"1970-01-01", 0), (b"1969-12-31 23:59:59", -1),
    (b"2000-02-29 12:34:56", _timegm(2000, 2, 29, 12, 34, 56)),
    (b"2024-02-29", _timegm(2024, 2, 29)), (b"2021-03-01 00:00:01", _timegm(2021, 3, 1, 0, 0, 1)),
    (b"0001-01-01 00:00:00", _timegm(1, 1, 1)), (b"9999-12-31 23:59:59", _timegm(9999, 12, 31, 23, 59, 59)),
    (b"1600-02-29", _timegm(1600, 2, 29)),
    # year 0 (a leap year of the proleptic calendar) is 719528 days before 1970
    (b"0000-01-01 00:00:00", -719528 * 86400), (b"0000-02-29", -719528 * 86400 + 59 * 86400),
    (b'"2020-07-04 01:02:03"', _timegm(2020, 7, 4, 1, 2, 3)), (b"", 0),
]
TS_BAD = [b"1900-02-29", b"2023-02-29", b"2021-04-31", b"2021-13-01", b"2021-00-10",
          b"2021-01-00", b"2021-01-01 24:00:00", b"2021-01-01 23:60:00", b"2021-01-01 23:59:60",
          b"2021-1-01", b"2021/01/01", b"2021-01-01T00:00:00", b"2021-01-01 00:00", b" 2021-01-01",
          b"2021-01-01 ", b"-021-01-01", b"2021-01-01 00:00:0x", b"20210101"]


@pytest.mark.parametrize("text,val", TS_OK)
def test_timestamp_conversion_matches_timegm(text, val):
    cols, st = O.csv_parse(text + b"\n", ["ts"])
    assert st["error"] == 0
    assert int(cols[0][0]) == val


@pytest.mark.parametrize("text", TS_BAD)
def test_timestamp_syntax_errors(text):
    cols, st = O.csv_parse(b"7," + text + b"\n", ["i32", "ts"])
    assert st["error"] == O.E_NUM_SYNTAX and st["first_error_offset"] == 2
    assert int(cols[1][0]) == 0


def test_timestamps_random_days_match_timegm():
    import random
    rng = random.Random(7)
    lines, want = [], []
    for _ in range(3000):
        y, mo = rng.randint(1, 9999), rng.randint(1, 12)
        d = rng.randint(1, 28 if mo == 2 else 30)
        h, mi, s = rng.randint(0, 23), rng.randint(0, 59), rng.randint(0, 59)
        lines.append(b"%04d-%02d-%02d %02d:%02d:%02d" % (y, mo, d, h, mi, s))
        want.append(_timegm(y, mo, d, h, mi, s))
    cols, st = O.csv_parse(b"\n".join(lines) + b"\n", ["ts"])
    assert st["error"] == 0
    assert cols[0].tolist() == want


# ------------------------------------------------------------ CRLF line ends
# Reading: with CRLF line ends, a carriage return outside quotes is a
# control symbol (dropped from the value, the field stays open); inside
# quotes it is data.  Record delimiter LF.
CRLF_CASES = [
    (b"a,b\r\nc,d\r\n", [[b"a", b"b"], [b"c", b"d"]], 0),
    (b'"x",y\r\n', [[b"x", b"y"]], 0),
    (b'"a\r\nb",c\r\n', [[b"a\r\nb", b"c"]], 0),            # CRLF inside quotes is data
    (b"a,\r\n,\r\n", [[b"a", b""], [b"", b""]], 0),
    (b"\r\n\r\n", [[b""], [b""]], 0),                       # empty lines
    (b"a\rb,c\r\n", [[b"ab", b"c"]], 0),                    # a bare CR is dropped too
    (b"a,b\r\nc,d", [[b"a", b"b"], [b"c", b"d"]], 0),       # no final line end
    (b"a,b\r", [[b"a", b"b"]], 0),
]


@pytest.mark.parametrize("data,want,err", CRLF_CASES)
def test_crlf_cases(data, want, err):
    n = len(want[0])
    cols, st = O.csv_parse(data, ["str"] * n, crlf=True)
    assert st["error"] == err and st["n_records"] == len(want)
    for c in range(n):
        offs, chars = cols[c]
        got = [bytes(chars[offs[r]:offs[r + 1]]) for r in range(len(want))]
        assert got == [row[c] for row in want]


def test_crlf_invalid_after_cr():
    # a quote after a dropped CR is a quote inside an unquoted field
    _, st = O.csv_parse(b'"a"\r"b"\r\n', ["str"], crlf=True)
    assert st["error"] & O.E_INVALID_INPUT and st["first_error_offset"] == 4
    # without CRLF handling the CR is plain data, so "a" followed by it is invalid at 3
    _, st = O.csv_parse(b'"a"\r\n', ["str"])
    assert st["error"] & O.E_INVALID_INPUT and st["first_error_offset"] == 3


def test_crlf_equals_lf_after_removing_unquoted_cr():
    """On generated quoted CSV, CRLF line ends parse to the same columns as
    the LF original (quoted newlines keep their bytes in both)."""
    data, info, _ = datagen.generate("csv4_1mib", target=64 * 1024)
    lf = bytes(data)
    # add a CR before every record delimiter only: walk the oracle's tags
    _, tags, _ = O.tags(lf)
    out = bytearray()
    for b, t in zip(lf, tags):
        if t == O.TAG_RD:
            out += b"\r"
        out.append(b)
    cols = datagen.WORKLOADS["csv4_1mib"]["cols"]
    a, sa = O.csv_parse(lf, cols)
    b, sb = O.csv_parse(bytes(out), cols, crlf=True)
    assert sa == sb and sa["error"] == 0
    for (oa, ca), (ob, cb) in zip(a, b):
        assert np.array_equal(oa, ob) and np.array_equal(ca, cb)


def test_bruteforce_csv_crlf_len7():
    """The CRLF variant's scan-derived chunk start states and column offsets
    equal the sequential walk on every string of length 1..7 over one byte
    per symbol group."""
    bad, checked = O.bruteforce(O.KIND_CSV_CRLF, b'",\n\ra', 7)
    assert checked == sum(5 ** k for k in range(1, 8))
    assert bad == 0


# ------------------------------------------------- column-count inference
COUNT_CASES = [
    (b"", (0, 0), 0, 0),
    (b"1,Apples\n2\n", (1, 2), 2, 0),                  # the pages' example of varying counts
    (b"a,b,c\n", (3, 3), 1, 0),
    (b"\n\n", (1, 1), 2, 0),                          # empty lines: one empty field each
    (b"a,b\nc", (1, 2), 2, 0),                        # a tail without a delimiter
    (b'a,"x,\ny",c\n,\n', (2, 3), 2, 0),              # delimiters inside quotes are data
    (b",,,,\n", (5, 5), 1, 0),
    (b'"ab', (0, 0), 0, O.E_BAD_END_STATE),           # ends inside quotes
]


@pytest.mark.parametrize("data,mm,recs,err", COUNT_CASES)
def test_count_fields_cases(data, mm, recs, err):
    got, st = O.count_fields(data)
    assert st["error"] == err
    if not err:
        assert got == mm and st["n_records"] == recs


def test_count_fields_invalid_offset():
    _, st = O.count_fields(b'ab,c"d\n')
    assert st["error"] == O.E_INVALID_INPUT and st["first_error_offset"] == 4


@pytest.mark.parametrize("name", ["csv4_1mib", "csv16_256mib", "csv3_1gib", "csv18_2gib"])
def test_count_fields_generated_schema(name):
    """The generator writes a fixed number of columns per record, so the
    inferred min and max are both that number, and the record count is the
    generator's."""
    data, info, _ = datagen.generate(name, target=1 << 20)
    (mn, mx), st = O.count_fields(data)
    n = len(datagen.WORKLOADS[name]["cols"])
    assert st["error"] == 0 and (mn, mx) == (n, n) and st["n_records"] == info["n_records"]


def test_count_fields_agrees_with_a_row_split():
    """Min and max fields equal those of an independent split of each row on
    its unquoted commas (rows whose quotes are balanced)."""
    rng = random.Random(3)
    rows = []
    for _ in range(400):
        k = rng.randint(1, 9)
        rows.append(b",".join(rng.choice([b"x", b'"a,b"', b"", b'"\n"']) for _ in range(k)))
    data = b"\n".join(rows) + b"\n"
    (mn, mx), st = O.count_fields(data)
    # recount independently: split each row on its unquoted commas
    def nfields(r):
        n, q = 1, False
        for ch in r:
            if ch == ord('"'):
                q = not q
            elif ch == ord(",") and not q:
                n += 1
        return n
    counts = [nfields(r) for r in rows]
    assert st["error"] == 0 and (mn, mx) == (min(counts), max(counts)) and st["n_records"] == 400
