"""GPU parity: libpp (through its C ABI) against the CPU oracle, element by
element, on seeded inputs spanning many tiles and ragged tails, plus the
edge cases of the method (empty input, tails without a delimiter, fields
crossing tiles, invalid input, column-count errors, capacity limits)."""
import random

import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import compare_csv, compare_tags, compare_tokens, run_gpu_csv, to_dev

pytestmark = pytest.mark.gpu
TILE = 16384


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)
    assert pp.tile_bytes() == TILE


def _rand_csv(rng, n, alpha=b'",\nab'):
    return bytes(rng.choice(alpha) for _ in range(n))


# ------------------------------------------------------------------ tags
@pytest.mark.parametrize("n", [0, 1, 31, 32, 33, 1000, TILE - 1, TILE, TILE + 1, 3 * TILE + 777])
def test_tags_csv_random(n):
    rng = random.Random(n)
    data = _rand_csv(rng, n, alpha=b'"' + b",\naaaaaaa")
    compare_tags(data)


@pytest.mark.parametrize("name", ["csv4_1mib", "csv3_1gib"])
def test_tags_csv_generated(name):
    data, _, _ = datagen.generate(name, target=5 * TILE + 123)
    compare_tags(data)
    compare_tags(data, offset=3)


@pytest.mark.parametrize("n", [0, 5, 4 * TILE + 9])
def test_tags_lexer(n):
    data, _, _ = datagen.generate("json_2gib", target=max(n, 1))
    compare_tags(data[:n], kind=O.KIND_LEX)
    rng = random.Random(n)
    junk = bytes(rng.choice(b' {"\\-+01.exa]:,') for _ in range(n))
    compare_tags(junk, kind=O.KIND_LEX)


# ---------------------------------------------------------------- parse
@pytest.mark.parametrize("name,target", [
    ("csv4_1mib", None),                 # the full 1 MiB workload
    ("csv4_1mib", 3 * TILE + 101),
    ("csv16_256mib", 2 << 20),
    ("csv16_256mib", 5 * TILE + 3),
    ("csv3_1gib", 4 << 20),
    ("csv3_1gib", 2 * TILE + 17),
    ("csv18_2gib", 2 << 20),
    ("csv18_2gib", TILE + 1),
])
def test_parse_workloads(name, target):
    data, info, _ = datagen.generate(name, target=target)
    st = compare_csv(data, datagen.WORKLOADS[name]["cols"])
    assert st["error"] == 0 and st["n_records"] == info["n_records"]


@pytest.mark.parametrize("name", ["csv16_256mib", "csv18_2gib"])
def test_parse_many_tiles(name):
    """About 40 MB: more than 2048 tiles, so the tile scan runs in several
    blocks chained by look-back and every warp of a scan block holds tiles."""
    data, info, _ = datagen.generate(name, target=40 << 20)
    st = compare_csv(data, datagen.WORKLOADS[name]["cols"])
    assert st["error"] == 0 and st["n_records"] == info["n_records"]


@pytest.mark.parametrize("shift", [0, 1, 13, 31])
def test_parse_quoted_newlines_everywhere(shift):
    """Quoted fields holding record delimiters, field delimiters and doubled
    quotes, with lengths that walk them across every chunk and tile offset."""
    rng = random.Random(shift)
    parts = [b'0,"' + b"p" * shift + b'",0.5\n']
    size = len(parts[0])
    while size < 3 * TILE + 500:
        k = rng.randrange(0, 70)
        body = bytes(rng.choice(b'ab\n,"') for _ in range(k)).replace(b'"', b'""')
        rec = b"%d,\"%s\",%d.5\n" % (rng.randrange(-99, 99), body, rng.randrange(1000))
        parts.append(rec)
        size += len(rec)
    data = b"".join(parts)
    compare_csv(data, ["i32", "str", "f64"])
    compare_csv(data, ["i32", "skip", "f64"])
    compare_csv(data, ["str", "str", "str"])


def test_parse_tiny_records():
    """Tiles with more fields than the per-tile field list holds."""
    data = b"".join(b"%d,%d\n" % (i % 10, i % 7) for i in range(3 * TILE // 4 + 9))
    compare_csv(data, ["i32", "i8"])
    compare_csv(data, ["str", "i64"])
    compare_csv(b"\n" * (2 * TILE + 3), ["str"])
    compare_csv(b",\n" * (2 * TILE + 3), ["str", "i32"])


@pytest.mark.parametrize("offset", [1, 7])
def test_parse_misaligned_input(offset):
    data, _, _ = datagen.generate("csv16_256mib", target=3 * TILE + 5)
    compare_csv(data, datagen.WORKLOADS["csv16_256mib"]["cols"], offset=offset)


def test_parse_empty_and_tiny():
    for data in [b"", b"a", b"\n", b",", b'"', b'""', b'"a"', b"a\n", b"a,b", b"\n\n\n", b",\n,,\n"]:
        compare_csv(data, ["str", "str"])


def test_parse_no_trailing_newline():
    data, _, _ = datagen.generate("csv18_2gib", target=3 * TILE)
    cols = datagen.WORKLOADS["csv18_2gib"]["cols"]
    compare_csv(bytes(data[:-1]), cols)          # last record unterminated
    compare_csv(bytes(data[:-7]), cols)


def test_parse_field_spanning_many_tiles():
    rng = random.Random(5)
    body = bytes(rng.choice(b"abc,\n\"") for _ in range(5 * TILE + 333))
    quoted = b'"' + body.replace(b'"', b'""') + b'"'
    data = b"1," + quoted + b",2\n3,x,4\n" + b"5," + quoted + b",6\n"
    compare_csv(data, ["i32", "str", "i32"])
    compare_csv(data, ["i32", "skip", "i8"])


@pytest.mark.parametrize("k", range(-6, 7))
def test_parse_tile_boundary_patterns(k):
    """Place quotes, doubled quotes and delimiters at every offset around the
    first tile boundary (and a numeric field straddling it)."""
    for pat in [b'"a,""b\nc"', b'""', b'"x"', b',\n', b'12345.678']:
        fill = TILE + k - 2
        head = (b"q" * (fill - 1)) + b","
        data = head + b'1,' + pat + b"\n7,8,9\n"
        if pat == b'12345.678':
            compare_csv(data, ["str", "i32", "f64"])
        else:
            compare_csv(data, ["str", "i32", "str"])


@pytest.mark.parametrize("pos", [0, 5, 31, 32, TILE - 1, TILE, TILE + 40, 2 * TILE + 3])
def test_parse_invalid_quote(pos):
    data, _, _ = datagen.generate("csv18_2gib", target=3 * TILE)
    b = bytearray(data)
    # put a quote right after an unquoted data byte -> invalid at that byte
    while b[pos - 1:pos] in (b",", b"\n") or pos == 0:
        pos += 1
    b[pos] = ord('"')
    st = compare_csv(bytes(b), datagen.WORKLOADS["csv18_2gib"]["cols"])
    assert st["error"] & pp.ERR_INVALID_INPUT and st["first_error_offset"] == pos


def test_parse_bad_end_state():
    data, _, _ = datagen.generate("csv4_1mib", target=2 * TILE)
    st = compare_csv(bytes(data) + b'a,"unterminated,\n', ["str"] * 4)
    assert st["error"] & pp.ERR_BAD_END_STATE


def test_parse_colcount_defaults():
    rows = [b"1,a,2.5", b"2", b"3,b", b"4,c,1e3,extra,more", b"", b"5,d,-0"]
    data = b"\n".join(rows) * 700 + b"\n"
    st = compare_csv(data, ["i64", "str", "f64"])
    assert st["error"] == pp.ERR_COLCOUNT


def test_parse_numeric_errors():
    rows = [b"1,2.5", b"x,1", b"99999999999,3", b"+,4", b"5,1.2.3", b'"6","7.5"', b"7,", b",8e1"]
    data = (b"\n".join(rows) + b"\n") * 900
    st = compare_csv(data, ["i32", "f64"])
    assert st["error"] == pp.ERR_NUM_SYNTAX | pp.ERR_NUM_OVERFLOW
    compare_csv(data, ["i8", "f64"])
    compare_csv(data, ["i64", "str"])


def test_parse_float_hard_cases():
    rng = random.Random(17)
    vals = ["0", "-0", "1e308", "1e309", "-1e400", "4.9406564584124654e-324",
            "2.4703282292062328e-324", "9007199254740993", "123456789012345678901234567890",
            "179769313486231580793728971405301e276", "1.7976931348623159e308",
            "0.000000000000000000000000000001", "2.2250738585072011e-308"]
    for _ in range(30000):
        mant = "".join(rng.choice("0123456789") for _ in range(rng.randint(1, 25)))
        if rng.random() < 0.5:
            k = rng.randint(0, len(mant))
            mant = mant[:k] + "." + mant[k:]
            if mant == ".":
                mant = "0."
        s = ("-" if rng.random() < 0.3 else "") + mant
        if rng.random() < 0.6:
            s += rng.choice("eE") + rng.choice(["", "+", "-"]) + str(rng.randint(0, 340))
        vals.append(s)
    data = ("\n".join(vals) + "\n").encode()
    compare_csv(data, ["f64"])


def test_parse_custom_delimiters():
    data, _, _ = datagen.generate("csv16_256mib", target=3 * TILE)
    b = bytes(data).replace(b",", b"|").replace(b"\n", b";")
    compare_csv(b, datagen.WORKLOADS["csv16_256mib"]["cols"], fd=b"|", rd=b";", quote=b'"')


def test_parse_random_small_inputs():
    rng = random.Random(99)
    for trial in range(300):
        n = rng.randint(0, 200)
        data = _rand_csv(rng, n, alpha=b'",\n1a-.')
        compare_csv(data, ["str", "i32", "f64"])


def test_parse_lookback_timeout_is_reported_and_recoverable():
    """A wait that runs out ends with an error status, not a hang: with the
    first tile withholding its look-back posts (flags nothing sets) and a
    short spin limit, the tiles after it give up and report the timeout;
    the next normal call on the same context is clean."""
    data = b"ab,cd\n" * ((40 << 20) // 6)  # > 2048 tiles: several scan blocks
    try:
        pp.debug_set_spin_limit(2000)
        pp.debug_set_withhold(True)
        out, st = run_gpu_csv(data, ["str", "str"])
        assert st["error"] & pp.ERR_LOOKBACK_TIMEOUT, st
    finally:
        pp.debug_set_withhold(False)
        pp.debug_set_spin_limit(0)
    out, st = run_gpu_csv(data, ["str", "str"])
    assert st["error"] == 0 and st["n_records"] == len(data) // 6, st
    torch.cuda.synchronize()


def test_parse_capacity_too_small():
    data, info, _ = datagen.generate("csv18_2gib", target=2 * TILE)
    cols = datagen.WORKLOADS["csv18_2gib"]["cols"]
    out, st = run_gpu_csv(data, cols, records_capacity=info["n_records"] - 3)
    _, ost = O.csv_parse(data, cols, records_capacity=info["n_records"] - 3)
    assert ost["error"] == O.E_CAPACITY
    assert st["error"] == ost["error"] and st["n_records"] == ost["n_records"]
    out, st = run_gpu_csv(data, cols, chars_capacity=[100] * len(cols))
    _, ost = O.csv_parse(data, cols, chars_capacity=[100] * len(cols))
    assert ost["error"] == O.E_CAPACITY
    assert st["error"] == ost["error"] and st["n_records"] == ost["n_records"]


def test_parse_sizing_pass():
    data, info, _ = datagen.generate("csv4_1mib", target=4 * TILE + 11)
    d_in = to_dev(data)
    st = pp.new_status()
    pp.pp_parse(d_in, data.size, pp.desc_csv(), ["str"] * 4, None, None, None, 0, None, st)
    s = pp.read_status(st, 4)
    _, rst = O.csv_parse(data, ["str"] * 4)
    assert s["error"] == 0 and s["n_records"] == rst["n_records"]
    assert s["chars_len"] == rst["chars_len"]


def test_parse_repeat_calls_identical():
    data, _, _ = datagen.generate("csv3_1gib", target=8 * TILE)
    cols = datagen.WORKLOADS["csv3_1gib"]["cols"]
    a, sa = run_gpu_csv(data, cols)
    b, sb = run_gpu_csv(data, cols)
    assert sa == sb
    for x, y in zip(a.results(sa), b.results(sb)):
        if isinstance(x, tuple):
            assert torch.equal(x[0], y[0]) and torch.equal(x[1], y[1])
        else:
            assert torch.equal(x, y)


def test_count_byte():
    data, _, _ = datagen.generate("csv3_1gib", target=3 * TILE + 5)
    for off in (0, 1):
        d = to_dev(data, off)
        assert pp.count_byte(d, 10) == int(np.count_nonzero(data == 10))


# -------------------------------------------------------------- tokenize
@pytest.mark.parametrize("target", [1, 100, TILE - 3, 6 * TILE + 71, 1 << 20])
def test_tokenize_generated(target):
    data, info, _ = datagen.generate("json_2gib", target=target)
    st = compare_tokens(data)
    assert st["n_tokens"] == info["n_tokens"]


def test_tokenize_misaligned_and_edges():
    data, _, _ = datagen.generate("json_2gib", target=2 * TILE)
    compare_tokens(data, offset=5)
    for s in [b"", b" ", b"1", b"-", b'"abc', b"1.", b"1e", b"[1,2]", b'"\\u00E9"', b"\x7f", b"00"]:
        compare_tokens(s)


def test_tokenize_random_including_invalid():
    rng = random.Random(4)
    for _ in range(200):
        n = rng.randint(0, 300)
        compare_tokens(bytes(rng.choice(b' {"\\-+01.exa]:,E\t') for _ in range(n)))


def test_tokenize_dense_and_long_tokens():
    """Tiles with more tokens than are staged (a token per byte) and tokens
    spanning several tiles (long strings and whitespace runs)."""
    compare_tokens(b"1," * (3 * TILE // 2 + 7))
    compare_tokens(b"[" * (2 * TILE + 5) + b"]" * (2 * TILE + 5))
    long_str = b'"' + (b"ab" + b"\\" + b'"' + b"cd") * (TILE // 3) + b'"'  # escaped quotes
    compare_tokens(b"[" + long_str + b", 12, " + long_str + b"]")
    compare_tokens(b" " * (3 * TILE + 11) + b"1")


def test_tokenize_capacity():
    data, info, _ = datagen.generate("json_2gib", target=3 * TILE)
    d_in = to_dev(data)
    cap = info["n_tokens"] // 2
    ids = torch.empty(cap, dtype=torch.uint8, device="cuda")
    starts = torch.empty(cap, dtype=torch.int64, device="cuda")
    lens = torch.empty(cap, dtype=torch.int32, device="cuda")
    st = pp.new_status()
    pp.pp_tokenize(d_in, data.size, pp.desc_json_lexer(), ids, starts, lens, cap, st)
    s = pp.read_status(st)
    assert s["error"] & pp.ERR_CAPACITY and s["n_tokens"] == info["n_tokens"]
    (rids, rstarts, rlens), _ = O.tokenize(data)
    assert np.array_equal(starts.cpu().numpy().astype(np.uint64), rstarts[:cap])


# ------------------------------------------------------------ timestamps
def test_parse_timestamps_generated():
    """The 2 GiB numeric workload's layout with its timestamp columns typed."""
    cols = datagen.WORKLOADS["csv18ts_2gib"]["cols"]
    for target in (2 << 20, 3 * TILE + 7):
        data, info, _ = datagen.generate("csv18ts_2gib", target=target)
        st = compare_csv(data, cols)
        assert st["error"] == 0 and st["n_records"] == info["n_records"]


def test_parse_timestamp_edge_cases():
    good = [b"1970-01-01 00:00:00", b"1969-12-31 23:59:59", b"2000-02-29", b"0000-01-01",
            b"9999-12-31 23:59:59", b'"2020-07-04 01:02:03"', b'"2021-""01-02"', b""]
    bad = [b"1900-02-29", b"2021-04-31", b"2021-01-01 24:00:00", b"2021-1-01",
           b"2021-01-01T00:00:00", b"2021-01-01 00:00", b"20210101", b'"2021-01-01 "']
    rows = [b"%d,%s\n" % (i, t) for i, t in enumerate(good + bad)]
    compare_csv(b"".join(rows), ["i32", "ts"])
    compare_csv(b"".join(rows[: len(good)]), ["i32", "ts"])


@pytest.mark.parametrize("shift", range(-21, 4, 3))
def test_parse_timestamp_across_tile_boundary(shift):
    """A timestamp field starting at every position around the first tile
    edge, plain and quoted: a field that began in an earlier tile is re-read
    from global memory by the tile that closes it."""
    for ts in (b"2024-02-29 13:14:15", b'"2024-02-29 13:14:15"', b"1999-12-31"):
        first = b"0,0000-01-01\n"
        filler = b"x" * (TILE + shift - len(first) - 1)  # the timestamp starts at TILE + shift
        rest = b"".join(b"%d,%s\n" % (i, ts) for i in range(50))
        data = first + filler + b"," + ts + b"\n" + rest
        assert data.index(ts, len(first)) == TILE + shift
        compare_csv(data, ["str", "ts"])


# ------------------------------------------------------------ CRLF line ends
def _with_crlf(data):
    """A CR before every record delimiter (found by the oracle's tags)."""
    lf = bytes(data)
    _, tags, _ = O.tags(lf)
    out = bytearray()
    for b, t in zip(lf, tags):
        if t == O.TAG_RD:
            out += b"\r"
        out.append(b)
    return bytes(out)


@pytest.mark.parametrize("name,target", [("csv4_1mib", 3 * TILE + 101), ("csv16_256mib", 2 << 20),
                                         ("csv18_2gib", 2 << 20), ("csv3_1gib", 4 << 20)])
def test_parse_crlf_generated(name, target):
    data, info, _ = datagen.generate(name, target=target)
    st = compare_csv(_with_crlf(data), datagen.WORKLOADS[name]["cols"], crlf=True)
    assert st["error"] == 0 and st["n_records"] == info["n_records"]


@pytest.mark.parametrize("k", range(-3, 4))
def test_parse_crlf_at_tile_boundary(k):
    """CR and LF on either side of a tile edge, after plain, quoted and
    numeric fields, and bare CRs inside fields."""
    rows = []
    n = 0
    while n < TILE + 64:
        r = b"%d,ab\rc,\"q\r\nx\"\r\n" % n
        rows.append(r)
        n += len(r)
    data = b"z" * (TILE + k - 3) + b",,\r\n" + b"".join(rows)  # CR at TILE + k - 1, LF after it
    compare_csv(data, ["str", "str", "str"], crlf=True)
    compare_csv(data[: TILE + k + 40], ["i64", "str", "str"], crlf=True)


# ------------------------------------------------- column-count inference
def compare_count_fields(data, crlf=False, offset=0):
    desc = pp.desc_csv_crlf() if crlf else pp.desc_csv()
    got, st = pp.count_fields(to_dev(data, offset), desc)
    ref, rst = O.count_fields(data, crlf=crlf)
    assert st["error"] == rst["error"], (st, rst)
    assert st["first_error_offset"] == rst["first_error_offset"]
    if st["error"] & O.FATAL:
        return st
    assert got == ref and st["n_records"] == rst["n_records"], (got, ref, st, rst)
    return st


@pytest.mark.parametrize("name,target", [("csv4_1mib", None), ("csv16_256mib", 5 * TILE + 3),
                                         ("csv3_1gib", 4 << 20), ("csv18_2gib", 40 << 20)])
def test_count_fields_generated(name, target):
    data, info, _ = datagen.generate(name, target=target)
    n = len(datagen.WORKLOADS[name]["cols"])
    st = compare_count_fields(data)
    assert st["n_records"] == info["n_records"]
    assert pp.count_fields(to_dev(data))[0] == (n, n)


@pytest.mark.parametrize("seed", range(4))
def test_count_fields_varying_rows(seed):
    """Rows of 1..60 fields, some quoted with embedded delimiters, empty
    lines and a few rows longer than a tile, over many tiles."""
    rng = random.Random(seed)
    rows = []
    size = 0
    while size < 6 * TILE:
        if rng.random() < 0.02:
            r = b",".join(b"y" * rng.randint(0, 900) for _ in range(rng.randint(20, 60)))
        elif rng.random() < 0.05:
            r = b""
        else:
            r = b",".join(rng.choice([b"ab", b"", b'"x,\ny"', b'"q""q"', b"123"])
                          for _ in range(rng.randint(1, 12)))
        rows.append(r)
        size += len(r) + 1
    data = b"\n".join(rows) + (b"\n" if seed % 2 else b"")
    compare_count_fields(data)
    compare_count_fields(data, offset=3)


def test_count_fields_edges():
    for data in (b"", b"\n", b"\n\n\n", b"a", b"a,b,c", b",", b"a,b\n" * 10000 + b"c",
                 b"x" * (3 * TILE) + b",y\n", b"," * (2 * TILE + 5) + b"\n" + b"a\n"):
        compare_count_fields(data)
    compare_count_fields(b'a,"b')                        # ends inside quotes
    compare_count_fields(b"a\n" * 9000 + b'x"y\n')         # a quote inside a field
    crlf = b"\r\n".join(b",".join(b"v" for _ in range(k % 7 + 1)) for k in range(5000)) + b"\r\n"
    compare_count_fields(crlf, crlf=True)


@pytest.mark.parametrize("skew", [0, 1, 2])
def test_parse_crowded_and_sparse_fields(skew):
    """Chunks crowded with fields (runs of empty fields, 32 terminators in a
    chunk) next to chunks inside long fields, within and across tiles: each
    lane walks its chunk's terminators, however unevenly they are spread."""
    rng = random.Random(40 + skew)
    parts = []
    for i in range(4000):
        r = rng.random()
        if r < 0.02 * (skew + 1):
            parts.append("," * rng.randint(600, 1500))                          # > 512 fields per warp
        elif r < 0.1 * (skew + 1):
            parts.append(",".join("x" * rng.randint(0, 2) for _ in range(40)))   # a crowd of fields
        else:
            parts.append("y" * rng.randint(100, 400) + "," + str(i))            # few, long fields
    data = ("\n".join(parts) + "\n").encode()
    compare_csv(data, ["str", "str", "str"])


@pytest.mark.parametrize("last", ["short", "long", "one"])
def test_parse_write_out_across_tiles(last):
    """Tiles of one pass of rows leave their offsets and chars to be written
    during the next tile; tiles with more rows than a pass holds (short
    records, several passes) write theirs at once.  Regions of each kind
    alternate, a few tiles long and at ragged offsets, and the input ends
    in either kind of tile, or in a single tile, so that every hand-over
    between the two, and the last tile's write-out at the end of a block's
    tiles, meets the oracle."""
    rng = random.Random({"short": 71, "long": 72, "one": 73}[last])
    parts = []
    kinds = ["short", "long"] * 6 + [last]
    if last == "one":
        kinds = ["long"]
    size = 0
    for kind in kinds:
        target = size + (rng.randint(2000, 15000) if last == "one" else rng.randint(20000, 70000))
        while size < target:
            if kind == "short":  # six bytes a record: 2730 rows a tile, three passes
                rec = "%s,%s,%d\n" % (rng.choice("abc"), rng.choice(["", "d"]), rng.randint(0, 9))
            else:
                rec = "%s,%s,%d\n" % ("x" * rng.randint(100, 900), "y" * rng.randint(0, 40),
                                       rng.randint(-99999, 99999))
            parts.append(rec)
            size += len(rec)
    data = "".join(parts).encode()
    compare_csv(data, ["str", "str", "i64"])
