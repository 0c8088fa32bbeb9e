"""pp_parse_ex (the parse options of ParPaRaw Section 4) against the oracle
on the same bytes, element by element: column defaults for empty and
missing fields, rejecting records whose field count is not the schema's,
skipping records and skipping rows, alone and together, on inputs of many
tiles whose dropped records and skipped rows fall across tile boundaries."""
import random
import struct

import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import to_dev, ulp_diff

pytestmark = pytest.mark.gpu
TILE = 16384


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _bits(x):
    return struct.unpack("<Q", struct.pack("<d", x))[0]


def compare_ex(data, col_types, **opts):
    arr = np.frombuffer(bytes(data), np.uint8) if isinstance(data, (bytes, bytearray)) else data
    n = arr.size
    R = int(np.count_nonzero(arr == 10)) + 1
    out = pp.CsvOutputs(col_types, R, [max(n, 1)] * len(col_types))
    out.run_ex(to_dev(arr), n, pp.desc_csv(), **opts)
    st = pp.read_status(out.status, len(col_types))
    oo = dict(opts)
    if "skip_rows" in oo:
        oo["skip_rows_"] = oo.pop("skip_rows")
    ref, rst = O.csv_parse(arr, col_types, **oo)
    assert st["error"] == rst["error"], (st, rst)
    assert st["first_error_offset"] == rst["first_error_offset"], (st, rst)
    if st["error"] & O.FATAL:
        return st
    assert st["n_records"] == rst["n_records"] and st["n_dropped"] == rst["n_dropped"], (st, rst)
    got = out.results(st)
    for c, t in enumerate(col_types):
        if t == "str":
            assert st["chars_len"][c] == rst["chars_len"][c], c
            assert np.array_equal(got[c][0].cpu().numpy(), ref[c][0]), f"offsets col {c}"
            assert np.array_equal(got[c][1].cpu().numpy(), ref[c][1]), f"chars col {c}"
        elif t == "f64":
            g = got[c].cpu().numpy()
            d = ulp_diff(g, ref[c])
            assert d.size == 0 or int(d.max()) <= 1, f"f64 col {c}"
            assert np.array_equal(np.signbit(g), np.signbit(ref[c]))
        elif t != "skip":
            assert np.array_equal(got[c].cpu().numpy(), ref[c]), f"col {c}"
    return st


def _ragged(rng, n_rows, k, max_extra=1, quoted=True):
    """Rows of k +- max_extra fields (some quoted with delimiters inside)."""
    lines = []
    for _ in range(n_rows):
        nf = max(1, k + rng.randint(-max_extra, max_extra))
        f = []
        for c in range(nf):
            r = rng.random()
            if r < 0.2:
                f.append("")
            elif r < 0.6:
                f.append(str(rng.randint(-500, 500)))
            elif quoted and r < 0.7:
                f.append('"q,' + "x" * rng.randint(0, 40) + '\n""z"')
            else:
                f.append("".join(rng.choice("abcdef") for _ in range(rng.randint(1, 30))))
        lines.append(",".join(f))
    return ("\n".join(lines) + "\n").encode()


def test_defaults_on_ragged_rows():
    rng = random.Random(1)
    data = _ragged(rng, 6000, 4, quoted=False)
    types = ["i64", "str", "i32", "f64"]
    cols_num = [c for c, t in enumerate(types)]
    d = [11, 0, -7 & 0xFFFFFFFFFFFFFFFF, _bits(-2.25)]
    st = compare_ex(data, ["i64", "i32", "i8", "f64"], defaults=d)
    assert st["error"] & pp.ERR_COLCOUNT


def test_defaults_all_empty_and_quoted_empty():
    data = b',,,\n"","",,""\n' * 3000
    compare_ex(data, ["i64", "f64", "ts", "i8"], defaults=[5, _bits(0.5), 86400, 0x80])


@pytest.mark.parametrize("seed", range(3))
def test_reject_ragged_rows_across_tiles(seed):
    rng = random.Random(10 + seed)
    data = _ragged(rng, 8000, 3)
    st = compare_ex(data, ["i64", "str", "str"], reject=True)
    assert st["n_dropped"] > 0


def test_reject_long_records_spanning_tiles():
    """Records longer than a tile: whether one is emitted is known only in
    the tile holding its record delimiter, after tiles that hold its chars."""
    rng = random.Random(4)
    lines = []
    for i in range(40):
        nf = 2 if i % 3 else 3
        lines.append(",".join("".join(rng.choice("ghij") for _ in range(rng.randint(1, 12000)))
                              for _ in range(nf)))
    data = ("\n".join(lines) + "\n").encode()
    st = compare_ex(data, ["str", "str"], reject=True)
    assert st["n_dropped"] == 14


@pytest.mark.parametrize("name,target", [("csv16_256mib", 3 << 20), ("csv3_1gib", 2 << 20),
                                         ("csv18_2gib", 2 << 20)])
def test_skip_records_on_workloads(name, target):
    data, info, _ = datagen.generate(name, target=target)
    rng = random.Random(7)
    R = info["n_records"]
    skip = sorted(rng.sample(range(R), min(R // 10, 3000))) + [0, R - 1]
    st = compare_ex(data, datagen.WORKLOADS[name]["cols"], skip_records=sorted(set(skip)))
    assert st["n_dropped"] == len(set(skip))


def test_skip_records_exempts_column_count_and_numbers():
    data = b"h1,h2,h3\n1,2\n" + b"3,4\n" * 5000 + b"x,y,z\n5,6\n"
    # the header (3 fields) and "x,y,z" (not numbers) are skipped: no error
    st = compare_ex(data, ["i32", "i32"], skip_records=[0, 5002])
    assert st["error"] == 0 and st["n_records"] == 5002
    st = compare_ex(data, ["i32", "i32"], skip_records=[0], reject=True)
    assert st["error"] == pp.ERR_COLCOUNT  # "x,y,z" is rejected, never converted


@pytest.mark.parametrize("seed", range(2))
def test_skip_rows_inside_quoted_records(seed):
    rng = random.Random(20 + seed)
    data = _ragged(rng, 5000, 3, max_extra=0)
    n_lines = data.count(b"\n") + 1
    rows = sorted(rng.sample(range(n_lines), 300))
    compare_ex(data, ["str", "str", "str"], skip_rows=rows)


def test_skip_rows_header_and_tail():
    data, info, _ = datagen.generate("csv18_2gib", target=1 << 20)
    n_lines = int(np.count_nonzero(data == 10))
    compare_ex(data, datagen.WORKLOADS["csv18_2gib"]["cols"],
               skip_rows=[0, 1, 2, n_lines - 1, n_lines + 10])


def test_all_options_together():
    rng = random.Random(33)
    data = _ragged(rng, 7000, 3)
    n_lines = data.count(b"\n") + 1
    compare_ex(data, ["i64", "str", "i32"], defaults=[3, 0, 9], reject=True,
               skip_records=sorted(rng.sample(range(5000), 400)),
               skip_rows=sorted(rng.sample(range(n_lines), 200)))


def test_options_edge_cases():
    compare_ex(b"", ["str"], reject=True, skip_records=[0], skip_rows=[0])
    compare_ex(b"a\nb\n", ["str"], skip_records=[0, 1])           # every record skipped
    compare_ex(b"a,b\nc\n" * 4000, ["str"], reject=True)          # every other record rejected
    compare_ex(b"a,b\nc,d", ["str", "str"], skip_rows=[1])        # the tail line without newline
    compare_ex(b"1,2\n" * 9000, ["i32", "i32"], skip_rows=list(range(0, 9000, 2)))


# ------------------------------------------------------------ type inference
def compare_infer(data, n_cols):
    arr = np.frombuffer(bytes(data), np.uint8) if isinstance(data, (bytes, bytearray)) else data
    got, st = pp.infer_types(to_dev(arr), n_cols, n_bytes=arr.size)
    ref, rst = O.infer_types(arr, n_cols)
    assert (st["error"], st["first_error_offset"]) == (rst["error"], rst["first_error_offset"])
    assert st["n_records"] == rst["n_records"]
    assert got == ref, (got, ref)
    return got


@pytest.mark.parametrize("name,target", [("csv16_256mib", 3 << 20), ("csv18_2gib", 2 << 20),
                                         ("csv3_1gib", 2 << 20), ("csv4_1mib", None)])
def test_infer_types_on_workloads(name, target):
    data, _, _ = datagen.generate(name, target=target)
    k = len(datagen.WORKLOADS[name]["cols"])
    got = compare_infer(data, k + 1)   # and one column that never has a field
    assert got[-1] == "i8"


def test_infer_types_mixed_and_spanning():
    rng = random.Random(61)
    pool = [b"1", b"-7", b"300", b"-40000", b"5000000000", b"2.5", b"1e9", b"", b"ab",
            b'"9"', b"9223372036854775808", b'"1""2"']
    lines = [b",".join(rng.choice(pool) for _ in range(rng.randint(1, 6))) for _ in range(20000)]
    # a long numeric field spanning tiles, and one invalid-for-ints float in column 1 late
    lines.insert(7000, b"1," + b"7" * 40000)
    compare_infer(b"\n".join(lines) + b"\n", 6)
    compare_infer(b"1,2\n" * 9000 + b"1,2.0\n", 2)
    compare_infer(b"", 3)
