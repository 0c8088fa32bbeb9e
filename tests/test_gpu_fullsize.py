"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (one pp_parse / pp_tokenize call over the whole input on the
current stream, outputs preallocated from the generator's counts).

Every output element is compared with the oracle:

* the input is cut into pieces of whole records (whole top-level values for
  the token stream) at the record starts the generator wrote down, so each
  piece begins in the DFA's start state, which is where the oracle begins;
* the oracle parses every piece (several pieces at a time on the host's
  cores: the oracle is a C library called through ctypes, which releases
  the interpreter lock), and the GPU's rows (tokens) of that piece must
  equal the oracle's: Arrow offsets rebased to the piece's first row, chars,
  integers and token triples bit-exact, floats within 1 ulp with the same
  sign;
* whole-output properties that hold at any size are checked as well: clean
  status, the record (token) count and the value bytes per string column
  equal to what the generator wrote, offsets that start at 0, never decrease
  and end at the chars length; token starts strictly increasing, each token
  ending where the next starts, the last one at the input's end.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import ulp_diff

pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]

PIECE_BYTES = 48 << 20   # oracle work per piece (whole records)


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _roff_cap(name):
    """Room for every record's start: all workloads average over 64 bytes a
    record except the 1 MiB one, which the constant term covers."""
    return datagen.WORKLOADS[name]["target"] // 64 + (1 << 20)


def _to_device(data):
    n = data.size
    d_in = torch.empty(n + 16, dtype=torch.uint8, device="cuda")[:n]
    d_in.copy_(torch.from_numpy(data))
    return d_in


def _pieces(roff, n):
    """(first unit, end unit, first byte, end byte) of pieces of whole units
    (records or top-level values) of about PIECE_BYTES each."""
    cuts = [0]
    nxt = PIECE_BYTES
    while True:
        k = int(np.searchsorted(roff, nxt))
        if k >= roff.size:
            break
        if k > cuts[-1]:
            cuts.append(k)
        nxt = int(roff[k]) + PIECE_BYTES
    out = []
    for i, u0 in enumerate(cuts):
        u1 = cuts[i + 1] if i + 1 < len(cuts) else roff.size
        b0 = int(roff[u0])
        b1 = int(roff[u1]) if u1 < roff.size else n
        out.append((u0, u1, b0, b1))
    return out


def _workers():
    return max(1, min(16, os.cpu_count() or 1))


@pytest.mark.parametrize("name", ["csv4_1mib", "csv16_256mib", "csv3_1gib", "csv18_2gib",
                                  "csv18ts_2gib"])
def test_parse_full_size(name):
    w = datagen.WORKLOADS[name]
    cols = w["cols"]
    data, info, _ = datagen.generate(name, record_offsets=True,
                                     record_offsets_cap=_roff_cap(name))
    roff = info["record_offsets"]
    R = info["n_records"]
    assert roff.size == R
    n = data.size
    d_in = _to_device(data)
    chars_cap = [info["col_value_bytes"][c] if t == "str" else 0 for c, t in enumerate(cols)]
    out = pp.CsvOutputs(cols, R, chars_cap)
    stream = torch.cuda.current_stream()
    out.run(d_in, n, pp.desc_csv(), stream)
    st = pp.read_status(out.status, len(cols))
    assert st["error"] == 0, st
    assert st["n_records"] == R
    got = out.results(st)
    del d_in

    # whole-output properties
    for c, t in enumerate(cols):
        if t == "str":
            assert st["chars_len"][c] == info["col_value_bytes"][c], c
            off = got[c][0]
            assert int(off[0]) == 0 and int(off[-1]) == st["chars_len"][c]
            assert bool((off[1:] >= off[:-1]).all()), f"offsets col {c} decrease"

    # every record against the oracle, piece by piece
    host = []
    for c, t in enumerate(cols):
        if t == "str":
            host.append((got[c][0].cpu().numpy().astype(np.int64), got[c][1].cpu().numpy()))
        elif t == "skip":
            host.append(None)
        else:
            host.append(got[c].cpu().numpy())
    del got, out
    torch.cuda.empty_cache()

    def check(piece):
        r0, r1, b0, b1 = piece
        ref, rst = O.csv_parse(data[b0:b1], cols)
        assert rst["error"] == 0 and rst["n_records"] == r1 - r0, (piece, rst)
        for c, t in enumerate(cols):
            if t == "str":
                off = host[c][0][r0:r1 + 1]
                ro, rc = ref[c]
                assert np.array_equal(off - off[0], ro), f"offsets col {c} rows {r0}..{r1}"
                assert np.array_equal(host[c][1][off[0]:off[-1]], rc), \
                    f"chars col {c} rows {r0}..{r1}"
            elif t == "f64":
                g = host[c][r0:r1]
                d = ulp_diff(g, ref[c])
                assert d.size == 0 or int(d.max()) <= 1, \
                    f"f64 col {c} rows {r0}..{r1}: {d.max()} ulp"
                assert np.array_equal(np.signbit(g), np.signbit(ref[c]))
            elif t != "skip":
                assert np.array_equal(host[c][r0:r1], ref[c]), f"col {c} rows {r0}..{r1}"
        return r1 - r0

    pieces = _pieces(roff, n)
    with ThreadPoolExecutor(_workers()) as ex:
        checked = sum(ex.map(check, pieces))
    assert checked == R


def test_tokenize_full_size():
    name = "json_2gib"
    data, info, _ = datagen.generate(name, record_offsets=True, record_offsets_cap=_roff_cap(name))
    assert info["n_tokens"] > 0
    roff = info["record_offsets"].astype(np.int64)
    assert roff.size < _roff_cap(name), "every top-level value's start is recorded"
    assert roff[0] == 0
    n = data.size
    T = info["n_tokens"]
    d_in = _to_device(data)
    ids = torch.empty(T, dtype=torch.uint8, device="cuda")
    starts = torch.empty(T, dtype=torch.int64, device="cuda")
    lens = torch.empty(T, dtype=torch.int32, device="cuda")
    status = pp.new_status()
    stream = torch.cuda.current_stream()
    pp.pp_tokenize(d_in, n, pp.desc_json_lexer(), ids, starts, lens, T, status, stream)
    st = pp.read_status(status)
    assert st["error"] == 0, st
    assert st["n_tokens"] == T

    # whole-output properties
    assert int(starts[0]) == 0
    assert bool((starts[1:] > starts[:-1]).all())
    assert bool((starts[:-1] + lens[:-1].to(torch.int64) == starts[1:]).all())
    assert int(starts[-1]) + int(lens[-1]) == n
    assert bool((ids != 255).all())
    assert int(lens.to(torch.int64).sum()) == n
    h_ids = ids.cpu().numpy()
    h_starts = starts.cpu().numpy()
    h_lens = lens.cpu().numpy().astype(np.uint32)
    del d_in, ids, starts, lens
    torch.cuda.empty_cache()

    # every token against the oracle, in pieces of whole top-level values: a
    # value starts with '{' at the input's start or after a whitespace run,
    # so it begins a token in the lexer's start context
    def check(piece):
        _, _, b0, b1 = piece
        (rids, rstarts, rlens), rst = O.tokenize(data[b0:b1])
        assert rst["error"] == 0, (piece, rst)
        t0 = int(np.searchsorted(h_starts, b0))
        m = rids.size
        assert t0 < T and int(h_starts[t0]) == b0, f"no token starts at byte {b0}"
        assert t0 + m <= T
        assert np.array_equal((h_starts[t0:t0 + m] - b0).astype(np.uint64), rstarts), \
            f"starts from byte {b0}"
        assert np.array_equal(h_lens[t0:t0 + m], rlens), f"lengths from byte {b0}"
        assert np.array_equal(h_ids[t0:t0 + m], rids), f"ids from byte {b0}"
        if t0 + m < T:
            assert int(h_starts[t0 + m]) == b1
        else:
            assert b1 == n
        return m

    pieces = _pieces(roff, n)
    with ThreadPoolExecutor(_workers()) as ex:
        checked = sum(ex.map(check, pieces))
    assert checked == T
