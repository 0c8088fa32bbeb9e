"""pp_parse_host and pp_tokenize_host (host input and outputs, streamed
through the device in chunks) against the oracle on the same bytes, element
by element (integers, offsets, chars and token triples bit-exact, floats
within 1 ulp with the same sign), and against pp_parse / pp_tokenize: for
chunk sizes that put chunk boundaries inside quoted fields, inside quoted
newlines, between a CR and its LF and inside records, and for the edge cases
of the carry-over (no trailing newline, empty input, a record or token
longer than the chunk, errors in later chunks).  The streamed calls run
kernel modes a single pp_parse never runs (a chunk whose last record stays
open, the carried partial record, offsets rebased on the device), so the
oracle, not the library, is the reference."""
import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import to_dev, ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _device_run(arr, col_types, desc):
    n = arr.size
    R = int(np.count_nonzero(arr == 10)) + 1
    out = pp.CsvOutputs(col_types, R, [max(n, 1)] * len(col_types))
    out.run(to_dev(arr), n, desc)
    return out, pp.read_status(out.status, len(col_types)), R


def _host_run(arr, col_types, desc, R, chunk):
    n = arr.size
    h_in = torch.empty(max(n, 1), dtype=torch.uint8, pin_memory=True)
    if n:
        h_in[:n].copy_(torch.from_numpy(arr))
    out = pp.CsvOutputs(col_types, R, [max(n, 1)] * len(col_types), device="cpu")
    out.run_host(h_in, n, desc, chunk_bytes=chunk)
    return out, pp.read_status(out.status, len(col_types))


def _assert_same(col_types, dev, sdev, host, shost):
    assert shost["error"] == sdev["error"], (shost, sdev)
    assert shost["first_error_offset"] == sdev["first_error_offset"]
    assert shost["n_records"] == sdev["n_records"]
    assert shost["chars_len"] == sdev["chars_len"]
    if sdev["error"]:
        return  # outputs are defined only without errors
    rd, rh = dev.results(sdev), host.results(shost)
    for c, t in enumerate(col_types):
        if t == "str":
            assert torch.equal(rd[c][0].cpu(), rh[c][0]), f"offsets col {c}"
            assert torch.equal(rd[c][1].cpu(), rh[c][1]), f"chars col {c}"
        elif t != "skip":
            assert torch.equal(rd[c].cpu(), rh[c]), f"col {c}"


def _assert_oracle(arr, col_types, host, shost, crlf=False):
    """Streamed outputs equal the oracle's for the same bytes."""
    ref, rst = O.csv_parse(arr, col_types, crlf=crlf)
    assert shost["error"] == rst["error"], (shost, rst)
    assert shost["first_error_offset"] == rst["first_error_offset"], (shost, rst)
    if rst["error"] & O.FATAL:
        return
    assert shost["n_records"] == rst["n_records"]
    got = host.results(shost)
    for c, t in enumerate(col_types):
        if t == "str":
            assert shost["chars_len"][c] == rst["chars_len"][c], c
            assert np.array_equal(got[c][0].numpy(), ref[c][0]), f"offsets col {c}"
            assert np.array_equal(got[c][1].numpy(), ref[c][1]), f"chars col {c}"
        elif t == "f64":
            g = got[c].numpy()
            d = ulp_diff(g, ref[c])
            assert d.size == 0 or int(d.max()) <= 1, f"f64 col {c}: {d.max()} ulp"
            assert np.array_equal(np.signbit(g), np.signbit(ref[c]))
        elif t != "skip":
            assert np.array_equal(got[c].numpy(), ref[c]), f"col {c}"


@pytest.mark.parametrize("name,target,chunk", [
    ("csv4_1mib", None, 16 << 10),       # quoted newlines across many boundaries
    ("csv4_1mib", None, 96 << 10),
    ("csv16_256mib", 6 << 20, 1 << 20),
    ("csv3_1gib", 3 << 20, 64 << 10),    # long quoted texts: chunks start mid-quote
    ("csv18_2gib", 12 << 20, 2 << 20),
    ("csv18_2gib", 3 << 20, 0),          # default chunk: one chunk
])
def test_host_stream_matches_device_parse(name, target, chunk):
    data, info, _ = datagen.generate(name, target=target)
    col_types = datagen.WORKLOADS[name]["cols"]
    desc = pp.desc_csv()
    dev, sdev, R = _device_run(data, col_types, desc)
    assert sdev["error"] == 0 and sdev["n_records"] == info["n_records"]
    host, shost = _host_run(data, col_types, desc, R, chunk)
    _assert_oracle(data, col_types, host, shost)
    _assert_same(col_types, dev, sdev, host, shost)


def test_host_stream_without_trailing_newline_and_empty():
    col_types = ["str", "i32", "f64"]
    desc = pp.desc_csv()
    rng = np.random.default_rng(7)
    lines = [f'"r{i},\n{i}",{int(rng.integers(-9, 9))},{rng.random():.3f}' for i in range(5000)]
    arr = np.frombuffer("\n".join(lines).encode(), np.uint8)  # no final newline
    dev, sdev, R = _device_run(arr, col_types, desc)
    assert sdev["error"] == 0 and sdev["n_records"] == 5000
    host, shost = _host_run(arr, col_types, desc, R, 16 << 10)
    _assert_oracle(arr, col_types, host, shost)
    _assert_same(col_types, dev, sdev, host, shost)
    empty = np.zeros(0, np.uint8)
    host, shost = _host_run(empty, col_types, desc, 1, 16 << 10)
    assert shost["error"] == 0 and shost["n_records"] == 0


def test_host_stream_reports_errors_at_global_offsets():
    col_types = ["str", "i32"]
    desc = pp.desc_csv()
    body = b"".join(b"abc%d,%d\n" % (i, i % 100) for i in range(40000))
    bad = bytearray(body)
    p = len(bad) * 3 // 4
    p = bad.index(b"\n", p) + 1
    bad[p:p + 4] = b'a"b,'        # a quote inside an unquoted field: invalid
    arr = np.frombuffer(bytes(bad), np.uint8)
    dev, sdev, R = _device_run(arr, col_types, desc)
    assert sdev["error"] & pp.ERR_INVALID_INPUT
    host, shost = _host_run(arr, col_types, desc, R, 32 << 10)
    assert shost["error"] & pp.ERR_INVALID_INPUT
    assert shost["first_error_offset"] == sdev["first_error_offset"] == p + 1
    _assert_oracle(arr, col_types, host, shost)


def test_host_stream_rejects_record_longer_than_chunk():
    col_types = ["str", "i32"]
    desc = pp.desc_csv()
    long_field = b"x" * (40 << 10)
    arr = np.frombuffer(b"a,1\n" + long_field + b",2\nb,3\n", np.uint8)
    host = pp.CsvOutputs(col_types, 4, [arr.size] * 2, device="cpu")
    h_in = torch.from_numpy(arr.copy()).pin_memory()
    with pytest.raises(RuntimeError, match=r"pp_parse_host failed: .*\(5\)"):
        host.run_host(h_in, arr.size, desc, chunk_bytes=16 << 10)
    st = pp.read_status(host.status, 2)
    assert st["error"] & pp.ERR_CAPACITY and st["n_records"] == 1


# ---------------------------------------------------------------- tokens
def _device_tokens(arr, desc):
    n = arr.size
    d_in = to_dev(arr)
    st = pp.new_status()
    pp.pp_tokenize(d_in, n, desc, None, None, None, 0, st)
    T = pp.read_status(st)["n_tokens"]
    ids = torch.empty(max(T, 1), dtype=torch.uint8, device="cuda")
    starts = torch.empty(max(T, 1), dtype=torch.int64, device="cuda")
    lens = torch.empty(max(T, 1), dtype=torch.int32, device="cuda")
    pp.pp_tokenize(d_in, n, desc, ids, starts, lens, T, st)
    s = pp.read_status(st)
    return (ids[:T].cpu(), starts[:T].cpu(), lens[:T].cpu()), s


def _assert_tokens_oracle(arr, triples, sh):
    (rids, rstarts, rlens), rst = O.tokenize(arr)
    assert sh["error"] == rst["error"] and sh["n_tokens"] == rst["n_tokens"], (sh, rst)
    hi, hs, hl = triples
    assert np.array_equal(hi.numpy(), rids)
    assert np.array_equal(hs.numpy().astype(np.uint64), rstarts)
    assert np.array_equal(hl.numpy().astype(np.uint32), rlens)


def _host_tokens(arr, desc, cap, chunk):
    h_in = torch.empty(max(arr.size, 1), dtype=torch.uint8, pin_memory=True)
    if arr.size:
        h_in[:arr.size].copy_(torch.from_numpy(arr))
    out = pp.TokenOutputs(cap)
    s = out.run_host(h_in, arr.size, desc, chunk_bytes=chunk)
    return out.results(s), s, out


@pytest.mark.parametrize("target,chunk", [(2 << 20, 16 << 10), (6 << 20, 1 << 20), (1 << 20, 0)])
def test_host_tokens_match_device_tokens(target, chunk):
    data, info, _ = datagen.generate("json_2gib", target=target)
    desc = pp.desc_json_lexer()
    (di, ds_, dl), sd = _device_tokens(data, desc)
    assert sd["error"] == 0 and sd["n_tokens"] == info["n_tokens"]
    (hi, hs, hl), sh, _ = _host_tokens(data, desc, sd["n_tokens"], chunk)
    assert sh["error"] == 0 and sh["n_tokens"] == sd["n_tokens"]
    _assert_tokens_oracle(data, (hi, hs, hl), sh)
    assert torch.equal(hi, di) and torch.equal(hs, ds_) and torch.equal(hl, dl)


def test_host_tokens_dense_long_and_errors():
    desc = pp.desc_json_lexer()
    # one-byte tokens everywhere, then a string token longer than a tile
    dense = b"[" + b",".join(b"1" for _ in range(30000)) + b"]"
    long_str = b'"' + b"ab\\\"cd" * 5000 + b'"'
    arr = np.frombuffer(dense + b" " + long_str + b" " + dense, np.uint8)
    (di, ds_, dl), sd = _device_tokens(arr, desc)
    assert sd["error"] == 0
    (hi, hs, hl), sh, _ = _host_tokens(arr, desc, sd["n_tokens"], 48 << 10)
    assert sh["n_tokens"] == sd["n_tokens"] and sh["error"] == 0
    _assert_tokens_oracle(arr, (hi, hs, hl), sh)
    assert torch.equal(hi, di) and torch.equal(hs, ds_) and torch.equal(hl, dl)
    # a token longer than the chunk
    with pytest.raises(RuntimeError, match=r"pp_tokenize_host failed: .*\(5\)"):
        _host_tokens(arr, desc, sd["n_tokens"], 16 << 10)
    # an invalid byte in a later chunk: same first error offset as on the device
    bad = bytearray(dense * 3)
    p = len(bad) * 2 // 3
    bad[p] = 0x01
    arr = np.frombuffer(bytes(bad), np.uint8)
    _, sd = _device_tokens(arr, desc)
    assert sd["error"] & pp.ERR_INVALID_INPUT
    _, sh, _ = _host_tokens(arr, desc, max(sd["n_tokens"], 1), 16 << 10)
    assert sh["error"] & pp.ERR_INVALID_INPUT
    assert sh["first_error_offset"] == sd["first_error_offset"]
    _, rst = O.tokenize(arr)
    assert (sh["error"], sh["first_error_offset"]) == (rst["error"], rst["first_error_offset"])


def test_host_stream_timestamps_and_crlf():
    """Streamed timestamp columns (8 bytes a value) and CRLF line ends,
    with chunk boundaries between a CR and its LF."""
    data, info, _ = datagen.generate("csv18ts_2gib", target=3 << 20)
    col_types = datagen.WORKLOADS["csv18ts_2gib"]["cols"]
    desc = pp.desc_csv()
    dev, sdev, R = _device_run(data, col_types, desc)
    assert sdev["error"] == 0 and sdev["n_records"] == info["n_records"]
    host, shost = _host_run(data, col_types, desc, R, 256 << 10)
    _assert_oracle(data, col_types, host, shost)
    _assert_same(col_types, dev, sdev, host, shost)
    crlf = np.frombuffer(bytes(data).replace(b"\n", b"\r\n"), dtype=np.uint8)
    cdesc = pp.desc_csv_crlf()
    dev, sdev, R = _device_run(crlf, col_types, cdesc)
    assert sdev["error"] == 0 and sdev["n_records"] == info["n_records"]
    for chunk in (256 << 10, (256 << 10) + 1):
        host, shost = _host_run(crlf, col_types, cdesc, R, chunk)
        _assert_oracle(crlf, col_types, host, shost, crlf=True)
        _assert_same(col_types, dev, sdev, host, shost)
