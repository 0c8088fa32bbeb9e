"""pp_parse_host (host input and outputs, streamed through the device in
chunks) against pp_parse on the same bytes: status and every output column
equal, for chunk sizes that put chunk boundaries inside quoted fields,
inside quoted newlines and inside records, and for the edge cases of the
carry-over (no trailing newline, empty input, a record longer than the
chunk, errors in later chunks)."""
import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
from gpu_util import to_dev

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
