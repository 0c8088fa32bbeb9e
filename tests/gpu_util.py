"""Helpers shared by the GPU parity tests: run the library and the oracle on
the same bytes and compare element by element (floats within 1 ulp)."""
import numpy as np
import torch

import dfa_parsing_delimiter_gb300 as pp
import oracle as O


def to_dev(a, offset=0):
    """Copy bytes to the GPU; offset > 0 yields a deliberately misaligned view."""
    a = np.frombuffer(bytearray(a), dtype=np.uint8) if isinstance(a, (bytes, bytearray)) else a
    buf = torch.empty(a.size + offset + 16, dtype=torch.uint8, device="cuda")
    if a.size:
        buf[offset:offset + a.size].copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return buf[offset:offset + a.size]


def ulp_diff(a, b):
    """|a - b| in units in the last place (ordered integer view of binary64)."""
    def ordered(x):
        i = np.ascontiguousarray(x, dtype=np.float64).view(np.int64)
        return np.where(i < 0, np.int64(-0x8000000000000000) - i, i)
    return np.abs(ordered(a) - ordered(b))


def run_gpu_csv(data, col_types, desc=None, records_capacity=None, chars_capacity=None,
                offset=0):
    desc = desc or pp.desc_csv()
    arr = np.frombuffer(bytes(data), np.uint8) if isinstance(data, (bytes, bytearray)) else data
    n = arr.size
    d_in = to_dev(arr, offset)
    if records_capacity is None:
        records_capacity = int(np.count_nonzero(arr == desc_rd(desc))) + 1
    if chars_capacity is None:
        chars_capacity = [n] * len(col_types)
    out = pp.CsvOutputs(col_types, records_capacity, chars_capacity)
    out.run(d_in, n, desc)
    st = pp.read_status(out.status, len(col_types))
    return out, st


def desc_rd(desc):
    for b in range(256):
        if desc.byte_to_group[b] == 2:
            return b
    return 10


def compare_csv(data, col_types, desc=None, offset=0, fd=b",", rd=b"\n", quote=b'"',
                crlf=False, encoding=None):
    """Parse with both; assert identical status and columns.  Returns status.
    With `encoding` ("utf-8", "utf-16-le") fd, rd and quote are characters."""
    if encoding:
        desc = pp.desc_csv_enc(encoding, fd, rd, quote)
        out, st = run_gpu_csv(data, col_types, desc=desc, offset=offset,
                              records_capacity=len(data) + 1)
        ref, rst = O.csv_parse(data, col_types, fd=fd, rd=rd, quote=quote, encoding=encoding)
    else:
        desc = desc or (pp.desc_csv_crlf(fd, quote) if crlf else pp.desc_csv(fd, rd, quote))
        out, st = run_gpu_csv(data, col_types, desc=desc, offset=offset)
        ref, rst = O.csv_parse(data, col_types, fd=fd, rd=rd, quote=quote, crlf=crlf)
    assert st["error"] == rst["error"], (st, rst)
    assert st["first_error_offset"] == rst["first_error_offset"], (st, rst)
    if st["error"] & O.FATAL:
        return st
    assert st["n_records"] == rst["n_records"]
    got = out.results(st)
    for c, t in enumerate(col_types):
        if t == "str":
            go, gc = got[c]
            ro, rc = ref[c]
            assert st["chars_len"][c] == rst["chars_len"][c], c
            assert np.array_equal(go.cpu().numpy(), ro), f"offsets col {c}"
            assert np.array_equal(gc.cpu().numpy(), rc), f"chars col {c}"
        elif t == "f64":
            g = got[c].cpu().numpy()
            assert g.shape == ref[c].shape
            d = ulp_diff(g, ref[c])
            assert d.size == 0 or int(d.max()) <= 1, f"f64 col {c}: max ulp {d.max()}"
            assert np.array_equal(np.signbit(g), np.signbit(ref[c]))
        elif t != "skip":
            assert np.array_equal(got[c].cpu().numpy(), ref[c]), f"col {c}"
    return st


def compare_tags(data, kind=O.KIND_CSV, offset=0):
    desc = pp.desc_csv() if kind == O.KIND_CSV else pp.desc_json_lexer()
    d_in = to_dev(data, offset)
    sb, tg, st = pp.tags(d_in, desc)
    rsb, rtg, end = O.tags(data, kind=kind)
    assert np.array_equal(sb.cpu().numpy(), rsb)
    assert np.array_equal(tg.cpu().numpy(), rtg)
    return st


def compare_tokens(data, offset=0):
    d_in = to_dev(data, offset)
    (ids, starts, lens), st = pp.tokenize(d_in)
    (rids, rstarts, rlens), rst = O.tokenize(data)
    assert st["error"] == rst["error"], (st, rst)
    assert st["first_error_offset"] == rst["first_error_offset"]
    assert st["n_tokens"] == rst["n_tokens"]
    if st["error"] & O.FATAL:
        return st
    assert np.array_equal(starts.cpu().numpy().astype(np.uint64), rstarts)
    assert np.array_equal(lens.cpu().numpy().astype(np.uint32), rlens)
    assert np.array_equal(ids.cpu().numpy(), rids)
    return st
