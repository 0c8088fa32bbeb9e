"""ORACLE — test infrastructure only.

Python access to the plain sequential CPU parser in ``pp_oracle.c``.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package; the GPU library never calls it and has no fallback
to it.  It shares no code with the CUDA path.

Parity pins live in ``tests/test_oracle_*.py``; every function here is the
plain definition (sequential DFA walk) of ParPaRaw's result, or a direct
restatement of one of the method's steps for those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")

# error bits (values are part of the library ABI, restated here)
E_INVALID_INPUT = 1
E_BAD_END_STATE = 2
E_COLCOUNT = 4
E_NUM_SYNTAX = 8
E_NUM_OVERFLOW = 16
E_CAPACITY = 32
FATAL = E_INVALID_INPUT | E_BAD_END_STATE | E_CAPACITY

TAG_DATA, TAG_FD, TAG_RD, TAG_CTRL, TAG_INVALID, TAG_BEGIN = range(6)
COL_CODES = {"str": 0, "i8": 1, "i32": 2, "i64": 3, "f64": 4, "skip": 5, "ts": 6}
NUMPY_OF = {"i8": np.int8, "i32": np.int32, "i64": np.int64, "f64": np.float64, "ts": np.int64}
KIND_CSV, KIND_LEX, KIND_CSV_CRLF = 0, 1, 2
U64MAX = (1 << 64) - 1


class Status(ctypes.Structure):
    _fields_ = [("error", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("first_error_offset", ctypes.c_uint64), ("n_records", ctypes.c_uint64),
                ("n_tokens", ctypes.c_uint64), ("chars_len", ctypes.c_uint64 * 64),
                ("n_dropped", ctypes.c_uint64)]

    def as_dict(self, n_cols=0):
        return dict(error=int(self.error), first_error_offset=int(self.first_error_offset),
                    n_records=int(self.n_records), n_tokens=int(self.n_tokens),
                    chars_len=[int(self.chars_len[i]) for i in range(n_cols)],
                    n_dropped=int(self.n_dropped))


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "pp_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-o", _SO, src])
    return _SO


_lib = None
_vp = ctypes.c_void_p
_u8, _u64 = ctypes.c_uint8, ctypes.c_uint64


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        L.or_csv_parse.argtypes = [_vp, _u64, _u8, _u8, _u8, ctypes.c_int, ctypes.c_int, _vp,
                                   _vp, _vp, _vp, _u64, _vp, ctypes.POINTER(Status)]
        L.or_csv_parse_ex.argtypes = [_vp, _u64, _u8, _u8, _u8, ctypes.c_int, ctypes.c_int, _vp,
                                      _vp, ctypes.c_int, _vp, _u64, _vp, _vp, _vp, _u64, _vp,
                                      ctypes.POINTER(Status)]
        L.or_csv_parse_enc.argtypes = [_vp, _u64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                                       ctypes.c_uint32, ctypes.c_int, _vp, _vp, ctypes.c_int, _vp,
                                       _u64, _vp, _vp, _vp, _u64, _vp, ctypes.POINTER(Status)]
        L.or_skip_rows.argtypes = [_vp, _u64, _u8, _vp, _u64, _vp]
        L.or_infer_types.argtypes = [_vp, _u64, _u8, _u8, _u8, ctypes.c_int, ctypes.c_int, _vp,
                                     ctypes.POINTER(Status)]
        L.or_skip_rows.restype = _u64
        L.or_count_fields.argtypes = [_vp, _u64, _u8, _u8, _u8, ctypes.c_int, _vp,
                                      ctypes.POINTER(Status)]
        L.or_tokenize.argtypes = [_vp, _u64, _vp, _vp, _vp, _u64, ctypes.POINTER(Status)]
        L.or_tags.argtypes = [ctypes.c_int, _u8, _u8, _u8, _vp, _u64, _vp, _vp]
        L.or_tags.restype = ctypes.c_int
        L.or_stv.argtypes = [ctypes.c_int, _u8, _u8, _u8, _vp, _u64, _vp]
        L.or_compose.argtypes = [ctypes.c_int, _vp, _vp, _vp]
        L.or_chunk_start_states.argtypes = [ctypes.c_int, _u8, _u8, _u8, _vp, _u64, _u64, _vp]
        L.or_bruteforce.argtypes = [ctypes.c_int, _u8, _u8, _u8, _vp, ctypes.c_int,
                                    ctypes.c_int, ctypes.POINTER(_u64)]
        L.or_bruteforce.restype = _u64
        _lib = L
    return _lib


def _arr(x) -> np.ndarray:
    if isinstance(x, (bytes, bytearray)):
        return np.frombuffer(bytes(x), dtype=np.uint8)
    return np.ascontiguousarray(x, dtype=np.uint8)


def skip_rows(data, rows, rd=b"\n"):
    """The input without the listed rows (lines ended by rd; ParPaRaw
    Section 4, "Skipping rows")."""
    L = _load()
    a = _arr(data)
    r = np.ascontiguousarray(sorted(set(int(x) for x in rows)), dtype=np.uint64)
    out = np.zeros(max(a.size, 1), dtype=np.uint8)
    w = L.or_skip_rows(a.ctypes.data, a.size, rd[0], r.ctypes.data if r.size else None, r.size,
                       out.ctypes.data)
    return out[:w]


ENCODINGS = {"utf-8": 1, "utf-16-le": 2}


def _cp(x):
    return x if isinstance(x, int) else ord(x.decode() if isinstance(x, bytes) else x)


def csv_parse(data, col_types, fd=b",", rd=b"\n", quote=b'"', records_capacity=None,
              chars_capacity=None, crlf=False, defaults=None, reject=False,
              skip_records=None, skip_rows_=None, encoding=None):
    """Sequentially parse quoted CSV (crlf: carriage returns outside quotes
    are dropped, so CRLF line ends work with rd = LF).

    With `encoding` ("utf-8" or "utf-16-le", ParPaRaw Section 3.4) the DFA
    reads symbols of that encoding and fd, rd and quote are characters (or
    code points); values keep all bytes of their symbols.

    Options (ParPaRaw Section 4): `defaults` (n_cols integer bit patterns)
    are stored for empty or missing numeric fields instead of 0; with
    `reject`, records whose field count is not len(col_types) are not
    emitted; `skip_records` lists record indices not to emit; `skip_rows_`
    lists rows (lines) removed from the input before parsing.

    Returns (columns, status): columns[c] is (offsets int32[R+1], chars uint8)
    for string columns, a numpy array of R values for numeric ones, None for
    'skip'.  Output arrays are trimmed to the record / chars counts.
    """
    L = _load()
    if skip_rows_ is not None:
        data = skip_rows(data, skip_rows_, rd)
    a = _arr(data)
    n = a.size
    ncols = len(col_types)
    if records_capacity is None:
        records_capacity = (n + 1) if encoding else int(np.count_nonzero(a == rd[0])) + 1
    if chars_capacity is None:
        chars_capacity = [n] * ncols
    offs, chars, typed = [], [], []
    ptr_off = (_vp * max(ncols, 1))()
    ptr_chr = (_vp * max(ncols, 1))()
    ptr_typ = (_vp * max(ncols, 1))()
    for c, t in enumerate(col_types):
        if t == "str":
            o = np.zeros(records_capacity + 1, dtype=np.int32)
            ch = np.zeros(max(chars_capacity[c], 1), dtype=np.uint8)
            offs.append(o); chars.append(ch); typed.append(None)
            ptr_off[c] = o.ctypes.data; ptr_chr[c] = ch.ctypes.data
        elif t == "skip":
            offs.append(None); chars.append(None); typed.append(None)
        else:
            v = np.zeros(max(records_capacity, 1), dtype=NUMPY_OF[t])
            offs.append(None); chars.append(None); typed.append(v)
            ptr_typ[c] = v.ctypes.data
    codes = np.array([COL_CODES[t] for t in col_types] or [0], dtype=np.int32)
    ccap = np.array(list(chars_capacity) or [0], dtype=np.uint64)
    st = Status()
    dflt = None if defaults is None else np.ascontiguousarray(
        [int(x) & 0xFFFFFFFFFFFFFFFF for x in defaults], dtype=np.uint64)
    skr = np.ascontiguousarray(sorted(set(int(x) for x in (skip_records or []))), dtype=np.uint64)
    common = (ncols, codes.ctypes.data, dflt.ctypes.data if dflt is not None else None,
              int(bool(reject)), skr.ctypes.data if skr.size else None, skr.size,
              ctypes.addressof(ptr_off), ctypes.addressof(ptr_chr), ctypes.addressof(ptr_typ),
              records_capacity, ccap.ctypes.data, ctypes.byref(st))
    if encoding:
        assert not crlf and skip_rows_ is None
        L.or_csv_parse_enc(a.ctypes.data, n, ENCODINGS[encoding], _cp(fd), _cp(rd), _cp(quote),
                           *common)
    else:
        L.or_csv_parse_ex(a.ctypes.data, n, fd[0], rd[0], quote[0], int(bool(crlf)), *common)
    R = min(int(st.n_records), records_capacity)
    cols = []
    for c, t in enumerate(col_types):
        if t == "str":
            cols.append((offs[c][: R + 1], chars[c][: int(st.chars_len[c])]))
        elif t == "skip":
            cols.append(None)
        else:
            cols.append(typed[c][:R])
    return cols, st.as_dict(ncols)


INFER_NAMES = {1: "i8", 2: "i32", 3: "i64", 4: "f64", 0: "str"}


def infer_types(data, n_cols, fd=b",", rd=b"\n", quote=b'"', crlf=False):
    """Per column the smallest of int8 < int32 < int64 < float64 < string
    that backs every field (ParPaRaw Section 4, "Type inference"), as the
    library's column names, and the status."""
    L = _load()
    a = _arr(data)
    out = np.zeros(max(n_cols, 1), dtype=np.int32)
    st = Status()
    L.or_infer_types(a.ctypes.data, a.size, fd[0], rd[0], quote[0], int(bool(crlf)), n_cols,
                     out.ctypes.data, ctypes.byref(st))
    return [INFER_NAMES[int(x)] for x in out[:n_cols]], st.as_dict()


def count_fields(data, fd=b",", rd=b"\n", quote=b'"', crlf=False):
    """(min, max) fields per record over the input, and the status."""
    L = _load()
    a = _arr(data)
    out = np.zeros(2, dtype=np.uint64)
    st = Status()
    L.or_count_fields(a.ctypes.data, a.size, fd[0], rd[0], quote[0], int(bool(crlf)),
                      out.ctypes.data, ctypes.byref(st))
    return (int(out[0]), int(out[1])), st.as_dict()


def tokenize(data, capacity=None):
    """Sequentially lex the JSON-like token stream -> (ids, starts, lens), status."""
    L = _load()
    a = _arr(data)
    n = a.size
    cap = n + 1 if capacity is None else capacity
    ids = np.zeros(max(cap, 1), dtype=np.uint8)
    starts = np.zeros(max(cap, 1), dtype=np.uint64)
    lens = np.zeros(max(cap, 1), dtype=np.uint32)
    st = Status()
    L.or_tokenize(a.ctypes.data, n, ids.ctypes.data, starts.ctypes.data, lens.ctypes.data,
                  cap, ctypes.byref(st))
    T = min(int(st.n_tokens), cap)
    return (ids[:T], starts[:T], lens[:T]), st.as_dict()


def tags(data, kind=KIND_CSV, fd=b",", rd=b"\n", quote=b'"'):
    """Per-byte (state before, tag) of the sequential walk; also the end state."""
    L = _load()
    a = _arr(data)
    sb = np.zeros(max(a.size, 1), dtype=np.uint8)
    tg = np.zeros(max(a.size, 1), dtype=np.uint8)
    end = L.or_tags(kind, fd[0], rd[0], quote[0], a.ctypes.data, a.size, sb.ctypes.data,
                    tg.ctypes.data)
    return sb[: a.size], tg[: a.size], int(end)


def nstates(kind):
    return 16 if kind == KIND_LEX else 5


def stv(chunk, kind=KIND_CSV, fd=b",", rd=b"\n", quote=b'"'):
    L = _load()
    a = _arr(chunk)
    out = np.zeros(16, dtype=np.uint8)
    L.or_stv(kind, fd[0], rd[0], quote[0], a.ctypes.data, a.size, out.ctypes.data)
    return out[: nstates(kind)]


def compose(a, b):
    L = _load()
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.zeros(a.size, dtype=np.uint8)
    L.or_compose(a.size, a.ctypes.data, b.ctypes.data, out.ctypes.data)
    return out


def chunk_start_states(data, chunk, kind=KIND_CSV, fd=b",", rd=b"\n", quote=b'"'):
    L = _load()
    a = _arr(data)
    nch = (a.size + chunk - 1) // chunk
    out = np.zeros(max(nch, 1), dtype=np.uint8)
    L.or_chunk_start_states(kind, fd[0], rd[0], quote[0], a.ctypes.data, a.size, chunk,
                            out.ctypes.data)
    return out[:nch]


def bruteforce(kind, alphabet: bytes, max_len: int, fd=b",", rd=b"\n", quote=b'"'):
    """(mismatches, strings checked) of the scan-vs-sequential brute force."""
    L = _load()
    a = _arr(alphabet)
    checked = _u64(0)
    bad = L.or_bruteforce(kind, fd[0], rd[0], quote[0], a.ctypes.data, a.size, max_len,
                          ctypes.byref(checked))
    return int(bad), int(checked.value)


def timed_csv_parse(data, col_types, **kw):
    """csv_parse plus its wall time in seconds (parse only, input in RAM)."""
    t0 = time.perf_counter()
    out = csv_parse(data, col_types, **kw)
    return out, time.perf_counter() - t0


def timed_tokenize(data, **kw):
    t0 = time.perf_counter()
    out = tokenize(data, **kw)
    return out, time.perf_counter() - t0
