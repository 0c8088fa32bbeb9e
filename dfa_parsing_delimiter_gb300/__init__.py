"""Python binding of libpp (GB300 DFA-based parsing of delimiter-separated
raw data, after ParPaRaw).

Argument marshalling only: every step of the parse runs in libpp's CUDA
kernels.  PyTorch provides device memory and streams.  There is no CPU
fallback: if ``libpp.so`` is missing, loading fails with an error.

Names follow the C ABI in ``include/pp.h``:

  pp_parse / parse_csv          delimiter-separated input -> columns
  pp_parse_noalloc              pp_parse with a fixed, compiled-in scratch buffer
  pp_tokenize / tokenize        general DFA lexer -> (token_id, start, len)
  pp_tags / tags                per-byte state and tag (test hook)
  pp_count_byte / count_byte    byte count (record-capacity bound)
  desc_csv, desc_json_lexer     DFA descriptors
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpp.so")

PP_OK, PP_EINVAL, PP_ECUDA, PP_ENOMEM, PP_ETOOLARGE, PP_ECHUNK = 0, 1, 2, 3, 4, 5
COL = {"str": 0, "i8": 1, "i32": 2, "i64": 3, "f64": 4, "skip": 5, "ts": 6}
DTYPE = {"i8": torch.int8, "i32": torch.int32, "i64": torch.int64, "f64": torch.float64,
         "ts": torch.int64}
ERR_INVALID_INPUT, ERR_BAD_END_STATE, ERR_COLCOUNT = 1, 2, 4
ERR_NUM_SYNTAX, ERR_NUM_OVERFLOW, ERR_CAPACITY, ERR_LOOKBACK_TIMEOUT = 8, 16, 32, 64
ERR_FATAL = ERR_INVALID_INPUT | ERR_BAD_END_STATE | ERR_CAPACITY | ERR_LOOKBACK_TIMEOUT
TAG_DATA, TAG_FD, TAG_RD, TAG_CTRL, TAG_INVALID, TAG_BEGIN = range(6)
MAX_COLS = 64

_u8, _u16, _u32, _u64 = ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint32, ctypes.c_uint64
_vp, _sz = ctypes.c_void_p, ctypes.c_size_t


class DfaDesc(ctypes.Structure):
    """pp_dfa_desc (host memory)."""
    _fields_ = [("n_states", _u8), ("n_groups", _u8), ("start_state", _u8),
                ("invalid_state", _u8), ("accept_mask", _u16), ("background_group", _u8),
                ("encoding", _u8), ("byte_to_group", _u8 * 256), ("delta", (_u8 * 16) * 16),
                ("tag", (_u8 * 16) * 16), ("token_id", _u8 * 16), ("byte_token_id", _u8 * 256),
                ("n_syms", _u8), ("sym_group", _u8 * 8), ("reserved2", _u8 * 3),
                ("sym_cp", ctypes.c_uint32 * 8)]


class Status(ctypes.Structure):
    """pp_status (lives in device memory; this is its host image)."""
    _fields_ = [("error", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("first_error_offset", _u64), ("n_records", _u64), ("n_tokens", _u64),
                ("chars_len", _u64 * MAX_COLS), ("n_dropped", _u64)]


class ParseOpts(ctypes.Structure):
    """pp_parse_opts (host memory)."""
    _fields_ = [("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("col_default", ctypes.c_void_p), ("skip_records", ctypes.c_void_p),
                ("n_skip_records", _u64), ("skip_rows", ctypes.c_void_p), ("n_skip_rows", _u64)]


PARSE_REJECT = 1


STATUS_BYTES = ctypes.sizeof(Status)
_lib = None


def lib() -> ctypes.CDLL:
    """Load libpp.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpp.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.pp_parse.restype = ctypes.c_int
        L.pp_parse.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), ctypes.c_int, _vp, _vp, _vp, _vp,
                               _sz, _vp, _vp, _vp]
        L.pp_parse_noalloc.restype = ctypes.c_int
        L.pp_parse_noalloc.argtypes = L.pp_parse.argtypes
        L.pp_infer_types.restype = ctypes.c_int
        L.pp_infer_types.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), ctypes.c_int, _vp, _vp,
                                     _vp]
        L.pp_parse_ex.restype = ctypes.c_int
        L.pp_parse_ex.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), ctypes.c_int, _vp,
                                  ctypes.POINTER(ParseOpts), _vp, _vp, _vp, _sz, _vp, _vp, _vp]
        L.pp_parse_host.restype = ctypes.c_int
        L.pp_parse_host.argtypes = L.pp_parse.argtypes[:-1] + [_sz, _vp]
        L.pp_tokenize_host.restype = ctypes.c_int
        L.pp_tokenize_host.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), _vp, _vp, _vp, _sz, _vp,
                                       _sz, _vp]
        L.pp_tokenize.restype = ctypes.c_int
        L.pp_tokenize.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), _vp, _vp, _vp, _sz, _vp, _vp]
        L.pp_tags.restype = ctypes.c_int
        L.pp_tags.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), _vp, _vp, _vp, _vp]
        L.pp_count_byte.restype = ctypes.c_int
        L.pp_count_byte.argtypes = [_vp, _sz, _u8, _vp, _vp]
        L.pp_desc_csv_enc.restype = ctypes.c_int
        L.pp_desc_csv_enc.argtypes = [ctypes.POINTER(DfaDesc), ctypes.c_int, ctypes.c_uint32,
                                      ctypes.c_uint32, ctypes.c_uint32]
        L.pp_desc_csv.restype = ctypes.c_int
        L.pp_desc_csv.argtypes = [ctypes.POINTER(DfaDesc), _u8, _u8, _u8]
        L.pp_count_fields.restype = ctypes.c_int
        L.pp_count_fields.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), _vp, _vp, _vp]
        L.pp_desc_csv_crlf.restype = ctypes.c_int
        L.pp_desc_csv_crlf.argtypes = [ctypes.POINTER(DfaDesc), _u8, _u8]
        L.pp_desc_json_lexer.restype = ctypes.c_int
        L.pp_desc_json_lexer.argtypes = [ctypes.POINTER(DfaDesc)]
        L.pp_strerror.restype = ctypes.c_char_p
        L.pp_strerror.argtypes = [ctypes.c_int]
        L.pp_tile_bytes.restype = _sz
        L.pp_tile_bytes.argtypes = []
        L.pp_debug_set_spin_limit.restype = None
        L.pp_debug_set_spin_limit.argtypes = [_u32]
        L.pp_debug_set_withhold.restype = None
        L.pp_debug_set_withhold.argtypes = [ctypes.c_int]
        L.pp_debug_stage_timing.restype = ctypes.c_int
        L.pp_debug_stage_timing.argtypes = [ctypes.c_int]
        L.pp_debug_stage_ms.restype = ctypes.c_int
        L.pp_debug_stage_ms.argtypes = [_vp, ctypes.c_int]
        L.pp_debug_parse_tags.restype = ctypes.c_int
        L.pp_debug_parse_tags.argtypes = [_vp, _sz, ctypes.POINTER(DfaDesc), _vp, _vp, _vp]
        L.pp_debug_long_fields.restype = ctypes.c_int
        L.pp_debug_long_fields.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int]
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != PP_OK:
        raise RuntimeError(f"{what} failed: {lib().pp_strerror(rc).decode()} ({rc})")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def desc_csv(fd: bytes = b",", rd: bytes = b"\n", quote: bytes = b'"') -> DfaDesc:
    d = DfaDesc()
    _check(lib().pp_desc_csv(ctypes.byref(d), fd[0], rd[0], quote[0]), "pp_desc_csv")
    return d


ENC_UTF8, ENC_UTF16LE = 1, 2
ENCODINGS = {"utf-8": ENC_UTF8, "utf-16-le": ENC_UTF16LE}


def desc_csv_enc(encoding: str, fd: str = ",", rd: str = "\n", quote: str = '"') -> DfaDesc:
    """The quoted-CSV DFA over the symbols of an encoding ("utf-8" or
    "utf-16-le"); fd, rd and quote are characters (or code points)."""
    def cp(x):
        return x if isinstance(x, int) else ord(x)
    d = DfaDesc()
    _check(lib().pp_desc_csv_enc(ctypes.byref(d), ENCODINGS[encoding], cp(fd), cp(rd), cp(quote)),
           "pp_desc_csv_enc")
    return d


def desc_csv_crlf(fd: bytes = b",", quote: bytes = b'"') -> DfaDesc:
    """The quoted-CSV DFA for CRLF line ends (CR outside quotes dropped)."""
    d = DfaDesc()
    _check(lib().pp_desc_csv_crlf(ctypes.byref(d), fd[0], quote[0]), "pp_desc_csv_crlf")
    return d


def desc_json_lexer() -> DfaDesc:
    d = DfaDesc()
    _check(lib().pp_desc_json_lexer(ctypes.byref(d)), "pp_desc_json_lexer")
    return d


def tile_bytes() -> int:
    return int(lib().pp_tile_bytes())


def debug_set_spin_limit(polls: int) -> None:
    lib().pp_debug_set_spin_limit(int(polls))


def debug_set_withhold(on: bool) -> None:
    """Test hook: the first cross-tile scan block posts nothing, so later
    blocks time out (bounded) and report ERR_LOOKBACK_TIMEOUT."""
    lib().pp_debug_set_withhold(1 if on else 0)


STAGES = 6  # PP_STAGES


def debug_stage_timing(n_calls: int) -> None:
    """Record per-kernel CUDA events for the next n_calls pp_parse or
    pp_tokenize calls (0: stop).  Benchmark hook."""
    _check(lib().pp_debug_stage_timing(int(n_calls)), "pp_debug_stage_timing")


def debug_stage_ms(max_calls: int):
    """Per-call kernel durations (ms) recorded since debug_stage_timing, one
    row of STAGES per call: pp_parse (init, tile vectors, tile states, tile pass, long fields),
    pp_tokenize (init, stv, state scan, count, count scan, emit)."""
    import numpy as np
    out = np.zeros((max(int(max_calls), 1), STAGES), dtype=np.float32)
    n = lib().pp_debug_stage_ms(out.ctypes.data, int(max_calls))
    if n < 0:
        raise RuntimeError("pp_debug_stage_ms failed")
    return out[:n]


def debug_parse_tags(d_in: torch.Tensor, desc: DfaDesc, n_bytes: int = None, stream=None):
    """The tile pass's tag bitmaps (pp_debug_parse_tags) as three boolean
    numpy arrays over the input bytes: field delimiter, record delimiter,
    control symbol; and the status."""
    import numpy as np
    n = int(d_in.numel()) if n_bytes is None else int(n_bytes)
    words = torch.zeros(max(3 * ((n + 31) // 32), 3), dtype=torch.int32, device=d_in.device)
    st = new_status(d_in.device)
    _check(lib().pp_debug_parse_tags(_ptr(d_in), n, ctypes.byref(desc), _ptr(words), _ptr(st),
                                     _stream(stream)), "pp_debug_parse_tags")
    w = words.cpu().numpy().view(np.uint32).reshape(-1, 3)
    bits = [np.unpackbits(w[:, k].copy().view(np.uint8), bitorder="little")[:n].astype(bool)
            for k in range(3)]
    return bits[0], bits[1], bits[2], read_status(st)


def debug_long_fields(reset: bool = False) -> int:
    """Numeric fields converted by the long-field pass (a warp per field)
    on the current device since the last reset; reset=True zeroes it."""
    v = ctypes.c_uint64(0)
    _check(lib().pp_debug_long_fields(ctypes.byref(v), int(reset)), "pp_debug_long_fields")
    return int(v.value)


def new_status(device=None) -> torch.Tensor:
    return torch.empty(STATUS_BYTES, dtype=torch.uint8, device=device or "cuda")


def read_status(st: torch.Tensor, n_cols: int = 0) -> dict:
    """Copy a device pp_status to the host (synchronises)."""
    raw = bytes(st.cpu().numpy().tobytes())
    s = Status.from_buffer_copy(raw)
    return dict(error=int(s.error), first_error_offset=int(s.first_error_offset),
                n_records=int(s.n_records), n_tokens=int(s.n_tokens),
                chars_len=[int(s.chars_len[i]) for i in range(n_cols)],
                n_dropped=int(s.n_dropped))


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


# ------------------------------------------------------------------ raw calls
def pp_parse(d_in: torch.Tensor, n_bytes: int, desc: DfaDesc, col_types, out_offsets,
             out_chars, out_typed, records_capacity: int, chars_capacity, status: torch.Tensor,
             stream=None) -> None:
    """Direct pp_parse call: all tensors preallocated by the caller (device)."""
    n = len(col_types)
    ct = (ctypes.c_int * n)(*[COL[c] if isinstance(c, str) else int(c) for c in col_types])
    po = (_vp * n)(*[_ptr(x) for x in out_offsets]) if out_offsets is not None else None
    pc = (_vp * n)(*[_ptr(x) for x in out_chars]) if out_chars is not None else None
    pt = (_vp * n)(*[_ptr(x) for x in out_typed]) if out_typed is not None else None
    cc = (_sz * n)(*[int(x) for x in chars_capacity]) if chars_capacity is not None else None
    rc = lib().pp_parse(_ptr(d_in), int(n_bytes), ctypes.byref(desc), n, ctypes.addressof(ct),
                        ctypes.addressof(po) if po is not None else None,
                        ctypes.addressof(pc) if pc is not None else None,
                        ctypes.addressof(pt) if pt is not None else None,
                        int(records_capacity), ctypes.addressof(cc) if cc is not None else None,
                        _ptr(status), _stream(stream))
    _check(rc, "pp_parse")


def parse_opts(defaults=None, reject=False, skip_records=None, skip_rows=None):
    """A ParseOpts plus the host arrays it points to (keep both alive for
    the call)."""
    keep = []
    o = ParseOpts()
    o.flags = PARSE_REJECT if reject else 0
    if defaults is not None:
        a = np.ascontiguousarray([int(x) & 0xFFFFFFFFFFFFFFFF for x in defaults], dtype=np.uint64)
        keep.append(a)
        o.col_default = a.ctypes.data
    for name, lst in (("skip_records", skip_records), ("skip_rows", skip_rows)):
        if lst is not None and len(lst):
            a = np.ascontiguousarray(sorted(int(x) for x in lst), dtype=np.uint64)
            keep.append(a)
            setattr(o, name, a.ctypes.data)
            setattr(o, "n_" + name, a.size)
    return o, keep


def pp_parse_ex(d_in: torch.Tensor, n_bytes: int, desc: DfaDesc, col_types, opts, out_offsets,
                out_chars, out_typed, records_capacity: int, chars_capacity, status: torch.Tensor,
                stream=None) -> None:
    """Direct pp_parse_ex call (opts: a ParseOpts, or None)."""
    n = len(col_types)
    ct = (ctypes.c_int * n)(*[COL[c] if isinstance(c, str) else int(c) for c in col_types])
    arrs = [None if a is None else (_vp * n)(*[_ptr(x) for x in a])
            for a in (out_offsets, out_chars, out_typed)]
    cc = (_sz * n)(*[int(x) for x in chars_capacity]) if chars_capacity is not None else None
    rc = lib().pp_parse_ex(
        _ptr(d_in), int(n_bytes), ctypes.byref(desc), n, ctypes.addressof(ct),
        ctypes.byref(opts) if opts is not None else None,
        *[ctypes.addressof(a) if a is not None else None for a in arrs],
        int(records_capacity), ctypes.addressof(cc) if cc is not None else None,
        _ptr(status), _stream(stream))
    _check(rc, "pp_parse_ex")


TYPE_NAMES = {v: k for k, v in COL.items()}


def infer_types(d_in: torch.Tensor, n_cols: int, desc: DfaDesc = None, n_bytes: int = None,
                stream=None):
    """pp_infer_types: per column the smallest type backing every field, as
    column names ('i8', 'i32', 'i64', 'f64', 'str'), and the status."""
    desc = desc or desc_csv()
    n = d_in.numel() if n_bytes is None else n_bytes
    types = torch.empty(max(n_cols, 1), dtype=torch.int32, device=d_in.device)
    st = new_status(d_in.device)
    _check(lib().pp_infer_types(_ptr(d_in), int(n), ctypes.byref(desc), int(n_cols),
                                _ptr(types), _ptr(st), _stream(stream)), "pp_infer_types")
    return [TYPE_NAMES[int(x)] for x in types[:n_cols].cpu()], read_status(st)


def pp_parse_noalloc(d_in: torch.Tensor, n_bytes: int, desc: DfaDesc, col_types, out_offsets,
                     out_chars, out_typed, records_capacity: int, chars_capacity,
                     status: torch.Tensor, stream=None) -> None:
    """Direct pp_parse_noalloc call: pp_parse's arguments; the library
    allocates nothing; calls must not overlap on one device."""
    n = len(col_types)
    ct = (ctypes.c_int * n)(*[COL[c] if isinstance(c, str) else int(c) for c in col_types])
    arrs = [None if a is None else (_vp * n)(*[_ptr(x) for x in a])
            for a in (out_offsets, out_chars, out_typed)]
    cc = (_sz * n)(*[int(x) for x in chars_capacity]) if chars_capacity is not None else None
    rc = lib().pp_parse_noalloc(
        _ptr(d_in), int(n_bytes), ctypes.byref(desc), n, ctypes.addressof(ct),
        *[ctypes.addressof(a) if a is not None else None for a in arrs],
        int(records_capacity), ctypes.addressof(cc) if cc is not None else None,
        _ptr(status), _stream(stream))
    _check(rc, "pp_parse_noalloc")


def pp_tokenize(d_in, n_bytes, desc, out_id, out_start, out_len, capacity, status,
                stream=None) -> None:
    rc = lib().pp_tokenize(_ptr(d_in), int(n_bytes), ctypes.byref(desc), _ptr(out_id),
                           _ptr(out_start), _ptr(out_len), int(capacity), _ptr(status),
                           _stream(stream))
    _check(rc, "pp_tokenize")


def pp_tags(d_in, n_bytes, desc, d_state_before, d_tag, status, stream=None) -> None:
    rc = lib().pp_tags(_ptr(d_in), int(n_bytes), ctypes.byref(desc), _ptr(d_state_before),
                       _ptr(d_tag), _ptr(status), _stream(stream))
    _check(rc, "pp_tags")


def pp_count_byte(d_in, n_bytes, value: int, d_count, stream=None) -> None:
    rc = lib().pp_count_byte(_ptr(d_in), int(n_bytes), int(value), _ptr(d_count), _stream(stream))
    _check(rc, "pp_count_byte")


# ------------------------------------------------------------- convenience
def pp_parse_host(h_in: torch.Tensor, n_bytes: int, desc: DfaDesc, col_types, h_offsets,
                  h_chars, h_typed, records_capacity: int, chars_capacity, h_status: torch.Tensor,
                  chunk_bytes: int = 0, stream=None) -> None:
    """Direct pp_parse_host call: input, outputs and status in host memory
    (pinned for overlapped copies); returns when the results are there."""
    n = len(col_types)
    ct = (ctypes.c_int * n)(*[COL[c] if isinstance(c, str) else int(c) for c in col_types])
    po = (_vp * n)(*[_ptr(x) for x in h_offsets])
    pc = (_vp * n)(*[_ptr(x) for x in h_chars])
    pt = (_vp * n)(*[_ptr(x) for x in h_typed])
    cc = (_sz * n)(*[int(x) for x in chars_capacity])
    rc = lib().pp_parse_host(_ptr(h_in), int(n_bytes), ctypes.byref(desc), n, ctypes.addressof(ct),
                             ctypes.addressof(po), ctypes.addressof(pc), ctypes.addressof(pt),
                             int(records_capacity), ctypes.addressof(cc), _ptr(h_status),
                             int(chunk_bytes), _stream(stream))
    _check(rc, "pp_parse_host")


def pp_tokenize_host(h_in: torch.Tensor, n_bytes: int, desc: DfaDesc, h_ids, h_starts, h_lens,
                     capacity: int, h_status: torch.Tensor, chunk_bytes: int = 0,
                     stream=None) -> None:
    """Direct pp_tokenize_host call: input, triples and status in host memory
    (pinned for overlapped copies); returns when the results are there."""
    rc = lib().pp_tokenize_host(_ptr(h_in), int(n_bytes), ctypes.byref(desc), _ptr(h_ids),
                                _ptr(h_starts), _ptr(h_lens), int(capacity), _ptr(h_status),
                                int(chunk_bytes), _stream(stream))
    _check(rc, "pp_tokenize_host")


class TokenOutputs:
    """Preallocated pinned host triples (ids u8, starts i64, lens i32) for
    pp_tokenize_host."""

    def __init__(self, capacity: int):
        self.capacity = int(capacity)
        n = max(self.capacity, 1)
        self.ids = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        self.starts = torch.empty(n, dtype=torch.int64, pin_memory=True)
        self.lens = torch.empty(n, dtype=torch.int32, pin_memory=True)
        self.status = torch.empty(STATUS_BYTES, dtype=torch.uint8, pin_memory=True)

    def run_host(self, h_in: torch.Tensor, n_bytes: int, desc: DfaDesc, chunk_bytes: int = 0,
                 stream=None) -> dict:
        pp_tokenize_host(h_in, n_bytes, desc, self.ids, self.starts, self.lens, self.capacity,
                         self.status, chunk_bytes, stream)
        return read_status(self.status)

    def results(self, status: dict):
        T = min(status["n_tokens"], self.capacity)
        return self.ids[:T], self.starts[:T], self.lens[:T]


class CsvOutputs:
    """Preallocated pp_parse outputs for one input size / schema: device
    tensors, or pinned host tensors with device="cpu" (for pp_parse_host)."""

    def __init__(self, col_types, records_capacity: int, chars_capacity, device="cuda"):
        self.col_types = list(col_types)
        self.records_capacity = int(records_capacity)
        self.chars_capacity = [int(chars_capacity[i]) if t == "str" else 0
                               for i, t in enumerate(self.col_types)]
        self.offsets, self.chars, self.typed = [], [], []
        host = torch.device(device).type == "cpu"
        kw = dict(device=device, pin_memory=True) if host else dict(device=device)
        for i, t in enumerate(self.col_types):
            if t == "str":
                self.offsets.append(torch.empty(self.records_capacity + 1, dtype=torch.int32, **kw))
                self.chars.append(torch.empty(max(self.chars_capacity[i], 1), dtype=torch.uint8, **kw))
                self.typed.append(None)
            elif t == "skip":
                self.offsets.append(None); self.chars.append(None); self.typed.append(None)
            else:
                self.offsets.append(None); self.chars.append(None)
                self.typed.append(torch.empty(max(self.records_capacity, 1), dtype=DTYPE[t], **kw))
        self.status = (torch.empty(STATUS_BYTES, dtype=torch.uint8, pin_memory=True) if host
                       else new_status(device))

    def run(self, d_in: torch.Tensor, n_bytes: int, desc: DfaDesc, stream=None) -> None:
        pp_parse(d_in, n_bytes, desc, self.col_types, self.offsets, self.chars, self.typed,
                 self.records_capacity, self.chars_capacity, self.status, stream)

    def run_ex(self, d_in: torch.Tensor, n_bytes: int, desc: DfaDesc, stream=None,
               **options) -> None:
        """pp_parse_ex with options (defaults, reject, skip_records, skip_rows)."""
        opts, keep = parse_opts(**options)
        pp_parse_ex(d_in, n_bytes, desc, self.col_types, opts, self.offsets, self.chars,
                    self.typed, self.records_capacity, self.chars_capacity, self.status, stream)
        del keep

    def run_noalloc(self, d_in: torch.Tensor, n_bytes: int, desc: DfaDesc, stream=None) -> None:
        pp_parse_noalloc(d_in, n_bytes, desc, self.col_types, self.offsets, self.chars,
                         self.typed, self.records_capacity, self.chars_capacity, self.status,
                         stream)

    def run_host(self, h_in: torch.Tensor, n_bytes: int, desc: DfaDesc, chunk_bytes: int = 0,
                 stream=None) -> None:
        """pp_parse_host of a host input into these (host) outputs."""
        pp_parse_host(h_in, n_bytes, desc, self.col_types, self.offsets, self.chars, self.typed,
                      self.records_capacity, self.chars_capacity, self.status, chunk_bytes, stream)

    def output_bytes(self, n_records: int, chars_len) -> int:
        """Bytes the parse writes: offsets, chars and typed values."""
        b = 0
        for i, t in enumerate(self.col_types):
            if t == "str":
                b += 4 * (n_records + 1) + chars_len[i]
            elif t != "skip":
                b += DTYPE[t].itemsize * n_records
        return b

    def results(self, status: dict):
        """Trimmed views of the outputs (device tensors)."""
        R = min(status["n_records"], self.records_capacity)
        cols = []
        for i, t in enumerate(self.col_types):
            if t == "str":
                cols.append((self.offsets[i][: R + 1], self.chars[i][: status["chars_len"][i]]))
            elif t == "skip":
                cols.append(None)
            else:
                cols.append(self.typed[i][:R])
        return cols


def count_fields(d_in: torch.Tensor, desc: DfaDesc | None = None, stream=None):
    """Fewest and most fields per record of a device uint8 tensor ->
    ((min, max), status).  Synchronises to read the result."""
    desc = desc or desc_csv()
    out = torch.zeros(2, dtype=torch.int64, device=d_in.device)
    st = new_status(d_in.device)
    _check(lib().pp_count_fields(_ptr(d_in), d_in.numel(), ctypes.byref(desc), _ptr(out),
                                 _ptr(st), _stream(stream)), "pp_count_fields")
    mm = out.cpu().tolist()
    return (int(mm[0]), int(mm[1])), read_status(st)


def count_byte(d_in: torch.Tensor, value: int, stream=None) -> int:
    c = torch.zeros(1, dtype=torch.int64, device=d_in.device)
    pp_count_byte(d_in, d_in.numel(), value, c, stream)
    return int(c.item())


def parse_csv(d_in: torch.Tensor, col_types, desc: DfaDesc | None = None, rd: bytes = b"\n",
              stream=None):
    """Parse a device uint8 tensor; returns (columns, status dict).

    Output sizes: records <= (#record-delimiter bytes) + 1 (counted on the
    device by pp_count_byte), chars per string column <= input size.
    """
    desc = desc or desc_csv(rd=rd)
    n = d_in.numel()
    R = count_byte(d_in, rd[0], stream) + 1
    out = CsvOutputs(col_types, R, [n] * len(col_types), device=d_in.device)
    out.run(d_in, n, desc, stream)
    st = read_status(out.status, len(col_types))
    return out.results(st), st


def tokenize(d_in: torch.Tensor, desc: DfaDesc | None = None, capacity: int | None = None,
             stream=None):
    """Lex a device uint8 tensor -> ((ids u8, starts i64, lens i32), status).

    Without a capacity a counting pass sizes the outputs exactly.
    """
    desc = desc or desc_json_lexer()
    n = d_in.numel()
    st = new_status(d_in.device)
    if capacity is None:
        pp_tokenize(d_in, n, desc, None, None, None, 0, st, stream)
        capacity = read_status(st)["n_tokens"]
    ids = torch.empty(max(capacity, 1), dtype=torch.uint8, device=d_in.device)
    starts = torch.empty(max(capacity, 1), dtype=torch.int64, device=d_in.device)
    lens = torch.empty(max(capacity, 1), dtype=torch.int32, device=d_in.device)
    pp_tokenize(d_in, n, desc, ids, starts, lens, capacity, st, stream)
    s = read_status(st)
    T = min(s["n_tokens"], capacity)
    return (ids[:T], starts[:T], lens[:T]), s


def tags(d_in: torch.Tensor, desc: DfaDesc, stream=None):
    """Per-byte (state before, tag) and status."""
    n = d_in.numel()
    sb = torch.empty(max(n, 1), dtype=torch.uint8, device=d_in.device)
    tg = torch.empty(max(n, 1), dtype=torch.uint8, device=d_in.device)
    st = new_status(d_in.device)
    pp_tags(d_in, n, desc, sb, tg, st, stream)
    return sb[:n], tg[:n], read_status(st)


def parse_csv_host(h_in: torch.Tensor, col_types, desc: DfaDesc | None = None,
                   rd: bytes = b"\n", stream=None):
    """End-to-end parse of a HOST uint8 tensor (pinned for full speed).

    Copies the input to the device, sizes the outputs on the device
    (pp_count_byte), parses (pp_parse) and copies every result column back
    into pinned host tensors.  Returns (host columns, status, bytes moved
    host->device, bytes moved device->host).
    """
    dev = torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        d_in = h_in.to(dev, non_blocking=True)
        cols, st = parse_csv(d_in, col_types, desc=desc, rd=rd, stream=s)
        d2h = STATUS_BYTES + 8
        host = []
        for c in cols:
            if c is None:
                host.append(None)
            elif isinstance(c, tuple):
                o = torch.empty(c[0].shape, dtype=c[0].dtype, pin_memory=True)
                ch = torch.empty(c[1].shape, dtype=c[1].dtype, pin_memory=True)
                o.copy_(c[0], non_blocking=True)
                ch.copy_(c[1], non_blocking=True)
                d2h += o.numel() * 4 + ch.numel()
                host.append((o, ch))
            else:
                h = torch.empty(c.shape, dtype=c.dtype, pin_memory=True)
                h.copy_(c, non_blocking=True)
                d2h += h.numel() * h.element_size()
                host.append(h)
        s.synchronize()
    return host, st, int(h_in.numel()), int(d2h)


def tokenize_host(h_in: torch.Tensor, desc: DfaDesc | None = None, stream=None):
    """End-to-end lexing of a HOST uint8 tensor; returns (host (ids, starts,
    lens), status, bytes host->device, bytes device->host)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        d_in = h_in.to(dev, non_blocking=True)
        (ids, starts, lens), st = tokenize(d_in, desc=desc, stream=s)
        out = []
        d2h = 2 * STATUS_BYTES
        for t in (ids, starts, lens):
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t, non_blocking=True)
            d2h += h.numel() * h.element_size()
            out.append(h)
        s.synchronize()
    return tuple(out), st, int(h_in.numel()), int(d2h)
