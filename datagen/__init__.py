"""Seeded synthetic inputs shared by the CPU oracle and the GPU path.

The module only produces bytes (and, for small inputs, the ground truth the
generator encoded).  It contains none of the parsing method's arithmetic.

Workloads (sizes are byte targets; whole records are appended while the total
stays within the target, so CSV inputs end with '\\n'):

  csv4_1mib        1 MiB, 4 string columns, 10 % quoted fields holding
                   ',', '\\n' and doubled quotes
  csv16_256mib     256 MiB, 16 columns i f s i f s i f s i f s i i s s
                   (int64, float64 printed %.6g, strings 0..32 chars,
                   5 % quoted with embedded delimiters)
  csv3_1gib        1 GiB, int32 id, long quoted text (lognormal, mean
                   600 B, max 8 KiB), int8 score 1..5
  csv18_2gib       2 GiB, 18 unquoted columns: 2 timestamps
                   'YYYY-MM-DD HH:MM:SS', 10 int32 in 0..9, 6 float64 %.2f
  json_2gib        2 GiB JSON-like token stream (objects/arrays, strings
                   with backslash escapes, ints, floats, whitespace runs)
  csv18ts_2gib     the csv18_2gib bytes with the two timestamp columns
                   typed as timestamps (int64 seconds) instead of strings

Seeds are 0x5EED0000 + the workload number (1..5); random numbers come from
splitmix64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libdatagen.so")

# column kinds: 'str', 'i8', 'i32', 'i64', 'f64'
_W2 = {"i": "i64", "f": "f64", "s": "str"}
WORKLOADS = {
    "csv4_1mib": dict(index=1, target=1 << 20, kind="csv",
                      cols=["str"] * 4),
    "csv16_256mib": dict(index=2, target=256 << 20, kind="csv",
                         cols=[_W2[c] for c in "ifsifsifsifsiiss"]),
    "csv3_1gib": dict(index=3, target=1 << 30, kind="csv",
                      cols=["i32", "str", "i8"]),
    "csv18_2gib": dict(index=4, target=2 << 30, kind="csv",
                       cols=["str", "str"] + ["i32", "f64"] * 6 + ["i32"] * 4),
    "json_2gib": dict(index=5, target=2 << 30, kind="tokens", cols=None),
    # the 2 GiB numeric input with its timestamps converted to int64 seconds
    "csv18ts_2gib": dict(index=4, target=2 << 30, kind="csv",
                         cols=["ts", "ts"] + ["i32", "f64"] * 6 + ["i32"] * 4),
}
TOKEN_KINDS = ["{", "}", "[", "]", ",", ":", "string", "int", "float", "ws"]


class _Info(ctypes.Structure):
    _fields_ = [("n_bytes", ctypes.c_uint64), ("n_records", ctypes.c_uint64),
                ("n_fields", ctypes.c_uint64), ("n_tokens", ctypes.c_uint64),
                ("quoted_bytes", ctypes.c_uint64), ("side_len", ctypes.c_uint64),
                ("side_overflow", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("col_value_bytes", ctypes.c_uint64 * 64)]


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-o", _SO, src, "-lm"])
    return _SO


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        lib.dg_generate.restype = ctypes.c_int
        lib.dg_generate.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                    ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                    ctypes.c_uint64, ctypes.POINTER(_Info), ctypes.c_void_p,
                                    ctypes.c_uint64]
        _lib = lib
    return _lib


def seed_of(name: str) -> int:
    return 0x5EED0000 + WORKLOADS[name]["index"]


def generate(name: str, target: int | None = None, seed: int | None = None,
             out_ptr: int | None = None, out_cap: int | None = None,
             sidecar: bool = False, record_offsets: bool = False,
             record_offsets_cap: int | None = None):
    """Generate workload `name`.

    Returns (data, info, side): `data` is a numpy uint8 array (a view of the
    caller's buffer when `out_ptr` is given), `info` a dict with n_bytes,
    n_records, n_fields, n_tokens, quoted_bytes, and `side` the ground-truth
    sidecar bytes (or None).  With `record_offsets`, info["record_offsets"]
    holds the start offset of each record (top-level value for the token
    stream), the first `record_offsets_cap` of them (default: room for all).
    """
    w = WORKLOADS[name]
    target = w["target"] if target is None else int(target)
    seed = seed_of(name) if seed is None else int(seed)
    lib = _load()
    if out_ptr is None:
        buf = np.empty(target, dtype=np.uint8)
        ptr, cap = buf.ctypes.data, target
    else:
        buf, ptr, cap = None, int(out_ptr), int(out_cap)
    side_buf, side_cap = None, 0
    if sidecar:
        side_cap = 4 * target + 1024
        side_buf = np.empty(side_cap, dtype=np.uint8)
    info = _Info()
    roff = None
    if record_offsets:
        cap_r = target // 2 + 2 if record_offsets_cap is None else int(record_offsets_cap)
        roff = np.zeros(max(cap_r, 1), dtype=np.uint64)
    rc = lib.dg_generate(w["index"], target, seed, ptr, cap,
                         side_buf.ctypes.data if sidecar else None, side_cap,
                         ctypes.byref(info), roff.ctypes.data if roff is not None else None,
                         roff.size if roff is not None else 0)
    if rc != 0:
        raise RuntimeError(f"dg_generate({name}) failed: {rc}")
    if sidecar and info.side_overflow:
        raise RuntimeError("sidecar overflow")
    d = {k: int(getattr(info, k)) for k in
         ("n_bytes", "n_records", "n_fields", "n_tokens", "quoted_bytes")}
    d["col_value_bytes"] = [int(info.col_value_bytes[i]) for i in range(64)]
    if roff is not None:
        nrec = d["n_records"] if w["kind"] == "csv" else int(np.count_nonzero(roff)) + 1
        d["record_offsets"] = roff[: min(nrec, roff.size)]
    if buf is not None:
        data = buf[: info.n_bytes]
    else:
        data = np.ctypeslib.as_array((ctypes.c_uint8 * info.n_bytes).from_address(ptr))
    side = bytes(side_buf[: info.side_len]) if sidecar else None
    return data, d, side


def sidecar_fields(side: bytes) -> list[bytes]:
    """Split a CSV sidecar into the per-field ground-truth values."""
    parts = side.split(b"\x00")
    assert parts[-1] == b""
    return parts[:-1]


def sidecar_tokens(side: bytes) -> list[tuple[int, int]]:
    """Decode a token-stream sidecar into (kind, length) pairs."""
    a = np.frombuffer(side, dtype=np.uint8).reshape(-1, 5)
    kinds = a[:, 0].astype(np.int64)
    lens = (a[:, 1].astype(np.int64) | (a[:, 2].astype(np.int64) << 8)
            | (a[:, 3].astype(np.int64) << 16) | (a[:, 4].astype(np.int64) << 24))
    return list(zip(kinds.tolist(), lens.tolist()))
