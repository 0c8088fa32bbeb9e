"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/pp.h declares, its DFA descriptors agree cell by cell with
the oracle's independently written transition switches, and bad arguments
are rejected before any device work."""
import ctypes
import os
import re
from collections import deque

import numpy as np
import pytest

import dfa_parsing_delimiter_gb300 as pp
import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pp_\w+)\s*\(", src)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert {"pp_parse", "pp_tokenize", "pp_tags", "pp_desc_csv", "pp_desc_json_lexer",
            "pp_strerror", "pp_count_byte"} <= set(names)
    L = pp.lib()
    for n in names:
        assert hasattr(L, n), n


def test_struct_sizes():
    assert ctypes.sizeof(pp.DfaDesc) == 8 + 256 + 256 + 256 + 16 + 256 + 12 + 4 * 8
    assert pp.STATUS_BYTES == 32 + 8 * 64 + 8  # + n_dropped


def _reach(kind):
    """Shortest byte prefix reaching each DFA state (BFS over all bytes)."""
    ns = O.nstates(kind)
    start = 0
    prefix = {start: b""}
    q = deque([start])
    while q:
        s = q.popleft()
        for b in range(256):
            nx = int(O.stv(bytes([b]), kind=kind)[s])
            if nx not in prefix:
                prefix[nx] = prefix[s] + bytes([b])
                q.append(nx)
    assert len(prefix) == ns
    return prefix


@pytest.mark.parametrize("kind", [O.KIND_CSV, O.KIND_LEX, O.KIND_CSV_CRLF])
def test_desc_matches_oracle_cell_by_cell(kind):
    d = {O.KIND_CSV: pp.desc_csv, O.KIND_LEX: pp.desc_json_lexer,
         O.KIND_CSV_CRLF: pp.desc_csv_crlf}[kind]()
    ns = O.nstates(kind)
    assert d.n_states == ns
    prefix = _reach(kind)
    for b in range(256):
        g = d.byte_to_group[b]
        nxt = O.stv(bytes([b]), kind=kind)
        for s in range(ns):
            assert d.delta[g][s] == nxt[s], (kind, b, s)
            _, tg, _ = O.tags(prefix[s] + bytes([b]), kind=kind)
            assert d.tag[s][g] == tg[-1], (kind, b, s)


def test_desc_accepting_states():
    d = pp.desc_csv()
    # oracle: end-of-input error iff the state is not accepting
    for s, p in _reach(O.KIND_CSV).items():
        _, st = O.csv_parse(p, ["str"])
        bad_end = bool(st["error"] & O.E_BAD_END_STATE)
        if s == 4:
            continue
        assert bool((d.accept_mask >> s) & 1) == (not bad_end), s
    d = pp.desc_json_lexer()
    for s, p in _reach(O.KIND_LEX).items():
        _, st = O.tokenize(p)
        if s == 15:
            continue
        assert bool((d.accept_mask >> s) & 1) == (not st["error"] & O.E_BAD_END_STATE), s


def test_desc_csv_crlf_arguments():
    L = pp.lib()
    for fd, q in ((10, 34), (13, 34), (44, 10), (44, 13), (44, 44)):
        assert L.pp_desc_csv_crlf(ctypes.byref(pp.DfaDesc()), fd, q) == pp.PP_EINVAL
    d = pp.desc_csv_crlf(b";", b"'")
    assert d.n_groups == 5 and d.byte_to_group[13] == 4 and d.byte_to_group[10] == 2
    assert d.byte_to_group[ord(";")] == 1 and d.byte_to_group[ord("'")] == 0


def test_desc_csv_custom_delimiters():
    d = pp.desc_csv(b"|", b";", b"'")
    assert d.byte_to_group[ord("|")] == 1 and d.byte_to_group[ord(";")] == 2
    assert d.byte_to_group[ord("'")] == 0 and d.byte_to_group[ord(",")] == 3
    L = pp.lib()
    assert L.pp_desc_csv(ctypes.byref(pp.DfaDesc()), 44, 44, 34) == pp.PP_EINVAL


def test_bad_arguments_rejected_without_gpu():
    L = pp.lib()
    d = pp.desc_csv()
    ct = (ctypes.c_int * 1)(0)
    # NULL status
    assert L.pp_parse(None, 0, ctypes.byref(d), 1, ctypes.addressof(ct), None, None, None, 0,
                      None, None, None) == pp.PP_EINVAL
    # n_cols out of range
    assert L.pp_parse(None, 0, ctypes.byref(d), 0, ctypes.addressof(ct), None, None, None, 0,
                      None, 1, None) == pp.PP_EINVAL
    # bad column type
    bad = (ctypes.c_int * 1)(9)
    assert L.pp_parse(None, 0, ctypes.byref(d), 1, ctypes.addressof(bad), None, None, None, 0,
                      None, 1, None) == pp.PP_EINVAL
    # NULL input with n > 0
    assert L.pp_parse(None, 5, ctypes.byref(d), 1, ctypes.addressof(ct), None, None, None, 0,
                      None, 1, None) == pp.PP_EINVAL
    # a 16-state DFA is not accepted by pp_parse
    j = pp.desc_json_lexer()
    assert L.pp_parse(None, 0, ctypes.byref(j), 1, ctypes.addressof(ct), None, None, None, 0,
                      None, 1, None) == pp.PP_EINVAL
    # corrupt descriptor: a transition out of range
    d2 = pp.desc_csv()
    d2.delta[0][0] = 9
    assert L.pp_tags(1, 1, ctypes.byref(d2), 1, 1, 1, None) == pp.PP_EINVAL
    # background group that is not idempotent
    d3 = pp.desc_csv()
    d3.background_group = 0
    assert L.pp_parse(None, 0, ctypes.byref(d3), 1, ctypes.addressof(ct), None, None, None, 0,
                      None, 1, None) == pp.PP_EINVAL
    # tokenize: outputs missing with a capacity
    assert L.pp_tokenize(1, 1, ctypes.byref(j), None, None, None, 5, 1, None) == pp.PP_EINVAL
    assert L.pp_count_byte(None, 3, 10, 1, None) == pp.PP_EINVAL
    # count fields: no output, a bad descriptor, an input beyond 64 GiB
    csv = pp.desc_csv()
    assert L.pp_count_fields(1, 1, ctypes.byref(csv), None, 1, None) == pp.PP_EINVAL
    assert L.pp_count_fields(1, 1, ctypes.byref(d2), 1, 1, None) == pp.PP_EINVAL
    assert L.pp_count_fields(1, (1 << 36) + 1, ctypes.byref(csv), 1, 1, None) == pp.PP_ETOOLARGE
    assert L.pp_count_fields(1, 1, ctypes.byref(csv), 1, None, None) == pp.PP_EINVAL
    assert pp.lib().pp_strerror(pp.PP_EINVAL) == b"invalid argument"


def test_oracle_package_is_not_imported_by_library():
    import sys
    src = open(os.path.join(ROOT, "dfa_parsing_delimiter_gb300", "__init__.py")).read()
    assert "oracle" not in src.replace("no CPU fallback", "")
    for f in os.listdir(os.path.join(ROOT, "dfa_parsing_delimiter_gb300", "csrc")):
        text = open(os.path.join(ROOT, "dfa_parsing_delimiter_gb300", "csrc", f)).read()
        assert "pp_oracle" not in text and "or_csv_parse" not in text


def test_encoded_csv_descriptor():
    """pp_desc_csv_enc: the byte CSV DFA's table, with quote, field and
    record delimiter as code points (ASCII ones through byte_to_group, the
    others through the symbol table); bad code points are refused."""
    b = pp.desc_csv()
    d = pp.desc_csv_enc("utf-8", "\u00a7", "\u2028", '"')
    assert d.encoding == pp.ENC_UTF8 and d.n_syms == 2
    assert [(d.sym_cp[k], d.sym_group[k]) for k in range(2)] == [(0xA7, 1), (0x2028, 2)]
    assert d.byte_to_group[ord('"')] == 0 and d.byte_to_group[ord(",")] == 3
    assert d.byte_to_group[0x80] == 3 and d.byte_to_group[10] == 3
    for g in range(4):
        for st in range(5):
            assert d.delta[g][st] == b.delta[g][st] and d.tag[st][g] == b.tag[st][g]
    u = pp.desc_csv_enc("utf-16-le")
    assert u.encoding == pp.ENC_UTF16LE and u.n_syms == 0 and u.byte_to_group[ord(",")] == 1
    for bad in ((0xD800, 10, 34), (44, 44, 34), (0x110000, 10, 34)):
        with pytest.raises(RuntimeError):
            pp.desc_csv_enc("utf-8", *bad)
