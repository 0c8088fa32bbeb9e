"""Pins for the oracle on inputs whose symbols span several bytes (ParPaRaw
Section 3.4: UTF-8 and UTF-16 symbols that may cross chunk boundaries).
The references are independent of the oracle: Python's codecs decode the
input and Python's csv module (an RFC-4180 reader that takes any one
character as delimiter) parses the text; every string over a small
alphabet of 1-, 2- and 4-byte symbols is checked."""
import csv
import io
import itertools

import pytest

import oracle as O

ALPHABET = ["a", "é", "§", '"', "\n", "😀"]   # 1, 2, 2, 1, 1, 4 bytes in UTF-8


def _ref(text, fd):
    rows = list(csv.reader(io.StringIO(text, newline=""), delimiter=fd))
    return [r if r else [""] for r in rows]      # an empty line is one empty field


def _fields(cols, st, k, enc):
    out = []
    for r in range(st["n_records"]):
        out.append([bytes(cols[c][1][cols[c][0][r]:cols[c][0][r + 1]]).decode(enc)
                    for c in range(k)])
    return out


@pytest.mark.parametrize("enc", ["utf-8", "utf-16-le"])
def test_bruteforce_against_csv_module(enc):
    """Every string of up to 5 symbols, '§' as field delimiter: where the
    oracle reports no error, its fields are Python's."""
    checked = 0
    for n in range(6):
        for tup in itertools.product(ALPHABET, repeat=n):
            text = "".join(tup)
            data = text.encode(enc)
            ref = _ref(text, "§")
            k = max((len(r) for r in ref), default=1)
            cols, st = O.csv_parse(data, ["str"] * k, fd="§", rd="\n", quote='"', encoding=enc)
            if st["error"] & ~O.E_COLCOUNT:
                continue
            got = _fields(cols, st, k, enc)
            want = [r + [""] * (k - len(r)) for r in ref]
            assert got == want, (text, got, want)
            checked += 1
    assert checked > 1500


def test_utf8_mode_equals_byte_mode_on_ascii_specials():
    """With ASCII delimiters and valid UTF-8 text the symbol walk and the
    byte walk give the same columns."""
    text = 'aé,"§,😀\n""x",b\n\n😀😀,é"\n'
    data = text.encode()
    a, sa = O.csv_parse(data, ["str", "str"], encoding="utf-8", fd=",", rd="\n", quote='"')
    b, sb = O.csv_parse(data, ["str", "str"])
    assert sa == sb
    for (oa, ca), (ob, cb) in zip(a, b):
        assert oa.tolist() == ob.tolist() and bytes(ca) == bytes(cb)


def test_offsets_are_those_of_a_symbols_last_byte():
    """An invalid transition and a record delimiter are reported at their
    symbol's last byte; a field starts after its delimiter's last byte."""
    # '"ab"é': after the closing quote, 'é' (bytes 4, 5) is invalid at byte 5
    _, st = O.csv_parse('"ab"é\n'.encode(), ["str"], encoding="utf-8", fd=",", rd="\n")
    assert st["error"] == O.E_INVALID_INPUT and st["first_error_offset"] == 5
    # record delimiter U+2028 (3 bytes): a record of 1 field ends at its last byte
    data = "x§y\u2028z\u2028".encode()
    _, st = O.csv_parse(data, ["str", "str"], encoding="utf-8", fd="§", rd="\u2028")
    assert st["n_records"] == 2 and st["error"] == O.E_COLCOUNT
    assert st["first_error_offset"] == len("x§y\u2028z".encode()) + 2
    # numbers: an error is reported at the field's first byte, after the delimiter
    cols, st = O.csv_parse("1§x\n".encode(), ["i32", "i32"], encoding="utf-8", fd="§", rd="\n")
    assert st["error"] == O.E_NUM_SYNTAX and st["first_error_offset"] == 3
    assert cols[0].tolist() == [1]


def test_ill_formed_utf8_is_one_other_symbol():
    # a stray continuation byte at the start, a truncated sequence, an
    # overlong ',' (C0 AC) and a byte 0xFF: none is a delimiter
    data = b"\xa7,\xc2\xc0\xac,\xff\n"
    cols, st = O.csv_parse(data, ["str", "str", "str"], encoding="utf-8", fd=",", rd="\n")
    assert st["error"] == 0
    offs, chars = cols[0]
    assert bytes(chars[offs[0]:offs[1]]) == b"\xa7"
    offs, chars = cols[1]
    assert bytes(chars[offs[0]:offs[1]]) == b"\xc2\xc0\xac"
    # '§' = C2 A7 followed by a stray continuation byte is not the delimiter
    cols, st = O.csv_parse(b"a\xc2\xa7\x80b\n", ["str"], encoding="utf-8", fd="§", rd="\n")
    assert st["error"] == 0 and bytes(cols[0][1]) == b"a\xc2\xa7\x80b"


def test_utf16_surrogates_and_odd_end():
    text = "😀§\ud83d"                                   # a pair, the delimiter, a lone high surrogate
    data = text.encode("utf-16-le", "surrogatepass") + b"\n\x00" + b"x"   # and an odd last byte
    cols, st = O.csv_parse(data, ["str", "str"], encoding="utf-16-le", fd="§", rd="\n")
    assert st["n_records"] == 2 and st["error"] == O.E_COLCOUNT
    offs, chars = cols[0]
    assert bytes(chars[offs[0]:offs[1]]) == "😀".encode("utf-16-le")
    assert bytes(chars[offs[1]:offs[2]]) == b"x"
    offs, chars = cols[1]
    assert bytes(chars[offs[0]:offs[1]]) == "\ud83d".encode("utf-16-le", "surrogatepass")
