"""Pins for the oracle's capacity path: outputs smaller than the input needs
set the CAPACITY bit, counts still cover the whole input, and what fits is
what an unbounded run writes.  Exact capacities are the edge that must not
flag.  Expected counts come from the text of the inputs (records are lines
here, with no quotes), not from the oracle."""
import numpy as np

import oracle as O

ROWS = [b"a,1", b"bb,22", b"ccc,333", b"dddd,4444", b"eeeee,55555"]
DATA = b"\n".join(ROWS) + b"\n"


def test_records_capacity_exact_and_short():
    cols, st = O.csv_parse(DATA, ["str", "i64"], records_capacity=len(ROWS))
    assert st["error"] == 0 and st["n_records"] == 5
    cols3, st3 = O.csv_parse(DATA, ["str", "i64"], records_capacity=3)
    assert st3["error"] == O.E_CAPACITY and st3["n_records"] == 5
    assert cols3[1].tolist()[:3] == [1, 22, 333]
    offs, chars = cols3[0]
    assert offs.tolist()[:4] == [0, 1, 3, 6] and bytes(chars[:6]) == b"abbccc"


def test_chars_capacity_exact_and_short():
    total = sum(len(r.split(b",")[0]) for r in ROWS)          # 15 value bytes
    _, st = O.csv_parse(DATA, ["str", "skip"], chars_capacity=[total, 0])
    assert st["error"] == 0 and st["chars_len"][0] == total
    _, st = O.csv_parse(DATA, ["str", "skip"], chars_capacity=[total - 1, 0])
    assert st["error"] == O.E_CAPACITY and st["n_records"] == 5
    assert st["chars_len"][0] <= total - 1                      # nothing written past it


def test_tokenize_capacity_exact_and_short():
    data = b'[1, "ab", 2.5]'                                    # [ 1 , ws "ab" , ws 2.5 ]
    n_tok = 9
    (ids, starts, lens), st = O.tokenize(data, capacity=n_tok)
    assert st["error"] == 0 and st["n_tokens"] == n_tok
    assert starts.tolist() == [0, 1, 2, 3, 4, 8, 9, 10, 13]
    (ids4, starts4, lens4), st4 = O.tokenize(data, capacity=4)
    assert st4["error"] == O.E_CAPACITY and st4["n_tokens"] == n_tok
    assert starts4.tolist()[:4] == [0, 1, 2, 3]
    assert np.array_equal(lens4[:3], lens[:3]) and np.array_equal(ids4[:3], ids[:3])
