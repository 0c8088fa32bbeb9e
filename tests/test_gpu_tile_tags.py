"""The tag bitmaps the tile pass itself computes (ParPaRaw Section 3.1: the
field-delimiter, record-delimiter and control bitmaps; exported by
pp_debug_parse_tags), compared bit by bit with the oracle's sequential walk,
on inputs whose quoted fields, doubled quotes and CRLF line ends fall across
chunk and tile boundaries."""
import random

import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import to_dev

pytestmark = pytest.mark.gpu
TILE = 16384


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _compare(data, desc, kind, offset=0):
    fd, rd, ct, st = pp.debug_parse_tags(to_dev(data, offset), desc)
    _, tags, _ = O.tags(data, kind=kind)
    assert st["error"] & (O.E_INVALID_INPUT | O.E_BAD_END_STATE) == 0
    assert np.array_equal(fd, tags == 1)
    assert np.array_equal(rd, tags == 2)
    assert np.array_equal(ct, tags == 3)


@pytest.mark.parametrize("seed", range(3))
def test_tile_tags_quoted_csv(seed):
    data, _, _ = datagen.generate("csv4_1mib", target=6 * TILE + 1000 * seed + 17)
    _compare(bytes(data), pp.desc_csv(), O.KIND_CSV)


def test_tile_tags_long_quoted_text_misaligned():
    data, _, _ = datagen.generate("csv3_1gib", target=8 * TILE + 5)
    _compare(bytes(data), pp.desc_csv(), O.KIND_CSV, offset=3)


@pytest.mark.parametrize("at", [TILE - 2, TILE - 1, TILE, 2 * TILE - 33, 2 * TILE - 32])
def test_tile_tags_doubled_quotes_at_boundaries(at):
    rng = random.Random(at)
    head = "".join(rng.choice("ab,\n") for _ in range(at - 2))
    data = (head + '\n"x""' + 'y""' * 3 + '",z\n' + '"' + '""' * 600 + '"\n').encode()
    _compare(data, pp.desc_csv(), O.KIND_CSV)


def test_tile_tags_crlf():
    rng = random.Random(7)
    rows = []
    for _ in range(4000):
        f = ["".join(rng.choice("ab1 ") for _ in range(rng.randint(0, 8))) for _ in range(3)]
        if rng.random() < 0.2:
            f[1] = '"' + f[1] + '\r\n,""' + '"'
        rows.append(",".join(f))
    data = ("\r\n".join(rows) + "\r\n").encode()
    _compare(data, pp.desc_csv_crlf(), O.KIND_CSV_CRLF)
