"""Inputs whose symbols span several bytes (ParPaRaw Section 3.4: UTF-8 and
UTF-16 symbols crossing chunk boundaries), parsed with pp_desc_csv_enc
descriptors and compared with the oracle element by element: multi-byte
delimiters and quotes placed across every chunk and tile boundary offset,
non-BMP characters (4-byte symbols, surrogate pairs), numbers next to
multi-byte delimiters and fields begun in earlier tiles, ill-formed
sequences, invalid transitions and column-count errors at a symbol's last
byte, the options of pp_parse_ex and the fixed-scratch entry point."""
import random

import numpy as np
import pytest
import torch

import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import compare_csv, to_dev

pytestmark = pytest.mark.gpu
TILE = 16384
CB = 32


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _text(rng, n_rows, k, fd, alpha, quote='"', p_quote=0.2):
    rows = []
    for _ in range(n_rows):
        f = []
        for _ in range(k):
            v = "".join(rng.choice(alpha) for _ in range(rng.randint(0, 12)))
            if rng.random() < p_quote:
                v = quote + v.replace(quote, quote * 2) + fd + "\n" + quote
            else:
                v = v.replace(quote, "").replace(fd, "").replace("\n", "")
            f.append(v)
        rows.append(fd.join(f))
    return "\n".join(rows) + "\n"


@pytest.mark.parametrize("enc", ["utf-8", "utf-16-le"])
@pytest.mark.parametrize("seed", range(3))
def test_random_text_many_tiles(enc, seed):
    rng = random.Random(seed)
    alpha = list("ab ,x1") + ["é", "§", "中", "😀", '"']
    text = _text(rng, 3000, 4, "§", alpha)
    data = text.encode(enc)
    assert len(data) > 6 * TILE
    compare_csv(data, ["str"] * 4, fd="§", rd="\n", quote='"', encoding=enc)


@pytest.mark.parametrize("enc", ["utf-8", "utf-16-le"])
def test_delimiters_across_every_boundary_offset(enc):
    """A 2-byte (UTF-8) or surrogate-pair field delimiter and 4-byte values
    placed so that their bytes straddle chunk and tile boundaries at every
    offset."""
    fd = "§" if enc == "utf-8" else "😀"
    unit = 1 if enc == "utf-8" else 2
    for shift in range(0, 8):
        pad = "a" * ((TILE - 2 * CB) // unit - 1 + shift)
        recs = []
        for i in range(200):
            recs.append("x" * (i % 7) + fd + "😀" * (i % 3) + "é" + fd + '"' + "q" * (i % 5) + fd + '"')
        text = pad + fd + "b\n" + "\n".join(recs) + "\n"
        compare_csv(text.encode(enc), ["str"] * 3, fd=fd, rd="\n", quote='"', encoding=enc)


def test_multibyte_record_delimiter_and_quote():
    rng = random.Random(4)
    rows = []
    for i in range(2000):
        f = ["".join(rng.choice("ab«»é") for _ in range(rng.randint(0, 9))) for _ in range(3)]
        f[1] = "„" + f[1].replace("„", "„„") + "\u2028,„"
        rows.append(",".join(f))
    text = "\u2028".join(rows) + "\u2028"
    compare_csv(text.encode(), ["str"] * 3, fd=",", rd="\u2028", quote="„", encoding="utf-8")


def test_numbers_with_multibyte_delimiters():
    """Integer and float columns next to a 2-byte delimiter; long fields and
    fields spanning tiles (converted by the long-field pass, whose CSV walk
    decodes the symbols too)."""
    rng = random.Random(8)
    rows = []
    for i in range(3000):
        a = str(rng.randint(-10 ** 9, 10 ** 9))
        b = f"{rng.uniform(-1e3, 1e3):.5f}"
        if rng.random() < 0.02:
            b = "0" * rng.randint(300, 20000) + b.lstrip("-")
        if rng.random() < 0.05:
            a = '"' + a + '"'
        rows.append(a + "§" + b + "§" + "é" * (i % 4))
    data = ("\n".join(rows) + "\n").encode()
    pp.debug_long_fields(reset=True)
    compare_csv(data, ["i64", "f64", "str"], fd="§", rd="\n", quote='"', encoding="utf-8")
    assert pp.debug_long_fields() > 0


def test_errors_at_a_symbols_last_byte():
    # after a closing quote, 'é' crossing a chunk boundary is invalid at its last byte
    for pre in range(CB - 4, CB + 2):
        text = "a" * pre + '§"ab"é§x\n'
        compare_csv(text.encode(), ["str", "str", "str"], fd="§", rd="\n", encoding="utf-8")
    # column counts with a 3-byte record delimiter
    text = "a§b\u2028c\u2028d§e§f\u2028"
    compare_csv(text.encode(), ["str", "str"], fd="§", rd="\u2028", encoding="utf-8")


def test_ill_formed_utf8():
    rng = random.Random(12)
    parts = [b"a", b"\xc3\xa9", b"\xa7", b"\xc2", b"\xff", b"\xc2\xa7", b"\xc2\xa7\x80",
             b"\xe4\xb8", b"\n", b'"', b"\xf0\x9f\x98\x80"]
    data = b"".join(rng.choice(parts) for _ in range(40000))
    compare_csv(data, ["str"] * 3, fd="§", rd="\n", quote='"', encoding="utf-8")


def test_utf16_surrogates_and_odd_end():
    rng = random.Random(13)
    units = ["a", "é", ",", "\n", "😀", '"', "\ud83d", "\ude00"]
    text = "".join(rng.choice(units) for _ in range(30000))
    data = text.encode("utf-16-le", "surrogatepass")
    compare_csv(data, ["str"] * 2, fd=",", rd="\n", quote='"', encoding="utf-16-le")
    compare_csv(data + b"x", ["str"] * 2, fd=",", rd="\n", quote='"', encoding="utf-16-le")


def test_options_and_fixed_scratch_with_utf8():
    rng = random.Random(14)
    rows = []
    for i in range(1500):
        k = 2 if rng.random() < 0.9 else 3
        rows.append("§".join("é" * rng.randint(0, 5) + str(i) for _ in range(k)))
    data = ("\n".join(rows) + "\n").encode()
    n = len(data)
    desc = pp.desc_csv_enc("utf-8", "§", "\n", '"')
    out = pp.CsvOutputs(["str", "i32"], n + 1, [n, 0])
    out.run_ex(to_dev(data), n, desc, reject=True, skip_records=[0, 5, 77])
    st = pp.read_status(out.status, 2)
    ref, rst = O.csv_parse(data, ["str", "i32"], fd="§", quote='"', encoding="utf-8",
                           reject=True, skip_records=[0, 5, 77])
    assert st["error"] == rst["error"] and st["first_error_offset"] == rst["first_error_offset"]
    assert st["n_records"] == rst["n_records"] and st["n_dropped"] == rst["n_dropped"]
    got = out.results(st)
    assert np.array_equal(got[0][0].cpu().numpy(), ref[0][0])
    assert np.array_equal(got[0][1].cpu().numpy(), ref[0][1])
    assert np.array_equal(got[1].cpu().numpy(), ref[1])
    out2 = pp.CsvOutputs(["str", "i32"], n + 1, [n, 0])
    out2.run_noalloc(to_dev(data), n, desc)
    s2 = pp.read_status(out2.status, 2)
    ref2, rs2 = O.csv_parse(data, ["str", "i32"], fd="§", quote='"', encoding="utf-8")
    assert s2["error"] == rs2["error"] and s2["n_records"] == rs2["n_records"]
    g2 = out2.results(s2)
    assert np.array_equal(g2[0][1].cpu().numpy(), ref2[0][1])
    assert np.array_equal(g2[1].cpu().numpy(), ref2[1])


def test_entry_points_without_encodings_refuse_them():
    desc = pp.desc_csv_enc("utf-8", "§")
    d_in = to_dev(b"a\n")
    st = pp.new_status()
    fields = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert pp.lib().pp_count_fields(d_in.data_ptr(), 2, desc, fields.data_ptr(), st.data_ptr(),
                                    None) == 1
    out = pp.CsvOutputs(["ts"], 2, [0])
    with pytest.raises(RuntimeError):
        out.run(d_in, 2, desc)
