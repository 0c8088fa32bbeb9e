"""pp_parse_noalloc (pp_parse with its scratch in a fixed buffer compiled
into the library) against the oracle and against pp_parse on the same
inputs: two calls in a row, each equal to the oracle's result and to
pp_parse's (integers, offsets and chars exactly, floats within 1 ulp), and
inputs too large for the buffer rejected.  The no-alloc call runs the
parse's own kernels with scratch carved from the fixed buffer; comparing
with the oracle as well keeps a fault the two calls share from passing
unnoticed.

Named to be collected last, so it also runs after every other test has used
the library in the same process."""
import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import to_dev, ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _outputs(col_types, n, n_rec):
    return pp.CsvOutputs(col_types, n_rec + 1, [n] * len(col_types))


def _assert_same(a, sa, b, sb, col_types):
    assert sa == sb, (sa, sb)
    ra, rb = a.results(sa), b.results(sb)
    for c, t in enumerate(col_types):
        if t == "str":
            assert torch.equal(ra[c][0], rb[c][0]), f"offsets col {c}"
            assert torch.equal(ra[c][1], rb[c][1]), f"chars col {c}"
        elif t == "f64":
            d = ulp_diff(ra[c].cpu().numpy(), rb[c].cpu().numpy())
            assert d.size == 0 or int(d.max()) <= 1, f"f64 col {c}"
        elif t != "skip":
            assert torch.equal(ra[c], rb[c]), f"col {c}"


def _assert_oracle(data, col_types, out, st):
    ref, rst = O.csv_parse(data, col_types)
    assert st["error"] == rst["error"] == 0, (st, rst)
    assert st["n_records"] == rst["n_records"]
    got = out.results(st)
    for c, t in enumerate(col_types):
        if t == "str":
            assert st["chars_len"][c] == rst["chars_len"][c], c
            assert np.array_equal(got[c][0].cpu().numpy(), ref[c][0]), f"offsets col {c}"
            assert np.array_equal(got[c][1].cpu().numpy(), ref[c][1]), f"chars col {c}"
        elif t == "f64":
            g = got[c].cpu().numpy()
            d = ulp_diff(g, ref[c])
            assert d.size == 0 or int(d.max()) <= 1, f"f64 col {c}"
            assert np.array_equal(np.signbit(g), np.signbit(ref[c]))
        elif t != "skip":
            assert np.array_equal(got[c].cpu().numpy(), ref[c]), f"col {c}"


@pytest.mark.parametrize("name,target", [
    ("csv4_1mib", None),
    ("csv16_256mib", 3 << 20),
    ("csv18_2gib", (2 << 20) + 77),
    ("csv3_1gib", 5 * 16384 + 3),
])
def test_noalloc_matches_pp_parse_on_two_calls_in_a_row(name, target):
    data, info, _ = datagen.generate(name, target=target)
    col_types = datagen.WORKLOADS[name]["cols"]
    n = len(data)
    d_in = to_dev(data)
    desc = pp.desc_csv()
    ref = _outputs(col_types, n, info["n_records"])
    ref.run(d_in, n, desc)
    sref = pp.read_status(ref.status, len(col_types))
    assert sref["error"] == 0 and sref["n_records"] == info["n_records"]
    first = _outputs(col_types, n, info["n_records"])
    second = _outputs(col_types, n, info["n_records"])
    first.run_noalloc(d_in, n, desc)
    second.run_noalloc(d_in, n, desc)   # same stream, right after the first
    torch.cuda.synchronize()
    for out in (first, second):
        st = pp.read_status(out.status, len(col_types))
        _assert_oracle(data, col_types, out, st)
        _assert_same(ref, sref, out, st, col_types)


def test_noalloc_sizing_pass_matches():
    data, info, _ = datagen.generate("csv16_256mib", target=1 << 20)
    col_types = datagen.WORKLOADS["csv16_256mib"]["cols"]
    d_in = to_dev(data)
    st = [pp.new_status(), pp.new_status()]
    for i, f in enumerate((pp.pp_parse, pp.pp_parse_noalloc)):
        f(d_in, len(data), pp.desc_csv(), col_types, None, None, None, 0,
          [0] * len(col_types), st[i])
    a, b = (pp.read_status(s, len(col_types)) for s in st)
    assert a == b and a["n_records"] == info["n_records"]


def test_noalloc_rejects_input_larger_than_its_buffer():
    # 64 columns, 16 of them strings: the buffer holds about 225 MiB of input
    col_types = ["str"] * 16 + ["i32"] * 48
    n = 240 << 20
    d_in = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = pp.CsvOutputs(col_types, 1, [1] * 64)
    with pytest.raises(RuntimeError, match=r"pp_parse_noalloc failed: .*\(4\)"):
        out.run_noalloc(d_in, n, pp.desc_csv())
    # a smaller input with the same schema is accepted
    small = d_in[: 1 << 20]
    out.run_noalloc(small, small.numel(), pp.desc_csv())
    torch.cuda.synchronize()
