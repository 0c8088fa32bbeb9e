"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (one pp_parse / pp_tokenize call over the whole input on the
current stream, outputs preallocated from the generator's counts).

The oracle is too slow to parse 2 GiB inside a test, so each workload is
checked two ways:

* properties over the whole output that hold at any size: the status is
  clean, the record (token) count and the value bytes per string column
  equal what the generator wrote, Arrow offsets start at 0, never decrease
  and end at the chars length; token starts are strictly increasing, each
  token ends where the next starts and the last ends at the input's end;
* element-by-element comparison with the oracle on sampled windows of whole
  records (top-level values for the token stream) spread over the input,
  including its first and last records.  The generator records where each
  record starts and which record it is, so a window's rows are known without
  the GPU's help; a record starts in the DFA's start state, which is where
  the oracle begins.  Floats within 1 ulp, everything else bit-exact.
"""
import numpy as np
import pytest
import torch

import datagen
import dfa_parsing_delimiter_gb300 as pp
import oracle as O
from gpu_util import ulp_diff

pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]

N_WINDOWS = 48
WINDOW_RECORDS = 24


@pytest.fixture(autouse=True, scope="module")
def _device():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)


def _windows(n_rec, seed):
    """Start record of each window: the first, the last and spread between."""
    rng = np.random.default_rng(seed)
    k = min(WINDOW_RECORDS, n_rec)
    starts = set([0, max(n_rec - k, 0)])
    starts.update(int(x) for x in rng.integers(0, max(n_rec - k, 1), N_WINDOWS - 2))
    return sorted(starts), k


def _roff_cap(name):
    """Room for every record's start: all workloads average over 64 bytes a
    record except the 1 MiB one, which the constant term covers."""
    return datagen.WORKLOADS[name]["target"] // 64 + (1 << 20)


def _to_device(data):
    n = data.size
    d_in = torch.empty(n + 16, dtype=torch.uint8, device="cuda")[:n]
    d_in.copy_(torch.from_numpy(data))
    return d_in


@pytest.mark.parametrize("name", ["csv4_1mib", "csv16_256mib", "csv3_1gib", "csv18_2gib",
                                  "csv18ts_2gib"])
def test_parse_full_size(name):
    w = datagen.WORKLOADS[name]
    cols = w["cols"]
    data, info, _ = datagen.generate(name, record_offsets=True,
                                     record_offsets_cap=_roff_cap(name))
    roff = info["record_offsets"]
    R = info["n_records"]
    assert roff.size == R
    n = data.size
    d_in = _to_device(data)
    chars_cap = [info["col_value_bytes"][c] if t == "str" else 0 for c, t in enumerate(cols)]
    out = pp.CsvOutputs(cols, R, chars_cap)
    stream = torch.cuda.current_stream()
    out.run(d_in, n, pp.desc_csv(), stream)
    st = pp.read_status(out.status, len(cols))
    assert st["error"] == 0, st
    assert st["n_records"] == R
    got = out.results(st)

    # whole-output properties
    for c, t in enumerate(cols):
        if t == "str":
            assert st["chars_len"][c] == info["col_value_bytes"][c], c
            off = got[c][0]
            assert int(off[0]) == 0 and int(off[-1]) == st["chars_len"][c]
            assert bool((off[1:] >= off[:-1]).all()), f"offsets col {c} decrease"

    # sampled windows against the oracle
    wins, k = _windows(R, datagen.seed_of(name))
    for r0 in wins:
        r1 = r0 + k
        b0 = int(roff[r0])
        b1 = int(roff[r1]) if r1 < R else n
        ref, rst = O.csv_parse(data[b0:b1], cols)
        assert rst["error"] == 0 and rst["n_records"] == k, (r0, rst)
        for c, t in enumerate(cols):
            if t == "str":
                off = got[c][0][r0:r1 + 1].cpu().numpy().astype(np.int64)
                ro, rc = ref[c]
                assert np.array_equal(off - off[0], ro), f"offsets col {c} rows {r0}.."
                chars = got[c][1][int(off[0]):int(off[-1])].cpu().numpy()
                assert np.array_equal(chars, rc), f"chars col {c} rows {r0}.."
            elif t == "f64":
                g = got[c][r0:r1].cpu().numpy()
                d = ulp_diff(g, ref[c])
                assert int(d.max()) <= 1, f"f64 col {c} rows {r0}..: {d.max()} ulp"
                assert np.array_equal(np.signbit(g), np.signbit(ref[c]))
            else:
                assert np.array_equal(got[c][r0:r1].cpu().numpy(), ref[c]), \
                    f"col {c} rows {r0}.."


def test_tokenize_full_size():
    name = "json_2gib"
    data, info, _ = datagen.generate(name, record_offsets=True, record_offsets_cap=_roff_cap(name))
    assert info["n_tokens"] > 0
    roff = info["record_offsets"].astype(np.int64)
    n = data.size
    T = info["n_tokens"]
    d_in = _to_device(data)
    ids = torch.empty(T, dtype=torch.uint8, device="cuda")
    starts = torch.empty(T, dtype=torch.int64, device="cuda")
    lens = torch.empty(T, dtype=torch.int32, device="cuda")
    status = pp.new_status()
    stream = torch.cuda.current_stream()
    pp.pp_tokenize(d_in, n, pp.desc_json_lexer(), ids, starts, lens, T, status, stream)
    st = pp.read_status(status)
    assert st["error"] == 0, st
    assert st["n_tokens"] == T

    # whole-output properties
    assert int(starts[0]) == 0
    assert bool((starts[1:] > starts[:-1]).all())
    assert bool((starts[:-1] + lens[:-1].to(torch.int64) == starts[1:]).all())
    assert int(starts[-1]) + int(lens[-1]) == n
    assert bool((ids != 255).all())
    assert int(lens.to(torch.int64).sum()) == n

    # sampled windows of whole top-level values against the oracle; a value
    # starts with '{' after a whitespace run, so it begins a token in the
    # lexer's start context
    cap = _roff_cap(name)
    n_vals = roff.size  # values recorded (all of them when fewer than cap)
    complete = n_vals < cap
    wins, k = _windows(n_vals, datagen.seed_of(name))
    for v0 in wins:
        if v0 + k < n_vals:
            b1 = int(roff[v0 + k])
        elif complete:
            b1 = n  # the input's last values, through to its end
        else:
            continue
        b0 = int(roff[v0])
        (rids, rstarts, rlens), rst = O.tokenize(data[b0:b1])
        assert rst["error"] == 0, (v0, rst)
        t0 = int(torch.searchsorted(starts, torch.tensor([b0], device="cuda")).item())
        m = rids.size
        assert t0 < T and int(starts[t0]) == b0, f"no token starts at value {v0} (byte {b0})"
        assert t0 + m <= T
        g_starts = starts[t0:t0 + m].cpu().numpy() - b0
        assert np.array_equal(g_starts.astype(np.uint64), rstarts), f"starts at value {v0}"
        assert np.array_equal(lens[t0:t0 + m].cpu().numpy().astype(np.uint32), rlens)
        assert np.array_equal(ids[t0:t0 + m].cpu().numpy(), rids)
        if t0 + m < T:
            assert int(starts[t0 + m]) == b1
        else:
            assert b1 == n
