"""f4: the fixed-width numeral grid converted back to the target's text format (VFlash paper (zh) §2.3).

The library's host function (fpd_grid_to_text) against the oracle's restatement on random grids, and the oracle
pinned to the worked fields of tests/golden/fixed_width_fields.txt and to hand-written blocks.  No GPU needed."""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fixed_width_fields.txt")
V = 151936
LAY = synth.layout_fixed_width(V)
DIGITS = list(range(1000, 1010))
PLUS, MINUS, SEP, PAD = 1010, 1011, 1012, V - 1


@pytest.fixture(scope="module")
def fpd():
    import __graft_entry__ as g
    g._compile_all()
    import block_diffusion_speculative_non_gb300 as pkg
    return pkg


def _field_tokens(text):
    """'+PP012' -> token ids (P = pad / mask)."""
    m = {"+": PLUS, "-": MINUS, "P": PAD}
    return [m[c] if c in m else DIGITS[int(c)] if c.isdigit() else 5 for c in text]


def test_oracle_field_values_match_the_worked_fields(oracle_lib):
    n = 0
    for ln in open(GOLDEN):
        if ln.startswith("#") or not ln.strip():
            continue
        field, valid, _, value = ln.split()
        v = oracle_lib.grid_field_value(_field_tokens(field), DIGITS, PLUS, MINUS, PAD)
        assert (v is not None) == (valid == "1"), field
        if v is not None:
            assert v == int(value), field
        n += 1
    assert n >= 10


def _block(fields_per_wp, n_wp=20):
    """A committed row (block positions 1..L-1) from per-waypoint field strings; missing waypoints are zeros."""
    L = LAY["block_len"]
    row = []
    for w in range(n_wp):
        fs = fields_per_wp[w] if w < len(fields_per_wp) else ["+PPPP0"] * 3
        for f in fs:
            row += _field_tokens(f)
        row.append(SEP)
    row = row[:L - 1] + [-1]
    assert len(row) == L
    return np.array(row, np.int32)


def test_oracle_hand_written_blocks(oracle_lib):
    """Expected strings written by hand from the rule: values without leading zeros, '-' only when negative,
    axes joined by ',', waypoints by ';', complete waypoints inside the accepted prefix, stop at a bad field."""
    per_wp = 3 * 6 + 1
    a = _block([["+PP012", "-PPPP7", "+00000"], ["+P1234", "-98765", "+PPP40"]])
    b = _block([["+PP012", "+4PP42", "+00001"], ["+P1234", "-98765", "+PPP40"]])   # second field malformed
    c = _block([["-PPPP0", "+PPPP9", "+PPPP9"]])
    texts = oracle_lib.grid_to_text(np.stack([a, a, a, b, c]), [2 * per_wp, per_wp + 17, per_wp - 1, 2 * per_wp, 18],
                                    DIGITS, PLUS, MINUS, PAD)
    assert texts == ["12,-7,0;1234,-98765,40", "12,-7,0", "12,-7,0", "", "0,9,9"]


def _random_rows(rng, B):
    L = LAY["block_len"]
    rows = np.empty((B, L), np.int32)
    for b in range(B):
        row = []
        for w in range(20):
            for a in range(3):
                v = int(rng.integers(-99999, 100000))
                s = str(abs(v))
                width = len(s) + int(rng.integers(0, 6 - len(s)))   # leading zeros sometimes
                digits = s.rjust(width, "0").rjust(5, "P")
                row += _field_tokens(("-" if v < 0 else "+") + digits)
            row.append(SEP)
        row = row[:L - 1] + [-1]
        for _ in range(int(rng.integers(0, 3))):   # corrupt a few slots
            row[int(rng.integers(0, L - 1))] = int(rng.choice([PAD, PLUS, MINUS, 7, DIGITS[3]]))
        rows[b] = row
    return rows


def test_library_matches_oracle_on_random_grids(fpd, oracle_lib):
    rng = np.random.default_rng(404)
    B = 400
    rows = _random_rows(rng, B)
    acc = rng.integers(0, LAY["block_len"], size=B).astype(np.int32)
    fmt = fpd.grid_format(DIGITS, PLUS, MINUS, PAD)
    got = fpd.fpd_grid_to_text(rows, acc, fmt)
    want = oracle_lib.grid_to_text(rows, acc, DIGITS, PLUS, MINUS, PAD)
    assert got == want
    assert sum(len(t) > 0 for t in got) > B // 4   # the sample is not all empty


def test_library_reports_a_short_buffer(fpd):
    import ctypes
    rows = _random_rows(np.random.default_rng(5), 2)
    fmt = fpd.grid_format(DIGITS, PLUS, MINUS, PAD)
    buf = ctypes.create_string_buffer(8)
    offs = (ctypes.c_size_t * 3)()
    acc = np.full(2, LAY["block_len"] - 1, np.int32)
    st = fpd.lib().fpd_grid_to_text(2, LAY["block_len"], rows.ctypes.data, acc.ctypes.data, ctypes.byref(fmt), buf, 8,
                                    offs)
    assert st == 3
