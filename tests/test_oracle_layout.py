"""Pins of the oracle's m16n8k16 accumulator map against the values printed
on the page that derives it (digit ranges, place values, span, the two stated
steps) and against the bijection argument made there."""
import os

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "acc_fragment_numeral.txt")


def _golden():
    digits, steps, span = {}, {}, None
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        parts = line.split()
        if parts[0] == "span":
            span = int(parts[1])
        elif parts[0] == "step":
            steps[parts[1]] = (int(parts[3]), int(parts[5]))
        else:
            digits[parts[0]] = (int(parts[1]), int(parts[2]))
    return digits, steps, span


def _digit_values(lane, j):
    return {"j&1": j & 1, "tig": lane % 4, "group": lane // 4, "j>>1": j >> 1}


def test_numeral_equals_row_col_form(orc):
    digits, _, _ = _golden()
    for lane in range(32):
        for j in range(4):
            r, c = orc.acc_coords(lane, j)
            vals = _digit_values(lane, j)
            for name, (rng, _) in digits.items():
                assert 0 <= vals[name] < rng
            numeral = sum(vals[name] * place for name, (_, place) in digits.items())
            assert r * 8 + c == numeral


def test_place_values_are_running_products_and_span(orc):
    digits, _, span = _golden()
    order = sorted(digits.items(), key=lambda kv: kv[1][1])
    running = 1
    for _, (rng, place) in order:
        assert place == running
        running *= rng
    assert running == span == 16 * 8


def test_bijection_by_ownership_map(orc):
    owner = [[None] * 8 for _ in range(16)]
    for lane in range(32):
        for j in range(4):
            r, c = orc.acc_coords(lane, j)
            assert 0 <= r < 16 and 0 <= c < 8
            assert owner[r][c] is None, "overlap"
            owner[r][c] = (lane, j)
    assert all(o is not None for row in owner for o in row), "gap"


def test_fragment_index_split_steps(orc):
    _, steps, _ = _golden()
    for lane in range(32):
        r0, c0 = orc.acc_coords(lane, 0)
        r1, c1 = orc.acc_coords(lane, 1)
        r2, c2 = orc.acc_coords(lane, 2)
        assert (r1 - r0, c1 - c0) == steps["j0->j1"]
        assert (r2 - r0, c2 - c0) == steps["j0->j2"]


def test_out_of_range_rejected(orc):
    import pytest
    for lane, j in ((-1, 0), (32, 0), (0, -1), (0, 4)):
        with pytest.raises(ValueError):
            orc.acc_coords(lane, j)
