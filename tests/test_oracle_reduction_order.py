"""The canonical order of the RMS sum of squares, pinned bit for bit.

`tests/golden/rstd_order.txt` holds rows derived by hand on the binary32 grid
(each derivation is written beside its row): for each, the sum of squares `ss`
in the documented order and, where it follows in closed form, the rstd.  The
oracle's single sum-of-squares routine must give exactly those bits through
every way it is reached: bf16 rows (the AdaLN producer), fp32 rows (the
residual fold) and heads (the QKV epilogue).

Each row also names the slips it separates: plausible mis-readings of the
order (a sequential sum, the 32-lane order of an earlier draft, groups added
in sequence, a reversed butterfly, ...).  The slips are written out here as
small variations of a restatement of the documented order; the tests check
that each named slip gives a different ss (and rstd, where the row lists one)
on its row, and that every slip is named by some row.  So a mistake of any of
these kinds in the oracle, or in a kernel compared with it, changes bits that
the hand-derived rows fix.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import golden_lines

F32 = np.float32


# --------------------------------------------------------------------------- #
# the hand-derived rows                                                         #
# --------------------------------------------------------------------------- #

def _bits(h: str) -> int:
    return int(h, 16)


def _f32_of(bits: int) -> F32:
    return np.array([bits], np.uint32).view(np.float32)[0]


def _bf16_value(bits: int) -> F32:
    return _f32_of(bits << 16)


def _load():
    records, cur = [], None
    for line in golden_lines("rstd_order.txt"):
        tok = line.split()
        if tok[0] in ("row", "head", "f32row"):
            n = int(tok[3])
            cur = {"kind": tok[0], "name": tok[1], "n": n, "eps": _f32_of(_bits(tok[5])),
                   "values": np.zeros(n, np.float32), "bf16": np.zeros(n, np.uint16),
                   "rstd": None, "slips": []}
            records.append(cur)
        elif tok[0] == "set":
            for col in tok[2:]:
                cur["bf16"][int(col)] = _bits(tok[1])
                cur["values"][int(col)] = _bf16_value(_bits(tok[1]))
        elif tok[0] == "set32":
            for col in tok[2:]:
                cur["values"][int(col)] = _f32_of(_bits(tok[1]))
        elif tok[0] == "ss":
            cur["ss"] = _bits(tok[1])
        elif tok[0] == "rstd":
            cur["rstd"] = _bits(tok[1])
        elif tok[0] == "slips":
            cur["slips"] = tok[1:]
        else:
            raise ValueError(f"unknown line in rstd_order.txt: {line}")
    return records


RECORDS = _load()


def _u32(x) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def _lanes(rec) -> int:
    return rec["n"] // 8 if rec["kind"] == "head" else 128


@pytest.mark.parametrize("rec", RECORDS, ids=[r["name"] for r in RECORDS])
def test_oracle_sum_of_squares_is_the_hand_derived_one(rec):
    ss = oracle.sumsq_f32(rec["values"], _lanes(rec))
    assert _u32(ss) == rec["ss"], f"{rec['name']}: ss {_u32(ss):#010x} != {rec['ss']:#010x}"
    if rec["kind"] == "row":
        assert _u32(oracle.sumsq_bf16(rec["bf16"])) == rec["ss"]


@pytest.mark.parametrize("rec", [r for r in RECORDS if r["rstd"] is not None],
                         ids=[r["name"] for r in RECORDS if r["rstd"] is not None])
def test_oracle_rstd_is_the_hand_derived_one(rec):
    eps = float(rec["eps"])
    if rec["kind"] == "head":
        got = [oracle.head_rstd(rec["values"], eps)]
    else:
        n = rec["n"]
        x = rec["bf16"][None, :]
        gamma = np.full(n, 0x3F80, np.uint16)                 # 1.0
        table = np.zeros((1, 2, n), np.uint16)
        got = [oracle.row_rstd(rec["bf16"], eps), oracle.row_rstd_f32(rec["values"], eps),
               oracle.adaln_rows(x, gamma, table, [0], eps, None)[2][0],
               # the residual fold with o = 0 leaves h as it is, so its rstd is the row's
               oracle.residual_adaln_rows(rec["values"][None, :], np.zeros((1, n), np.uint16), None,
                                          np.zeros((1, n), np.uint16), gamma, table, [0], eps, None)[3][0]]
    for g in got:
        assert _u32(g) == rec["rstd"], f"{rec['name']}: rstd {_u32(g):#010x} != {rec['rstd']:#010x}"


def test_fp32_row_sum_reaches_the_residual_fold():
    rec = next(r for r in RECORDS if r["kind"] == "f32row")
    n = rec["n"]
    gamma = np.full(n, 0x3F80, np.uint16)
    table = np.zeros((1, 2, n), np.uint16)
    eps = float(rec["eps"])
    rstd = oracle.residual_adaln_rows(rec["values"][None, :], np.zeros((1, n), np.uint16), None,
                                      np.zeros((1, n), np.uint16), gamma, table, [0], eps, None)[3][0]
    assert _u32(rstd) == _u32(oracle.row_rstd_f32(rec["values"], eps))
    assert _u32(rstd) == _u32(_rstd_of(_f32_of(rec["ss"]), n, rec["eps"]))


# --------------------------------------------------------------------------- #
# the slips                                                                     #
# --------------------------------------------------------------------------- #

def _round_f32(q: Fraction) -> F32:
    """An exact rational rounded to binary32, to nearest, ties to even (normal range)."""
    if q == 0:
        return F32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    scaled = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return F32(sign * float(Fraction(m) * Fraction(2) ** (e - 23)))


def _fma(x, p) -> F32:
    """fmaf(x, x, p): one rounding of x*x + p."""
    x, p = F32(x), F32(p)
    if x == 0:
        return p
    xx = np.float64(x) * np.float64(x)             # exact in binary64
    if np.float64(F32(xx)) == xx:                   # exact in binary32 too (bf16 inputs)
        return F32(F32(xx) + p)
    return _round_f32(Fraction(float(x)) ** 2 + Fraction(float(p)))


def _square_then_add(x, p) -> F32:
    return F32(F32(F32(x) * F32(x)) + F32(p))


def _partials(v, chunks, step=_fma):
    p = [F32(0.0)] * 8
    for c in chunks:
        for e in range(8):
            p[e] = step(v[8 * c + e], p[e])
    return p


def _pairwise(p):
    return F32(F32(F32(p[0] + p[1]) + F32(p[2] + p[3])) + F32(F32(p[4] + p[5]) + F32(p[6] + p[7])))


def _butterfly(t, distances):
    t = list(t)
    for o in distances:
        t = [F32(t[l] + t[l ^ o]) for l in range(len(t))]
    return t[0]


def _down(width):
    return [width >> k for k in range(1, width.bit_length()) if width >> k >= 1]


def _restated(v, lanes, *, lane_chunks=None, lane_total=_pairwise, distances=None,
              combine=None, step=_fma):
    """The documented order, written out again; keyword arguments swap one part."""
    chunks = len(v) // 8
    if lane_chunks is None:
        lane_chunks = lambda l: range(l, chunks, lanes)           # noqa: E731
    totals = [lane_total(_partials(v, lane_chunks(l), step)) for l in range(lanes)]
    width = min(lanes, 32)
    dist = _down(width) if distances is None else distances(width)
    groups = [_butterfly(totals[w * width:(w + 1) * width], dist) for w in range(lanes // width)]
    if len(groups) == 1:
        return groups[0]
    if combine is not None:
        return combine(groups)
    return F32(F32(groups[0] + groups[1]) + F32(groups[2] + groups[3]))


def _sequential(v, lanes):
    p = F32(0.0)
    for x in v:
        p = _fma(x, p)
    return p


def _one_partial(v, lanes_used, chunks_per_lane):
    def total(l):
        p = F32(0.0)
        for c in chunks_per_lane(l):
            for e in range(8):
                p = _fma(v[8 * c + e], p)
        return p
    return [total(l) for l in range(lanes_used)]


def _survey_32_lanes(v, lanes):
    chunks = len(v) // 8
    return _butterfly(_one_partial(v, 32, lambda l: range(l, chunks, 32)), [16, 8, 4, 2, 1])


def _partials_on_32_lanes(v, lanes):
    chunks = len(v) // 8
    totals = [_pairwise(_partials(v, range(l, chunks, 32))) for l in range(32)]
    return _butterfly(totals, [16, 8, 4, 2, 1])


def _one_partial_128(v, lanes):
    chunks = len(v) // 8
    totals = _one_partial(v, 128, lambda l: range(l, chunks, 128))
    g = [_butterfly(totals[32 * w:32 * w + 32], [16, 8, 4, 2, 1]) for w in range(4)]
    return F32(F32(g[0] + g[1]) + F32(g[2] + g[3]))


def _butterfly_128(v, lanes):
    chunks = len(v) // 8
    totals = [_pairwise(_partials(v, range(l, chunks, 128))) for l in range(128)]
    return _butterfly(totals, [64, 32, 16, 8, 4, 2, 1])


def _sum_in_sequence(p):
    acc = F32(0.0)
    for x in p:
        acc = F32(acc + x)
    return acc


SLIPS = {
    "sequential": _sequential,
    "survey_32_lanes": _survey_32_lanes,
    "partials_on_32_lanes": _partials_on_32_lanes,
    "one_partial_128": _one_partial_128,
    "butterfly_128": _butterfly_128,
    "groups_in_sequence": lambda v, lanes: _restated(
        v, lanes, combine=lambda g: F32(F32(F32(g[0] + g[1]) + g[2]) + g[3])),
    "groups_crossed": lambda v, lanes: _restated(
        v, lanes, combine=lambda g: F32(F32(g[0] + g[2]) + F32(g[1] + g[3]))),
    "butterfly_reversed": lambda v, lanes: _restated(
        v, lanes, distances=lambda w: list(reversed(_down(w)))),
    "partials_in_sequence": lambda v, lanes: _restated(v, lanes, lane_total=_sum_in_sequence),
    "partials_crossed": lambda v, lanes: _restated(
        v, lanes, lane_total=lambda p: F32(F32(F32(p[0] + p[4]) + F32(p[1] + p[5])) +
                                           F32(F32(p[2] + p[6]) + F32(p[3] + p[7])))),
    "chunks_blocked": lambda v, lanes: _restated(
        v, lanes, lane_chunks=lambda l: range(l * (len(v) // 8 // lanes), (l + 1) * (len(v) // 8 // lanes))),
    "chunks_decreasing": lambda v, lanes: _restated(
        v, lanes, lane_chunks=lambda l: reversed(range(l, len(v) // 8, lanes))),
    "square_rounded_first": lambda v, lanes: _restated(v, lanes, step=_square_then_add),
}


def _rstd_of(ss, n, eps):
    return F32(F32(1.0) / F32(np.sqrt(F32(F32(F32(ss) / F32(n)) + F32(eps)))))


@pytest.mark.parametrize("rec", RECORDS, ids=[r["name"] for r in RECORDS])
def test_restated_order_is_the_oracle_on_the_row(rec):
    """The restatement the slips are built from gives the hand-derived bits too."""
    assert _u32(_restated(rec["values"], _lanes(rec))) == rec["ss"]


@pytest.mark.parametrize("rec", RECORDS, ids=[r["name"] for r in RECORDS])
def test_each_row_separates_the_slips_it_names(rec):
    assert rec["slips"], f"{rec['name']} names no slip"
    for name in rec["slips"]:
        ss = SLIPS[name](rec["values"], _lanes(rec))
        assert _u32(ss) != rec["ss"], f"{rec['name']}: slip {name} gives the documented ss"
        if rec["rstd"] is not None:
            r = _rstd_of(ss, rec["n"], rec["eps"])
            assert _u32(r) != rec["rstd"], f"{rec['name']}: slip {name} gives the documented rstd"


def test_every_slip_is_named_by_some_row():
    named = {s for r in RECORDS for s in r["slips"]}
    assert named == set(SLIPS), f"unnamed: {set(SLIPS) - named}; unknown: {named - set(SLIPS)}"


@pytest.mark.parametrize("cols", [256, 1024, 4096])
def test_restated_order_is_the_oracle_on_random_rows(cols):
    """On dense random rows the restatement and the oracle agree as well, so each
    slip differs from the documented order in the one part its name says."""
    rng = np.random.default_rng(cols)
    for _ in range(3):
        x = (rng.standard_normal(cols) * np.exp(rng.standard_normal(cols))).astype(np.float32)
        bf = oracle.bf16_bits(x)
        v = (bf.astype(np.uint32) << 16).view(np.float32)
        assert _u32(_restated(v, 128)) == _u32(oracle.sumsq_bf16(bf))
    for hd in (64, 128, 256):
        v = oracle.bf16_value(oracle.bf16_bits(rng.standard_normal(hd).astype(np.float32) * 3))
        assert _u32(_restated(v, hd // 8)) == _u32(oracle.sumsq_f32(v, hd // 8))
