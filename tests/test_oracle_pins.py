"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.

Each pin is written as a function over an oracle-like object so that the same
battery can be run against deliberately wrong restatements (``test_mutants``):
every plausible mistake there must fail at least one pin.

Pages: geek-doc.cn "并行前缀和 scan: Hillis-Steele、Blelloch 与 warp shuffle
三种写法" (sections 一 to 五), lpnh.cn/news/2866224 "并行扫描 Scan/Prefix Sum"
(sections 2.1, 3.3, 4.1), pgsm.cn/news/414823 "SIMT数据依赖与并行前缀和"
(sections 2.2, 4.1-4.2).
"""
import math
import types
from fractions import Fraction
from functools import reduce

import numpy as np
import pytest

import oracle
from oracle import prior_art

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

MASK32 = 0xFFFFFFFF


# --------------------------------------------------------------------------
# independent helpers (Python integers, no oracle code)
# --------------------------------------------------------------------------
def _py_op(op, dtype):
    signed = np.dtype(dtype) == np.int32

    def to_s(v):
        v &= MASK32
        return v - (1 << 32) if (signed and v >= 1 << 31) else v

    if op == "add":
        return lambda a, b: to_s(a + b)
    if op == "xor":
        return lambda a, b: to_s((a & MASK32) ^ (b & MASK32))
    return lambda a, b: a if a >= b else b


def _brute_prefix(x, op, dtype, inclusive):
    """O(n^2): every prefix folded from scratch."""
    f = _py_op(op, dtype)
    ident = oracle.identity(op, dtype)
    vals = [int(v) for v in x]
    out = []
    for i in range(len(vals)):
        seg = vals[:i + 1] if inclusive else vals[:i]
        out.append(reduce(f, seg, ident))
    return out


# --------------------------------------------------------------------------
# the pin battery
# --------------------------------------------------------------------------
def pin_worked_example(o, golden):
    g = golden("worked_example.txt")
    x = np.array(g["x"], dtype=np.int32)
    assert o.scan(x, "add", True).tolist() == g["inclusive"]
    assert o.scan(x, "add", False).tolist() == g["exclusive"]
    flags = (x > g["predicate_threshold"][0]).astype(np.uint8)
    assert flags.tolist() == g["flags"]
    assert o.scan(flags.astype(np.int32), "add", False).tolist() == g["flag_positions"]
    assert o.compact(x, flags).tolist() == g["compacted"]


def pin_brute_force(o, golden):
    rng = np.random.default_rng(1234)
    for dtype in (np.int32, np.uint32):
        for op in ("add", "max", "xor"):
            for n in list(range(0, 65)):
                if op == "add":
                    x = rng.integers(-50 if dtype == np.int32 else 0, 50, n).astype(dtype)
                elif dtype == np.int32:
                    x = rng.integers(-2**31, 2**31, n, dtype=np.int32)
                else:
                    x = rng.integers(0, 2**32, n, dtype=np.uint32)
                for inclusive in (True, False):
                    got = [int(v) for v in o.scan(x, op, inclusive)]
                    assert got == _brute_prefix(x, op, dtype, inclusive), (dtype, op, n, inclusive)


def pin_relation(o, golden):
    """P1 section 一: y[i] = z[i+1]; z[0] is the identity; y[n-1] is the total."""
    rng = np.random.default_rng(99)
    for dtype in (np.int32, np.uint32, np.float32):
        for op in ("add", "max", "xor"):
            if dtype == np.float32 and op == "xor":
                continue
            x = (rng.random(5000).astype(np.float32) if dtype == np.float32
                 else rng.integers(0, 2**31 - 1, 5000).astype(dtype))
            y = o.scan(x, op, True)
            z = o.scan(x, op, False)
            assert np.array_equal(y[:-1], z[1:])
            assert z[0] == oracle.identity(op, dtype)


def pin_closed_forms(o, golden):
    n = 100_000
    ones = np.ones(n, dtype=np.int32)
    assert np.array_equal(o.scan(ones, "add", True), np.arange(1, n + 1, dtype=np.int32))
    ar = np.arange(n, dtype=np.uint32)
    tri = [(i * (i + 1) // 2) & MASK32 for i in range(n)]
    assert o.scan(ar, "add", True).tolist() == tri
    # xor of 0..i: i, 1, i+1, 0 for i mod 4 = 0, 1, 2, 3
    cf = [(i, 1, i + 1, 0)[i % 4] for i in range(n)]
    assert o.scan(ar, "xor", True).tolist() == cf
    asc = np.arange(-5000, 5000, dtype=np.int32)
    assert np.array_equal(o.scan(asc, "max", True), asc)
    desc = asc[::-1].copy()
    assert np.all(o.scan(desc, "max", True) == desc[0])
    big = np.array([2**31 - 1, 1], dtype=np.int32)
    assert o.scan(big, "add", True).tolist() == [2**31 - 1, -2**31]


def pin_identities(o, golden):
    x = np.array([5, -7, 3], dtype=np.int32)
    assert int(o.scan(x, "max", False)[0]) == -2**31
    assert int(o.scan(x.astype(np.uint32), "max", False)[0]) == 0
    assert float(o.scan(x.astype(np.float32), "max", False)[0]) == -math.inf
    assert o.scan(np.array([-3, -9, -1], dtype=np.int32), "max", True).tolist() == [-3, -3, -1]


def pin_f32_exact(o, golden):
    """fp32 add, accumulated in fp64, against exact rational prefix sums: the
    only error allowed is fp64 accumulation, |err| <= n * 2^-53 * sum|x|."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(3000) * 100).astype(np.float32)
    y = o.scan(x, "add", True)
    z = o.scan(x, "add", False)
    exact = Fraction(0)
    absum = Fraction(0)
    for i, v in enumerate(x.tolist()):
        assert abs(Fraction(float(z[i])) - exact) <= (i + 1) * Fraction(1, 2**53) * max(absum, Fraction(1, 2**60))
        exact += Fraction(v)
        absum += abs(Fraction(v))
        assert abs(Fraction(float(y[i])) - exact) <= (i + 1) * Fraction(1, 2**53) * absum
    # fp32 max is exact: NumPy's running maximum is an independent routine
    assert np.array_equal(o.scan(x, "max", True), np.maximum.accumulate(x).astype(np.float64))
    # the tolerance scale is the fp64 running sum of |x|
    s = o.abs_prefix(x)
    assert abs(s[-1] - math.fsum(abs(float(v)) for v in x)) <= 1e-9 * s[-1]


def pin_compaction(o, golden):
    """lpnh.cn section 4.1 / pgsm.cn section 4.1: keep flagged elements in
    order; count = number kept.  Any nonzero flag keeps its element."""
    rng = np.random.default_rng(11)
    for n in (0, 1, 2, 17, 1000, 65537):
        v = rng.integers(-2**31, 2**31, n, dtype=np.int32)
        f = rng.integers(0, 4, n).astype(np.uint8)  # 0 drops; 1, 2, 3 keep
        got = o.compact(v, f)
        assert got.tolist() == [int(a) for a, b in zip(v, f) if b != 0]
        assert got.size == int(np.count_nonzero(f))
        # the scan construction (exclusive scan of the 0/1 predicate gives
        # each kept element its output slot) agrees
        pos = o.scan((f != 0).astype(np.int32), "add", False)
        out = np.zeros(got.size, dtype=np.int32)
        out[pos[f != 0]] = v[f != 0]
        assert np.array_equal(out, got)


def pin_split(o, golden):
    """geek-doc.cn section 一 (radix sort): zeros of the bit first, ones
    after, each group in input order."""
    rng = np.random.default_rng(13)
    for n in (0, 1, 5, 333, 4096):
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        for bit in (0, 1, 7, 16, 30, 31):
            got, zeros = o.split_bit(k, bit)
            want = sorted(k.tolist(), key=lambda v: (v >> bit) & 1)  # Python sort is stable
            assert got.tolist() == want
            assert zeros == sum(1 for v in k.tolist() if not (v >> bit) & 1)


def pin_sort(o, golden):
    rng = np.random.default_rng(17)
    for n in (0, 1, 2, 1000, 50_000):
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        if n > 10:
            k[:10] = [0, 2**32 - 1, 5, 5, 5, 2**31, 2**31 - 1, 0, 1, 2**32 - 1]
        assert np.array_equal(o.sort_lsd(k), np.sort(k))


def _fold_py(vals, op, dtype):
    """Direct fold in Python integers / fractions (independent of the C
    oracle): add wraps modulo 2^32 for the integer types."""
    if dtype == np.float32:
        if op == "add":
            return float(sum(Fraction(float(v)) for v in vals))
        return float(max((float(v) for v in vals), default=float("-inf")))
    if op == "add":
        r = sum(int(v) for v in vals) % 2**32
    elif op == "xor":
        r = reduce(lambda a, b: a ^ b, (int(v) % 2**32 for v in vals), 0)
    else:
        r = max((int(v) for v in vals), default=(-2**31 if dtype == np.int32 else 0))
        r %= 2**32
    if dtype == np.int32 and r >= 2**31:
        r -= 2**32
    return r


def pin_segmented(o, golden):
    """lpnh.cn section 7.2 (segmented scan): a head restarts the fold at the
    identity.  Pinned by the hand-worked fixture, the two degenerate flag
    patterns, brute-force folds of each element's own segment, and the
    concatenation of plain scans of the segments."""
    g = golden("segmented.txt")
    x = np.array(g["x"], dtype=np.int32)
    h = np.array(g["heads"], dtype=np.uint8)
    assert o.segscan(x, h, "add", True).tolist() == g["inclusive"]
    assert o.segscan(x, h, "add", False).tolist() == g["exclusive"]
    assert o.segscan(x, h, "max", True).tolist() == g["max_inclusive"]
    h0 = np.array(g["heads_no_first"], dtype=np.uint8)
    assert o.segscan(x, h0, "add", True).tolist() == g["inclusive"]
    rng = np.random.default_rng(17)
    for dtype in (np.int32, np.uint32, np.float32):
        for op in ("add", "max", "xor"):
            if dtype == np.float32 and op == "xor":
                continue
            for n in (1, 2, 7, 33, 64):
                if dtype == np.float32:
                    xs = rng.integers(-50, 50, n).astype(np.float32)   # exact in fp64
                elif dtype == np.int32:
                    xs = rng.integers(-2**31, 2**31, n, dtype=np.int64).astype(np.int32)
                else:
                    xs = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
                hs = (rng.random(n) < 0.3).astype(np.uint8)
                for inclusive in (True, False):
                    got = o.segscan(xs, hs, op, inclusive)
                    for i in range(n):
                        start = max([j for j in range(i + 1) if hs[j]] + [0])
                        seg = xs[start:i + 1] if inclusive else xs[start:i]
                        assert got[i] == _fold_py(seg, op, dtype), (dtype, op, inclusive, n, i)
                # no heads: the plain scan; a head everywhere: x itself / the identity
                assert np.array_equal(o.segscan(xs, np.zeros(n, np.uint8), op, True), o.scan(xs, op, True))
                ones = np.ones(n, np.uint8)
                assert np.array_equal(o.segscan(xs, ones, op, True).astype(np.float64), xs.astype(np.float64))
                ident = o.identity(op, dtype)
                assert np.all(o.segscan(xs, ones, op, False) == ident)
    # concatenation of independent plain scans, on a longer array
    xs = rng.integers(-1000, 1000, 5000).astype(np.int32)
    hs = (rng.random(5000) < 0.01).astype(np.uint8)
    starts = [0] + [int(j) for j in np.nonzero(hs)[0] if j > 0] + [5000]
    for inclusive in (True, False):
        parts = [o.scan(xs[a:b], "add", inclusive) for a, b in zip(starts[:-1], starts[1:])]
        assert np.array_equal(o.segscan(xs, hs, "add", inclusive), np.concatenate(parts))
    # the fp32 tolerance scale restarts with the segments too
    xf = rng.standard_normal(300).astype(np.float32)
    hf = (rng.random(300) < 0.05).astype(np.uint8)
    s = o.seg_abs_prefix(xf, hf)
    for i in (0, 17, 150, 299):
        start = max([j for j in range(i + 1) if hf[j]] + [0])
        assert math.isclose(s[i], float(sum(Fraction(abs(float(v))) for v in xf[start:i + 1])), rel_tol=1e-15)


def pin_brackets(o, golden):
    """geek-doc.cn section 一: '(' = +1, ')' = -1; a negative prefix means a
    surplus ')', a nonzero total means unbalanced."""
    cases = {"(()": (False, True), "())(": (True, False), "(())": (False, False),
             "": (False, False), ")(": (True, False), "()()((": (False, True)}
    for s, want in cases.items():
        x = np.array([1 if c == "(" else -1 for c in s], dtype=np.int32)
        assert o.bracket_flags(o.scan(x, "add", True)) == want, s
    # exhaustive: among the 2^L sequences of L brackets exactly the Catalan
    # number C_{L/2} are balanced (Dyck words), and none when L is odd
    catalan = {0: 1, 2: 1, 4: 2, 6: 5, 8: 14, 10: 42, 12: 132}
    for length in range(13):
        balanced = 0
        for code in range(1 << length):
            x = np.array([1 if (code >> i) & 1 else -1 for i in range(length)], dtype=np.int32)
            balanced += o.bracket_flags(o.scan(x, "add", True)) == (False, False)
        assert balanced == catalan.get(length, 0), length


PINS = [pin_worked_example, pin_brute_force, pin_relation, pin_closed_forms,
        pin_identities, pin_f32_exact, pin_compaction, pin_split, pin_sort,
        pin_brackets, pin_segmented]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, golden):
    pin(oracle, golden)


def test_xor_rejected_on_f32():
    with pytest.raises(ValueError):
        oracle.scan(np.ones(4, dtype=np.float32), "xor", True)


# --------------------------------------------------------------------------
# the prior-art restatements against the pages' printed traces
# --------------------------------------------------------------------------
def test_hillis_steele_trace(golden):
    g = golden("hillis_steele.txt")
    res, steps, _ = prior_art.hillis_steele(g["x"])
    assert steps[0] == g["step1"]
    assert steps[2] == g["step3"] == res
    # the window rule: after step k cell i holds the sum of inputs
    # max(0, i - 2^(k+1) + 1) .. i
    for k, st in enumerate(steps):
        w = 2 ** (k + 1)
        assert st == [sum(g["x"][max(0, i - w + 1):i + 1]) for i in range(len(g["x"]))]
    # the page's printed second step is a misprint in exactly two cells
    bad = [i for i, (a, b) in enumerate(zip(steps[1], g["step2_printed"])) if a != b]
    assert bad == g["misprinted_cells"]
    assert oracle.scan(np.array(g["x"], dtype=np.int32), "add", True).tolist() == res


def test_blelloch_trace(golden):
    g = golden("blelloch.txt")
    excl, ups, downs, ops, steps, total = prior_art.blelloch(g["x"])
    assert excl == g["exclusive"]
    assert downs[0][3] == g["first_down_level_left_node"][0]
    assert downs[0][7] == g["first_down_level_right_node"][0]
    n = len(g["x"])
    assert ops == g["total_adds"][0] == 2 * n - 2
    assert sum(1 for a, b in zip(ups[-1], g["x"]) if a != b) <= g["upsweep_adds"][0]
    assert steps == g["steps"][0]
    assert total == sum(g["x"])


def test_three_phase_example(golden):
    g = golden("multiblock.txt")
    out, totals, offsets, locs = prior_art.three_phase(g["x"], g["block"][0])
    assert totals == g["totals"] and offsets == g["offsets"]
    assert locs[1] == g["block1_local_exclusive"]
    assert out[4:] == g["block1_global"]
    assert out == oracle.scan(np.array(g["x"], dtype=np.int32), "add", False).tolist()


def test_op_count_table(golden):
    g = golden("op_counts.txt")
    n = g["n"][0]
    assert n - 1 == g["serial_adds"][0]
    _, hs_steps, hs_ops = prior_art.hillis_steele(list(range(n)))
    assert len(hs_steps) == g["hillis_steele_steps"][0]
    # "about N log2 N": exactly N log2 N - (N - 1) once the idle left edge is skipped
    assert hs_ops == n * int(math.log2(n)) - (n - 1)
    assert abs(hs_ops - g["hillis_steele_adds_about"][0]) < 0.15 * g["hillis_steele_adds_about"][0]
    _, _, _, b_ops, b_steps, _ = prior_art.blelloch([1] * n)
    assert b_steps == g["blelloch_steps"][0] and b_ops == g["blelloch_adds"][0]
    _, unguarded_ops = prior_art.warp_shuffle_scan([1] * 32, guarded=False)
    assert unguarded_ops == g["warp_shuffle_adds"][0]
    assert int(math.log2(32)) == g["warp_steps"][0]


def test_warp_shuffle_guard():
    """The shuffle-up scan is only a scan when lanes without a source skip
    the combine (pgsm.cn section 2.2: such lanes get their own value back)."""
    rng = np.random.default_rng(3)
    x = rng.integers(0, 100, 32).tolist()
    good, _ = prior_art.warp_shuffle_scan(x, guarded=True)
    bad, _ = prior_art.warp_shuffle_scan(x, guarded=False)
    assert good == oracle.scan(np.array(x, dtype=np.int32), "add", True).tolist()
    assert bad != good and bad[0] == 32 * x[0]


def test_restatements_agree_on_random():
    rng = np.random.default_rng(5)
    for n in (1, 2, 3, 64, 100, 256):
        x = rng.integers(0, 1000, n).tolist()
        ref = oracle.scan(np.array(x, dtype=np.int32), "add", True).tolist()
        assert prior_art.hillis_steele(x)[0] == ref
        ex = oracle.scan(np.array(x, dtype=np.int32), "add", False).tolist()
        assert prior_art.three_phase(x, 7)[0] == ex
        if n & (n - 1) == 0:
            assert prior_art.blelloch(x)[0] == ex


# --------------------------------------------------------------------------
# planted mistakes: each wrong restatement must fail at least one pin
# --------------------------------------------------------------------------
def _mutant(**over):
    base = {name: getattr(oracle, name) for name in
            ("scan", "compact", "split_bit", "sort_lsd", "bracket_flags", "abs_prefix", "segscan",
             "seg_abs_prefix", "identity")}
    base.update(over)
    return types.SimpleNamespace(**base)


def _swap_incl_excl(x, op="add", inclusive=True):
    return oracle.scan(x, op, not inclusive)


def _excl_zero_identity(x, op="add", inclusive=True):
    y = oracle.scan(x, op, inclusive)
    if not inclusive and y.size:
        y = y.copy()
        y[0] = 0
    return y


def _drop_last_term(x, op="add", inclusive=True):
    x = np.asarray(x).copy()
    if x.size > 3:
        x[-1] = oracle.identity(op, x.dtype) if op != "add" else 0
    return oracle.scan(x, op, inclusive)


def _no_wrap(x, op="add", inclusive=True):
    y = oracle.scan(x, op, inclusive)
    if op == "add" and np.asarray(x).dtype == np.int32:
        acc = np.cumsum(np.asarray(x, dtype=np.int64))
        if not inclusive:
            acc = np.concatenate([[0], acc[:-1]])
        return np.clip(acc, -2**31, 2**31 - 1).astype(np.int32)
    return y


def _f32_accumulate_in_f32(x, op="add", inclusive=True):
    x = np.asarray(x)
    if x.dtype == np.float32 and op == "add":
        y = np.cumsum(x, dtype=np.float32).astype(np.float64)
        return y if inclusive else np.concatenate([[0.0], y[:-1]])
    return oracle.scan(x, op, inclusive)


def _compact_flag_is_one(values, flags):
    return oracle.compact(values, (np.asarray(flags) == 1).astype(np.uint8))


def _compact_skip_first(values, flags):
    f = np.asarray(flags).copy()
    if f.size:
        f[0] = 0
    return oracle.compact(values, f)


def _split_unstable(keys, bit):
    out, z = oracle.split_bit(keys, bit)
    out = out.copy()
    out[:z] = out[:z][::-1]
    return out, z


def _split_ones_first(keys, bit):
    out, z = oracle.split_bit(keys, bit)
    return np.concatenate([out[z:], out[:z]]), z


def _sort_31_passes(keys):
    k = np.asarray(keys, dtype=np.uint32)
    for b in range(31):
        k, _ = oracle.split_bit(k, b)
    return k


def _brackets_final_only(incl):
    neg, unb = oracle.bracket_flags(incl)
    return False, unb


def _seg_reset_after(x, heads, op="add", inclusive=True):
    """Restarts one element late: the head element still joins the old
    segment."""
    h = np.asarray(heads, dtype=np.uint8)
    shifted = np.concatenate([[1], h[:-1]]).astype(np.uint8) if h.size else h
    return oracle.segscan(x, shifted, op, inclusive)


def _seg_ignores_heads(x, heads, op="add", inclusive=True):
    return oracle.scan(x, op, inclusive)


def _seg_excl_carries_value(x, heads, op="add", inclusive=True):
    """Exclusive form that leaves the previous segment's total at a head."""
    y = oracle.segscan(x, heads, op, inclusive)
    if not inclusive:
        full = oracle.scan(x, op, False)
        h = np.asarray(heads, dtype=np.uint8)
        y = y.copy()
        y[h != 0] = full[h != 0]
    return y


MUTANTS = {
    "inclusive/exclusive swapped": _mutant(scan=_swap_incl_excl),
    "exclusive starts at 0 for every op": _mutant(scan=_excl_zero_identity),
    "last term dropped": _mutant(scan=_drop_last_term),
    "int32 add saturates instead of wrapping": _mutant(scan=_no_wrap),
    "fp32 add accumulated in fp32": _mutant(scan=_f32_accumulate_in_f32),
    "compaction keeps only flag == 1": _mutant(compact=_compact_flag_is_one),
    "compaction drops the first element": _mutant(compact=_compact_skip_first),
    "split not stable": _mutant(split_bit=_split_unstable),
    "split puts ones first": _mutant(split_bit=_split_ones_first),
    "sort misses the top bit": _mutant(sort_lsd=_sort_31_passes),
    "bracket check ignores negative prefixes": _mutant(bracket_flags=_brackets_final_only),
    "segment restarts one element late": _mutant(segscan=_seg_reset_after),
    "segmented scan ignores heads": _mutant(segscan=_seg_ignores_heads),
    "exclusive segment start keeps the old total": _mutant(segscan=_seg_excl_carries_value),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants(name, golden):
    o = MUTANTS[name]
    failed = []
    for pin in PINS:
        try:
            pin(o, golden)
        except Exception:  # an assertion, or a crash on the wrong result
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
