"""Step-by-step restatements of the pages' prior-art scan algorithms.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  These pure-Python
restatements exist only to pin the oracle: each is a different construction
of the same scan, so agreement between them and the serial loop on random
inputs is evidence for both, and their intermediate states can be checked
against the values the pages print.  They are for small inputs only.

Pages: geek-doc.cn "并行前缀和 scan: Hillis-Steele、Blelloch 与 warp shuffle
三种写法" -- section 二 (Hillis-Steele doubling), section 三 (Blelloch up-sweep
/ down-sweep), section 四 (three-phase multi-block scan), section 五 (warp
shuffle scan and the operation-count table).
"""
from __future__ import annotations


def _add(a, b):
    return a + b


def hillis_steele(x, op=_add):
    """Doubling scan (section 二): at step k every position i >= 2^k combines
    the value 2^k to its left into itself, all positions reading the old
    array.  Returns (inclusive result, list of arrays after each step,
    number of combine operations performed)."""
    cur = list(x)
    n = len(cur)
    steps = []
    ops = 0
    d = 1
    while d < n:
        nxt = list(cur)
        for i in range(d, n):
            nxt[i] = op(cur[i - d], cur[i])
            ops += 1
        cur = nxt
        steps.append(list(cur))
        d *= 2
    return cur, steps, ops


def blelloch(x, op=_add, identity=0):
    """Work-efficient scan (section 三) on a power-of-two length.

    Up-sweep: at stride d (1, 2, 4, ...) the element at i with (i+1) a
    multiple of 2d takes the combine of the element d to its left and
    itself.  Then the last element (the root) is replaced by the identity.
    Down-sweep: at stride d (n/2, ..., 1) each such node passes its value to
    its left child and gives the right child (left child's old value ⊕ own
    value).  Returns (exclusive result, up-sweep states, down-sweep states,
    number of combine operations, number of steps)."""
    a = list(x)
    n = len(a)
    if n & (n - 1):
        raise ValueError("length must be a power of two")
    ups, downs = [], []
    ops = 0
    steps = 0
    d = 1
    while d < n:
        for i in range(n):
            if (i + 1) % (2 * d) == 0:
                a[i] = op(a[i - d], a[i])
                ops += 1
        ups.append(list(a))
        steps += 1
        d *= 2
    total = a[n - 1] if n else identity
    if n:
        a[n - 1] = identity
    d = n // 2
    while d >= 1:
        for i in range(n):
            if (i + 1) % (2 * d) == 0:
                left_old = a[i - d]
                a[i - d] = a[i]
                a[i] = op(left_old, a[i])
                ops += 1
        downs.append(list(a))
        steps += 1
        d //= 2
    return a, ups, downs, ops, steps, total


def warp_shuffle_scan(lanes, guarded=True, op=_add):
    """32-lane (or shorter) shuffle-up scan (section 五): at deltas 1, 2, 4,
    8, 16 each lane reads the value ``delta`` lanes below.  A lane with no
    such source receives its own value back (the shuffle-up rule stated in
    pgsm.cn/news/414823 section 2.2); with ``guarded`` those lanes skip the
    combine, without it they combine their own value twice.  Returns
    (result, number of combines)."""
    v = list(lanes)
    w = len(v)
    ops = 0
    delta = 1
    while delta < 32:
        got = [v[i - delta] if i >= delta else v[i] for i in range(w)]
        nv = list(v)
        for i in range(w):
            if i >= delta or not guarded:
                nv[i] = op(got[i], v[i])
                ops += 1
        v = nv
        delta *= 2
    return v, ops


def three_phase(x, block, op=_add, identity=0):
    """Multi-block scan (section 四): each block scans its slice (exclusive)
    and records its total; the totals are scanned (exclusive) into block
    offsets; each block combines its offset into its slice.  Returns
    (exclusive result, block totals, block offsets, per-block local
    exclusive scans)."""
    n = len(x)
    locals_, totals = [], []
    for b in range(0, n, block):
        acc = identity
        loc = []
        for v in x[b:b + block]:
            loc.append(acc)
            acc = op(acc, v)
        locals_.append(loc)
        totals.append(acc)
    offsets = []
    acc = identity
    for t in totals:
        offsets.append(acc)
        acc = op(acc, t)
    out = []
    for off, loc in zip(offsets, locals_):
        out.extend(op(off, v) for v in loc)
    return out, totals, offsets, locals_
