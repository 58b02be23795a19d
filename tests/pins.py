"""Checks that pin the CPU oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:
  * the pages' worked example ("NCCL, NIXL, and Distributed GPU Communication",
    section "All-reduce": g0 + g1 + g2 + g3 on every GPU, DDP mean = / world_size);
  * the ring algorithm run literally as message passing: P-1 reduce-scatter
    steps then P-1 all-gather steps moving chunks between P arrays (same page,
    section "Reduce-scatter": all-reduce = reduce-scatter + all-gather;
    lecture_068 page, section 05: the ring takes 2(N-1) steps);
  * the two binary trees' combination expressions derived by hand (below);
  * order independence: integer sums (mod 2^32) and min / max give one answer
    whatever the order, so ring == tree == LL == numpy's plain reduction;
  * the textbook recursive-summation bound |y - sum| <= (P-1) u sum|x_i|;
  * exact power-of-two scaling and PyTorch's round-to-nearest-even bf16 cast.
The functions are shared by test_oracle_pins.py (the real oracle must pass)
and test_oracle_mutants.py (oracles with planted mistakes must fail one).
"""
from __future__ import annotations

import math
import os
import re

import numpy as np
import torch

from oracle import BF16, F32, I32, LL, MAX, MIN, RING, SUM, TREE, NP_DTYPE, OracleError

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Hand-derived from the reading of "NCCL and NVSHMEM -- two GPU communication
# models, side by side", section "double binary tree": labels 1..P in an
# in-order binary tree rooted at the largest power of two <= P; tree 0 puts
# rank r at label r+1, tree 1 shifts every rank by one (label v -> rank v mod P);
# node value = ((own + left) + right).  Worked by hand, e.g. P = 6: root 4 has
# left 2 (children 1, 3) and right 6 (left child 5, no label 7).
TREE_EXPRESSIONS = {
    1: ("x0", "x0"),
    2: ("(x1+x0)", "(x0+x1)"),
    3: ("((x1+x0)+x2)", "((x2+x1)+x0)"),
    4: ("(x3+((x1+x0)+x2))", "(x0+((x2+x1)+x3))"),
    5: ("((x3+((x1+x0)+x2))+x4)", "((x4+((x2+x1)+x3))+x0)"),
    6: ("((x3+((x1+x0)+x2))+(x5+x4))", "((x4+((x2+x1)+x3))+(x0+x5))"),
    7: ("((x3+((x1+x0)+x2))+((x5+x4)+x6))", "((x4+((x2+x1)+x3))+((x6+x5)+x0))"),
    8: ("(x7+((x3+((x1+x0)+x2))+((x5+x4)+x6)))", "(x0+((x4+((x2+x1)+x3))+((x6+x5)+x7)))"),
    # Above 8 the root is still label 8 and its left subtree is labels 1..7 as
    # for P = 8; what changes is the right spine, which P truncates:
    #   P = 9:  root 8 tries 8+4 = 12 and 8+2 = 10, both past 9, and takes 8+1 = 9,
    #           a leaf (two levels skipped at one node);
    #   P = 10: root 8 skips 12 and takes 10; label 10 (lowbit 2) has left 9 and no
    #           right child (11 > 10);
    #   P = 11: as 10, and label 10 gets the right child 11;
    #   P = 12: root 8 takes 12 (lowbit 4): left 10 (children 9, 11), and no right
    #           child (14 and 13 are past 12);
    #   P = 13: as 12, but label 12 skips 14 and takes 13.
    # Tree 0 writes label v as rank v - 1; tree 1 as rank v mod P, so the largest
    # label P becomes rank 0.
    9: ("((x7+((x3+((x1+x0)+x2))+((x5+x4)+x6)))+x8)",
        "((x8+((x4+((x2+x1)+x3))+((x6+x5)+x7)))+x0)"),
    10: ("((x7+((x3+((x1+x0)+x2))+((x5+x4)+x6)))+(x9+x8))",
         "((x8+((x4+((x2+x1)+x3))+((x6+x5)+x7)))+(x0+x9))"),
    11: ("((x7+((x3+((x1+x0)+x2))+((x5+x4)+x6)))+((x9+x8)+x10))",
         "((x8+((x4+((x2+x1)+x3))+((x6+x5)+x7)))+((x10+x9)+x0))"),
    12: ("((x7+((x3+((x1+x0)+x2))+((x5+x4)+x6)))+(x11+((x9+x8)+x10)))",
         "((x8+((x4+((x2+x1)+x3))+((x6+x5)+x7)))+(x0+((x10+x9)+x11)))"),
    13: ("((x7+((x3+((x1+x0)+x2))+((x5+x4)+x6)))+((x11+((x9+x8)+x10))+x12))",
         "((x8+((x4+((x2+x1)+x3))+((x6+x5)+x7)))+((x12+((x10+x9)+x11))+x0))"),
}

# P = 72, worked by hand: the root is label 64; its right child search skips
# 64+32 = 96 and 64+16 = 80 and takes 64+8 = 72.  Label 72 (lowbit 8) has the
# left child 68 and no right child (76, 74, 73 are past 72); 68 (lowbit 4) has
# children 66 and 70, which have the leaves 65, 67 and 69, 71.  The root's left
# child is label 32, the complete subtree of labels 1..63 -- the same subtree
# as the root's left child at P = 64.  So the expression is
# ((own(64) + S) + R) with S the P = 64 tree's left subtree and R below.
TREE72_RIGHT = ("(x71+((x67+((x65+x64)+x66))+((x69+x68)+x70)))",   # tree 0: label v -> rank v - 1
                "(x0+((x68+((x66+x65)+x67))+((x70+x69)+x71)))")    # tree 1: label 72 -> rank 0
TREE72_ROOT = ("x63", "x64")

VEC = {F32: 4, BF16: 8, I32: 4}   # elements per 16-byte vector


# ------------------------------------------------------------------ helpers

def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def bf16_bits_torch(x: np.ndarray) -> np.ndarray:
    """RNE fp32 -> bf16 by PyTorch's cast (a library routine, not the oracle's)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def mixed_f32(rng, n: int) -> np.ndarray:
    """Values whose magnitudes span 2^-12 .. 2^12, so the fold order shows."""
    sign = rng.choice([-1.0, 1.0], size=n)
    e = rng.integers(-12, 13, size=n)
    return (sign * np.ldexp(1.0 + rng.random(n), e)).astype(np.float32)


def random_inputs(rng, P: int, count: int, dtype: int):
    if dtype == F32:
        return [mixed_f32(rng, count) for _ in range(P)]
    if dtype == BF16:
        return [bf16_bits_torch(mixed_f32(rng, count)) for _ in range(P)]
    return [rng.integers(-2**31, 2**31, size=count, dtype=np.int64).astype(np.int32)
            for _ in range(P)]


def widened(a: np.ndarray, dtype: int):
    """Python-level scalars: np.float32 for fp32 / bf16, int for int32."""
    if dtype == BF16:
        return list(bf16_value(a))
    if dtype == F32:
        return list(a)
    return [int(v) for v in a]


def combine(acc, x, dtype: int, op: int):
    """acc (+) x exactly as the pages' ops define it, in the stated tie rule."""
    if dtype == I32:
        if op == SUM:
            s = (acc + x) & 0xFFFFFFFF
            return s - (1 << 32) if s >= (1 << 31) else s
        if op == MIN:
            return x if x < acc else acc
        return x if x > acc else acc
    if op == SUM:
        return np.float32(acc) + np.float32(x)
    if op == MIN:
        return x if x < acc else acc
    return x if x > acc else acc


def narrow(vals, dtype: int, scale: float):
    if dtype == I32:
        return np.array(vals, dtype=np.int64).astype(np.int32)
    f = np.array(vals, dtype=np.float32)
    if scale != 1.0:
        f = f * np.float32(scale)
    if dtype == BF16:
        return bf16_bits_torch(f)
    return f


def assert_bitwise(a: np.ndarray, b: np.ndarray, what: str):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    if not np.array_equal(a.view(np.uint8), b.view(np.uint8)):
        bad = np.nonzero(a != b)[0][:5]
        raise AssertionError(f"{what}: differs at {bad.tolist()}: {a[bad]} vs {b[bad]}")


# ------------------------------------------------------------ ring by steps

def ring_message_passing(sends, dtype: int, op: int, scale: float, widened_input: bool = False):
    """The ring all-reduce run literally: chunks travel between P buffers.

    Reduce-scatter: at step s (0 .. P-2) rank r sends its partial of chunk
    (r - s) mod P to rank r+1, which combines (incoming partial) (+) (own).
    After P-1 steps chunk c is complete at rank c-1, which applies the scale
    and narrowing.  All-gather: at step s rank r forwards chunk (r + 1 - s)
    mod P to rank r+1, which stores it.  Chunks are P equal pieces whose
    length is rounded up to a 16-byte multiple (trailing pieces may be empty).
    With widened_input the P inputs are already accumulator values (lists).
    """
    P = len(sends)
    count = len(sends[0])
    L = ceil_div(ceil_div(count, P), VEC[dtype]) * VEC[dtype]
    bounds = [(min(count, c * L), min(count, (c + 1) * L)) for c in range(P)]
    buf = [list(s) if widened_input else widened(s, dtype) for s in sends]
    for s in range(P - 1):
        msgs = []
        for r in range(P):
            c = (r - s) % P
            lo, hi = bounds[c]
            msgs.append(((r + 1) % P, c, buf[r][lo:hi]))
        for dst, c, data in msgs:
            lo, hi = bounds[c]
            for i, e in enumerate(range(lo, hi)):
                buf[dst][e] = combine(data[i], buf[dst][e], dtype, op)
    out = [None] * P
    for r in range(P):
        out[r] = np.zeros(count, dtype=NP_DTYPE[dtype])
    final = [None] * P   # narrowed chunk c, held by its owner
    for c in range(P):
        lo, hi = bounds[c]
        final[c] = narrow(buf[(c - 1) % P][lo:hi], dtype, scale)
    held = [{(r + 1) % P: final[(r + 1) % P]} for r in range(P)]
    for s in range(P - 1):
        msgs = []
        for r in range(P):
            c = (r + 1 - s) % P
            msgs.append(((r + 1) % P, c, held[r][c]))
        for dst, c, data in msgs:
            held[dst][c] = data
    for r in range(P):
        assert len(held[r]) == P, "all-gather did not reach every rank"
        for c in range(P):
            lo, hi = bounds[c]
            out[r][lo:hi] = held[r][c]
    return out


# ---------------------------------------------------------- tree expressions

def eval_expr(expr: str, xs, dtype: int, op: int):
    """Evaluates a '(a+b)' expression over x0..x{P-1} with combine()."""
    pos = 0

    def parse():
        nonlocal pos
        if expr[pos] == "(":
            pos += 1
            a = parse()
            assert expr[pos] == "+"
            pos += 1
            b = parse()
            assert expr[pos] == ")"
            pos += 1
            return combine(a, b, dtype, op)
        m = re.match(r"x(\d+)", expr[pos:])
        pos += m.end()
        return xs[int(m.group(1))]

    v = parse()
    assert pos == len(expr)
    return v


def expr_structure(expr: str):
    """(ranks in order of appearance, ranks that have children)."""
    ranks = [int(m) for m in re.findall(r"x(\d+)", expr)]
    interior = {int(m) for m in re.findall(r"\(x(\d+)\+", expr)}
    return ranks, interior


# ------------------------------------------------------------------- pins

def pin_worked_example(O):
    """Golden: "NCCL, NIXL, and Distributed GPU Communication", section "All-reduce"."""
    spec = {"before": {}, "after": {}}
    nranks = None
    with open(os.path.join(GOLDEN, "worked_example_allreduce_p4.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "ranks":
                nranks = int(rest[0])
            else:
                spec[key][int(rest[0])] = rest[1]
    assert nranks == 4 and len(spec["before"]) == 4 and len(spec["after"]) == 4
    rng = np.random.default_rng(2024)
    count = 4096 + 3
    for dtype, lim in ((F32, 1 << 20), (I32, 1 << 20), (BF16, 32)):
        ints = {spec["before"][r]: rng.integers(-lim, lim + 1, size=count) for r in range(4)}
        sends = []
        for r in range(4):
            v = ints[spec["before"][r]]
            if dtype == BF16:
                sends.append(bf16_bits_torch(v.astype(np.float32)))
            else:
                sends.append(v.astype(NP_DTYPE[dtype]))
        for algo in (RING, TREE, LL):
            scales = (1.0, 0.25) if dtype != I32 else (1.0,)
            for scale in scales:
                outs = O.allreduce(sends, dtype, SUM, algo, scale)
                for r in range(4):
                    terms = spec["after"][r].split("+")
                    exact = sum(ints[t] for t in terms)           # Python integers
                    if dtype == I32:
                        want = exact.astype(np.int32)
                    else:
                        want = (exact.astype(np.float64) * scale).astype(np.float32)
                        if dtype == BF16:
                            want = bf16_bits_torch(want)
                    assert_bitwise(outs[r], want, f"worked example dtype={dtype} algo={algo} "
                                                  f"scale={scale} rank={r}")


def pin_outputs_identical(O):
    """Every rank's receive buffer holds the same result (section "All-reduce")."""
    rng = np.random.default_rng(7)
    for P in (1, 2, 3, 5, 8, 13):
        for count in (0, 1, 7, 33, 100):
            for dtype in (F32, BF16, I32):
                sends = random_inputs(rng, P, count, dtype)
                for op in (SUM, MIN, MAX):
                    for algo in (RING, TREE, LL):
                        outs = O.allreduce(sends, dtype, op, algo)
                        for r in range(1, P):
                            assert_bitwise(outs[r], outs[0], f"rank {r} vs rank 0 P={P} "
                                                             f"count={count} algo={algo}")


def pin_ring_simulation(O, quick: bool = False):
    rng = np.random.default_rng(11)
    Ps = (1, 2, 3, 4, 5, 7, 8, 9) if not quick else (1, 3, 4, 8)
    counts = (0, 1, 3, 4, 5, 8, 17, 31, 40) if not quick else (1, 5, 17, 40)
    for P in Ps:
        for count in counts:
            for dtype in (F32, BF16, I32):
                sends = random_inputs(rng, P, count, dtype)
                for op in (SUM, MIN, MAX):
                    # 1/P: the DDP mean, not a power of two for most P, so scaling
                    # the inputs instead of the result would show
                    scales = (1.0, 0.125, 1.0 / P, 0.1) if (op == SUM and dtype != I32) else (1.0,)
                    for scale in scales:
                        want = ring_message_passing(sends, dtype, op, scale)
                        for algo in (RING, LL):
                            got = O.allreduce(sends, dtype, op, algo, scale)
                            for r in range(P):
                                assert_bitwise(got[r], want[r],
                                               f"ring sim P={P} count={count} dtype={dtype} "
                                               f"op={op} scale={scale} algo={algo} rank={r}")


def pin_tree_expressions(O):
    rng = np.random.default_rng(5)
    for P, exprs in TREE_EXPRESSIONS.items():
        for t in (0, 1):
            got = O.tree_expr(P, t)
            assert got == exprs[t], f"tree {t} for P={P}: {got} != {exprs[t]}"
        # numeric: the hand-derived expressions, evaluated in fp32, give the
        # oracle's tree all-reduce on both halves of the buffer
        # (count 65: ceil(count/2) and floor(count/2) round up to different splits)
        for dtype in (F32, BF16):
            for count in (65, 69, 3):
                sends = random_inputs(rng, P, count, dtype)
                V = VEC[dtype]
                H = min(count, ceil_div(ceil_div(count, 2), V) * V)
                outs = O.allreduce(sends, dtype, SUM, TREE)
                xs = [widened(s, dtype) for s in sends]
                want = []
                for e in range(count):
                    expr = exprs[0] if e < H else exprs[1]
                    want.append(eval_expr(expr, [x[e] for x in xs], dtype, SUM))
                assert_bitwise(outs[0], narrow(want, dtype, 1.0),
                               f"tree numeric P={P} dtype={dtype} count={count}")


def pin_tree72_spine(O):
    """The P = 72 trees against the hand-worked right spine above: the root's
    own rank, its left subtree (that of P = 64, whose root is label 64 too),
    then the truncated right subtree under label 72."""
    for t in (0, 1):
        e64 = O.tree_expr(64, t)
        root64 = "x63" if t == 0 else "x0"                 # label 64: rank 63 / rank 64 mod 64
        assert e64.startswith(f"({root64}+") and e64.endswith(")"), e64[:40]
        left = e64[len(root64) + 2:-1]
        want = f"(({TREE72_ROOT[t]}+{left})+{TREE72_RIGHT[t]})"
        got = O.tree_expr(72, t)
        assert got == want, f"P=72 tree {t}: ...{got[-90:]} != ...{want[-90:]}"


def pin_tree_structure(O):
    for P in range(1, 73):
        interiors = []
        for t in (0, 1):
            ranks, interior = expr_structure(O.tree_expr(P, t))
            assert sorted(ranks) == list(range(P)), f"P={P} tree {t}: ranks {ranks}"
            interiors.append(interior)
        if P % 2 == 0:
            # complementary trees: each rank is interior in exactly one tree
            assert not (interiors[0] & interiors[1]), f"P={P}: {interiors}"
            assert interiors[0] | interiors[1] == set(range(P)), f"P={P}: {interiors}"


def tree_from_definition(P: int, t: int) -> str:
    """The double binary tree written out from its definition ("NCCL and
    NVSHMEM -- two GPU communication models, side by side", the double binary
    tree paragraph, read as R2 / R4): labels 1..P in an in-order tree rooted at
    the largest power of two <= P; a label v with b = v & -v >= 2 has the left
    child v - b/2 and the right child v + h, h the largest of b/2, b/4, ... with
    v + h <= P; tree 0 gives label v to rank v - 1, tree 1 to rank v mod P; a
    node's value is ((own + left) + right)."""
    def rank(v):
        return v - 1 if t == 0 else v % P

    def node(v):
        b = v & -v
        expr = f"x{rank(v)}"
        if b >= 2:
            expr = f"({expr}+{node(v - b // 2)})"
            h = b // 2
            while h >= 1 and v + h > P:
                h //= 2
            if h >= 1:
                expr = f"({expr}+{node(v + h)})"
        return expr

    root = 1
    while root * 2 <= P:
        root *= 2
    return node(root)


def pin_tree_definition(O):
    """Every rank count the library takes (1..256): the oracle's two trees are
    the definition's, written out independently here."""
    for P in range(1, 257):
        for t in (0, 1):
            want = tree_from_definition(P, t)
            got = O.tree_expr(P, t)
            assert got == want, f"P={P} tree {t}: {got[:80]} != {want[:80]}"


def pin_signed_zero_ties(O):
    """Min / max keep the earlier operand of a +0 / -0 tie, in fold order.

    Worked by hand from the orders above, fp32, count 8 (two 4-element
    vectors).  P = 2, x0 = +0, x1 = -0: the ring's chunk 0 starts at rank 0
    and keeps +0, chunk 1 starts at rank 1 and keeps -0; the tree's first
    half is (x1 + x0) and keeps -0, its second half (x0 + x1) keeps +0.
    P = 4, x3 = -0, others +0: tree 0 = (x3 + (...)) keeps -0 on the first
    half, tree 1 = (x0 + (...)) keeps +0 on the second.
    """
    pz, nz = np.float32(0.0), np.float32(-0.0)
    p2 = [np.full(8, pz, np.float32), np.full(8, nz, np.float32)]
    p4 = [np.full(8, pz, np.float32)] * 3 + [np.full(8, nz, np.float32)]
    first_p, first_n = np.array([pz] * 4 + [nz] * 4), np.array([nz] * 4 + [pz] * 4)
    for op in (MIN, MAX):
        assert_bitwise(O.allreduce(p2, F32, op, RING)[0], first_p, f"P=2 ring tie op={op}")
        assert_bitwise(O.allreduce(p2, F32, op, LL)[0], first_p, f"P=2 LL tie op={op}")
        assert_bitwise(O.allreduce(p2, F32, op, TREE)[0], first_n, f"P=2 tree tie op={op}")
        assert_bitwise(O.allreduce(p4, F32, op, TREE)[0], first_n, f"P=4 tree tie op={op}")


def pin_order_independent(O):
    rng = np.random.default_rng(13)
    for P in (1, 2, 3, 8, 9, 72):
        for count in (1, 9, 257):
            sends = random_inputs(rng, P, count, I32)
            wide = np.stack([s.astype(np.int64) for s in sends])
            s = wide.sum(axis=0) & 0xFFFFFFFF
            s = np.where(s >= 2**31, s - 2**32, s).astype(np.int32)
            naive = {SUM: s, MIN: wide.min(axis=0).astype(np.int32),
                     MAX: wide.max(axis=0).astype(np.int32)}
            for op in (SUM, MIN, MAX):
                for algo in (RING, TREE, LL):
                    assert_bitwise(O.allreduce(sends, I32, op, algo)[0], naive[op],
                                   f"int32 op={op} algo={algo} P={P}")
            for dtype in (F32, BF16):
                sends = random_inputs(rng, P, count, dtype)
                stack = np.stack(sends)
                vals = stack if dtype == F32 else bf16_value(stack)
                for op, red in ((MIN, np.min), (MAX, np.max)):
                    want = red(vals, axis=0)
                    if dtype == BF16:
                        want = bf16_bits_torch(want)
                    for algo in (RING, TREE, LL):
                        assert_bitwise(O.allreduce(sends, dtype, op, algo)[0], want,
                                       f"dtype={dtype} op={op} algo={algo} P={P}")


def pin_error_bound(O):
    """|y - sum x_i| <= (P-1) u sum |x_i| (+ the final bf16 rounding)."""
    rng = np.random.default_rng(17)
    u = 2.0 ** -24
    for P in (2, 4, 8, 16, 72):
        count = 513
        for dtype in (F32, BF16):
            sends = random_inputs(rng, P, count, dtype)
            x = np.stack([s if dtype == F32 else bf16_value(s) for s in sends]).astype(np.float64)
            exact = x.sum(axis=0)                          # exact: few terms, wide range ok
            mag = np.abs(x).sum(axis=0)
            bound = (P - 1) * u * mag * (1 + 1e-6)
            for algo in (RING, TREE, LL):
                y = O.allreduce(sends, dtype, SUM, algo)[0]
                yv = (y if dtype == F32 else bf16_value(y)).astype(np.float64)
                b = bound if dtype == F32 else bound + 2.0 ** -8 * (np.abs(exact) + bound)
                err = np.abs(yv - exact)
                assert np.all(err <= b), f"bound P={P} dtype={dtype} algo={algo} " \
                                         f"worst {np.max(err - b)}"
    # and the bound is not vacuous: the ring order and the tree order do
    # differ somewhere on these inputs (so the order is really being applied)
    sends = random_inputs(rng, 8, 4096, F32)
    ring = O.allreduce(sends, F32, SUM, RING)[0]
    tree = O.allreduce(sends, F32, SUM, TREE)[0]
    assert not np.array_equal(ring, tree), "ring and tree orders gave identical fp32 sums"


def pin_scale(O):
    """DDP mean (section "All-reduce"): a power-of-two scale is exact."""
    rng = np.random.default_rng(19)
    for P in (2, 8):
        for dtype in (F32, BF16):
            sends = random_inputs(rng, P, 300, dtype)
            for algo in (RING, TREE, LL):
                y1 = O.allreduce(sends, dtype, SUM, algo, 1.0)[0]
                y8 = O.allreduce(sends, dtype, SUM, algo, 0.125)[0]
                if dtype == F32:
                    assert_bitwise(y8, (y1 * np.float32(0.125)).astype(np.float32), "scale f32")
                else:
                    assert_bitwise(y8, bf16_bits_torch(bf16_value(y1) * np.float32(0.125)),
                                   "scale bf16")
    sends = random_inputs(rng, 2, 10, I32)
    for bad in ((I32, SUM), (F32, MIN), (F32, MAX), (BF16, MAX)):
        dsends = sends if bad[0] == I32 else random_inputs(rng, 2, 10, bad[0])
        try:
            O.allreduce(dsends, bad[0], bad[1], RING, 0.5)
        except OracleError:
            continue
        raise AssertionError(f"scale accepted for dtype={bad[0]} op={bad[1]}")


def pin_bf16_rne(O):
    """Round-to-nearest-even against PyTorch's cast and hand-checked constants."""
    cases = [(1.0, 0x3F80), (1.0 + 2.0 ** -8, 0x3F80), (1.0 + 3 * 2.0 ** -8, 0x3F82),
             (-1.0 - 2.0 ** -8 - 2.0 ** -20, 0xBF81), (65504.0, 0x4780), (0.0, 0),
             (-0.0, 0x8000), (3.0e38, 0x7F62), (3.4e38, 0x7F80)]
    for x, want in cases:
        assert O.f32_to_bf16(x) == want, f"RNE({x}) = {O.f32_to_bf16(x):#x}, want {want:#x}"
    rng = np.random.default_rng(23)
    xs = np.concatenate([
        mixed_f32(rng, 3000),
        # exact halfway points between neighbouring finite bf16 values, both signs
        ((rng.integers(0, 0x7F80, size=2000).astype(np.uint32)
          | (rng.integers(0, 2, size=2000).astype(np.uint32) << 15)) << 16 | 0x8000
         ).astype(np.uint32).view(np.float32),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-30),
    ])
    want = bf16_bits_torch(xs)
    got = np.array([O.f32_to_bf16(float(v)) for v in xs], dtype=np.uint16)
    assert_bitwise(got, want, "oracle RNE vs torch bf16 cast")


def pin_sampled_matches_full(O):
    rng = np.random.default_rng(29)
    for P, count, dtype in ((8, 1003, F32), (8, 2050, BF16), (72, 400, I32), (3, 70, F32)):
        sends = random_inputs(rng, P, count, dtype)
        idx = np.unique(np.concatenate([[0, count - 1], rng.integers(0, count, 50)]))
        vals = np.stack([s[idx] for s in sends])
        for algo in (RING, TREE):
            ops = (SUM, MIN, MAX)
            for op in ops:
                full = O.allreduce(sends, dtype, op, algo)[0]
                assert_bitwise(O.allreduce_sampled(vals, idx, count, dtype, op, algo),
                               full[idx], f"sampled P={P} dtype={dtype} algo={algo} op={op}")


def pin_chunk_and_split_boundaries(O):
    """Where each element's fold starts, made visible.  Ranks 0..3 hold 2^24,
    1, 1, -2^24 (exact in fp32 and bf16).  Folded from rank 0 (ring chunk 0)
    the two 1s are absorbed by 2^24 and the result is 0; from rank 1, 2 or 3
    it is 2.  Tree 0 (x3 + ((x1 + x0) + x2)) gives 0, tree 1
    (x0 + ((x2 + x1) + x3)) gives 2.  So the output marks the end of ring
    chunk 0 and the tree split, which must sit on 16-byte boundaries: 4 fp32 or
    8 bf16 elements.  The expected boundaries below are worked by hand from
    the chunk rule (P pieces of ceil(count / P) rounded up to a 16-byte
    multiple) and the split rule (ceil(count / 2) rounded the same way)."""
    big = np.float32(2 ** 24)
    cols = np.array([big, 1.0, 1.0, -big], dtype=np.float32)
    # (dtype, count, end of ring chunk 0, tree split H)
    cases = ((F32, 40, 12, 20), (BF16, 40, 16, 24), (F32, 10, 4, 8), (BF16, 10, 8, 8),
             (BF16, 100, 32, 56), (F32, 7, 4, 4), (BF16, 3, 3, 3),
             (F32, 9, 4, 8), (BF16, 17, 8, 16))           # odd counts: ceil, not floor, of count / 2
    for dtype, count, c0, H in cases:
        sends = [np.full(count, v, dtype=np.float32) for v in cols]
        if dtype == BF16:
            sends = [bf16_bits_torch(x) for x in sends]
        for algo, edge in ((RING, c0), (LL, c0), (TREE, H)):
            y = np.array(widened(O.allreduce(sends, dtype, SUM, algo)[0], dtype), dtype=np.float64)
            want = np.where(np.arange(count) < edge, 0.0, 2.0)
            if not np.array_equal(y, want):
                raise AssertionError(f"boundaries dtype={dtype} count={count} algo={algo}: got {y.tolist()}")
    # Hierarchical order, P = 8 in G = 4 groups of Q = 2: rank 2g holds group g's
    # value above, rank 2g + 1 holds 0, so group g's partial is that value and
    # the fold across groups ends at 0 exactly where it starts at group 0 --
    # sub-chunk 0 of each intra-group chunk.  Chunks: Q pieces of ceil(count / Q)
    # rounded to 16 bytes; sub-chunks: G pieces of ceil(chunk length / G), rounded.
    hier_cases = ((F32, 40, [(0, 8), (20, 28)]),     # chunks [0,20) [20,40); sub-chunks of 8
                  (BF16, 40, [(0, 8), (24, 32)]),    # chunks [0,24) [24,40); sub-chunks of 8
                  (F32, 33, [(0, 8), (20, 24)]))     # chunks [0,20) [20,33); sub-chunks of 8, then 4
    for dtype, count, zeros in hier_cases:
        vals = [cols[0], 0.0, cols[1], 0.0, cols[2], 0.0, cols[3], 0.0]
        sends = [np.full(count, v, dtype=np.float32) for v in vals]
        if dtype == BF16:
            sends = [bf16_bits_torch(x) for x in sends]
        y = np.array(widened(O.allreduce_hier(sends, 2, dtype, SUM)[0], dtype), dtype=np.float64)
        want = np.full(count, 2.0)
        for lo, hi in zeros:
            want[lo:hi] = 0.0
        if not np.array_equal(y, want):
            raise AssertionError(f"hierarchical boundaries dtype={dtype} count={count}: got {y.tolist()}")


def pin_large_counts_match_small_problems(O):
    """Counts past 2^31, 2^32 and 2^33 elements.  Element e's fold depends on
    e only through its ring chunk e // L (L = roundup(ceil(count / P), V)) or
    its tree (e < H), so the sampled oracle at a huge count must equal the
    full oracle -- brute-force-pinned above -- on a small problem with the
    same P values in the same chunk (count P * V, chunk length V) or the same
    tree (count 2V, split V).  Catches 32-bit overflow in the chunk length, the
    chunk index or the split."""
    rng = np.random.default_rng(31)
    for P, count, dtype in ((3, 2 ** 31 + 2 ** 20 + 3, F32), (2, 2 ** 32 + 13, BF16), (9, 2 ** 31 + 9, BF16),
                            (8, 2 ** 33 + 5, F32), (72, 2 ** 32 + 1, I32)):
        V = 8 if dtype == BF16 else 4
        L = -(-(-(-count // P)) // V) * V
        H = min(count, -(-(-(-count // 2)) // V) * V)
        pts = {0, count - 1, 2 ** 31 - 1, 2 ** 31, 2 ** 32 - 1, 2 ** 32, H - 1, H, H + 1}
        pts |= {c * L + d for c in range(P + 1) for d in (-1, 0, 1)}
        pts |= set(rng.integers(0, count, 10).tolist())
        idx = np.array(sorted(i for i in pts if 0 <= i < count), dtype=np.uint64)
        vals = np.stack(random_inputs(rng, P, len(idx), dtype))
        for op, scale in ((SUM, 1.0 if dtype == I32 else 0.5), (MAX, 1.0)):
            for algo in (RING, TREE):
                got = O.allreduce_sampled(vals, idx, count, dtype, op, algo, scale)
                for i, e in enumerate(idx.tolist()):
                    if algo == RING:
                        n, pos = P * V, (e // L) * V
                    else:
                        n, pos = 2 * V, 0 if e < H else V
                    small = [np.zeros(n, dtype=NP_DTYPE[dtype]) for _ in range(P)]
                    for r in range(P):
                        small[r][pos] = vals[r, i]
                    want = O.allreduce(small, dtype, op, algo, scale)[0][pos]
                    assert_bitwise(np.array([got[i]]), np.array([want]),
                                   f"P={P} count={count} e={e} algo={algo} op={op}")


# ------------------------------------------- reduce-scatter and all-gather

def _golden(name):
    spec = {"before": {}, "after": {}}
    nranks = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "ranks":
                nranks = int(rest[0])
            else:
                spec[key][int(rest[0])] = rest[1:]
    return nranks, spec


def ring_reduce_scatter_steps(sends, dtype: int, op: int, scale: float):
    """Reduce-scatter run literally on a ring: shard s starts at rank s and
    travels s -> s+1 -> ...; at step k (0 .. P-2) rank r passes its partial of
    shard (r - k) mod P to rank r+1, which combines (partial) (+) (own).  After
    P-1 steps shard s is complete at rank s-1, which scales and narrows it
    and hands it to rank s."""
    P = len(sends)
    rc = len(sends[0]) // P
    buf = [widened(s, dtype) for s in sends]
    for k in range(P - 1):
        msgs = []
        for r in range(P):
            sh = (r - k) % P
            msgs.append(((r + 1) % P, sh, buf[r][sh * rc:(sh + 1) * rc]))
        for dst, sh, data in msgs:
            for i in range(rc):
                e = sh * rc + i
                buf[dst][e] = combine(data[i], buf[dst][e], dtype, op)
    return [narrow(buf[(sh - 1) % P][sh * rc:(sh + 1) * rc], dtype, scale) for sh in range(P)]


def pin_reduce_scatter_worked_example(O):
    """Golden: "NCCL, NIXL, ...", section "Reduce-scatter"."""
    n, spec = _golden("worked_example_reduce_scatter_p4.txt")
    assert n == 4
    rng = np.random.default_rng(41)
    rc = 257
    for dtype, lim in ((F32, 1 << 20), (I32, 1 << 20), (BF16, 32)):
        ints = {spec["before"][r][0]: rng.integers(-lim, lim + 1, size=4 * rc) for r in range(4)}
        sends = [(bf16_bits_torch(v.astype(np.float32)) if dtype == BF16 else v.astype(NP_DTYPE[dtype]))
                 for v in (ints[spec["before"][r][0]] for r in range(4))]
        out = O.reduce_scatter(sends, dtype, SUM)
        for r in range(4):
            words = spec["after"][r]
            assert words[0] == "shard" and words[2] == "of"
            sh = int(words[1])
            exact = sum(ints[t] for t in words[3].split("+"))[sh * rc:(sh + 1) * rc]
            want = exact.astype(np.int32) if dtype == I32 else exact.astype(np.float32)
            if dtype == BF16:
                want = bf16_bits_torch(want)
            assert_bitwise(out[r], want, f"reduce-scatter example dtype={dtype} rank={r}")


def pin_all_gather_worked_example(O):
    """Golden: "NCCL, NIXL, ...", section "All-gather"."""
    n, spec = _golden("worked_example_all_gather_p4.txt")
    assert n == 4
    rng = np.random.default_rng(43)
    for dtype in (F32, BF16, I32):
        x = {spec["before"][r][0]: random_inputs(rng, 1, 33, dtype)[0] for r in range(4)}
        out = O.all_gather([x[spec["before"][r][0]] for r in range(4)], dtype)
        for r in range(4):
            want = np.concatenate([x[sym] for sym in spec["after"][r]])
            assert_bitwise(out[r], want, f"all-gather example dtype={dtype} rank={r}")


def pin_allreduce_is_reduce_scatter_then_all_gather(O):
    """All-reduce = reduce-scatter + all-gather ("NCCL, NIXL, ...", section
    "Reduce-scatter"), bit for bit when each shard is whole 16-byte vectors."""
    rng = np.random.default_rng(47)
    for P in (1, 2, 3, 4, 8, 9):
        for dtype in (F32, BF16, I32):
            rc = VEC[dtype] * 5
            sends = random_inputs(rng, P, P * rc, dtype)
            for op in (SUM, MIN, MAX):
                scales = (1.0, 0.125) if (op == SUM and dtype != I32) else (1.0,)
                for scale in scales:
                    shards = O.reduce_scatter(sends, dtype, op, scale)
                    gathered = O.all_gather(shards, dtype)
                    ar = O.allreduce(sends, dtype, op, RING, scale)
                    for r in range(P):
                        assert_bitwise(gathered[r], ar[r], f"RS+AG vs AR P={P} dtype={dtype} "
                                                           f"op={op} scale={scale} rank={r}")


def pin_reduce_scatter_ring_steps(O):
    rng = np.random.default_rng(53)
    for P in (1, 2, 3, 5, 8):
        for rc in (1, 3, 6):
            for dtype in (F32, BF16, I32):
                sends = random_inputs(rng, P, P * rc, dtype)
                for op in (SUM, MIN, MAX):
                    scales = (1.0, 0.125, 1.0 / P, 0.1) if (op == SUM and dtype != I32) else (1.0,)
                    for scale in scales:
                        want = ring_reduce_scatter_steps(sends, dtype, op, scale)
                        got = O.reduce_scatter(sends, dtype, op, scale)
                        for r in range(P):
                            assert_bitwise(got[r], want[r], f"RS ring steps P={P} rc={rc} "
                                                            f"dtype={dtype} op={op} rank={r}")


def pin_collectives_order_independent(O):
    rng = np.random.default_rng(59)
    for P in (2, 7, 72):
        rc = 11
        sends = random_inputs(rng, P, P * rc, I32)
        wide = np.stack([x.astype(np.int64) for x in sends])
        total = wide.sum(axis=0) & 0xFFFFFFFF
        total = np.where(total >= 2 ** 31, total - 2 ** 32, total).astype(np.int32)
        shards = O.reduce_scatter(sends, I32, SUM)
        for r in range(P):
            assert_bitwise(shards[r], total[r * rc:(r + 1) * rc], f"RS int sum P={P} rank={r}")
        mx = O.reduce_scatter(sends, I32, MAX)
        for r in range(P):
            assert_bitwise(mx[r], wide.max(axis=0)[r * rc:(r + 1) * rc].astype(np.int32),
                           f"RS int max P={P} rank={r}")
        gathered = O.all_gather([x[:rc] for x in sends], I32)
        for r in range(P):
            assert_bitwise(gathered[r], np.concatenate([x[:rc] for x in sends]), f"AG P={P} rank={r}")


# ------------------------------------------------------------ hierarchical

def hierarchical_steps(sends, Q: int, dtype: int, op: int, scale: float):
    """The hierarchical all-reduce run phase by phase on P buffers (lecture_068
    page, section 06): a ring reduce-scatter inside every group of Q ranks,
    then, for each intra-group chunk, a ring all-reduce of the G holders'
    partials (the step-by-step ring of ring_message_passing, on that chunk),
    then the all-gather copies."""
    P = len(sends)
    G = P // Q
    count = len(sends[0])
    V = VEC[dtype]
    L1 = ceil_div(ceil_div(count, Q), V) * V
    # phase 1: within each group, chunk c1 folded from local rank c1 (ring RS)
    parts = []   # parts[g] = list of per-element partials (Python scalars)
    for g in range(G):
        xs = [widened(sends[g * Q + q], dtype) for q in range(Q)]
        part = [None] * count
        for c1 in range(Q):
            lo, hi = min(count, c1 * L1), min(count, (c1 + 1) * L1)
            for e in range(lo, hi):
                acc = xs[c1][e]
                for k in range(1, Q):
                    acc = combine(acc, xs[(c1 + k) % Q][e], dtype, op)
                part[e] = acc
        parts.append(part)
    # phase 2: per chunk c1, the literal ring all-reduce over the G partials
    out = np.zeros(count, dtype=NP_DTYPE[dtype])
    for c1 in range(Q):
        lo, hi = min(count, c1 * L1), min(count, (c1 + 1) * L1)
        if hi <= lo:
            continue
        chunk = [parts[g][lo:hi] for g in range(G)]
        red = ring_message_passing(chunk, dtype, op, scale, widened_input=True)
        out[lo:hi] = red[0]
    return [out.copy() for _ in range(P)]


def pin_hierarchical_steps(O, quick: bool = False):
    rng = np.random.default_rng(61)
    # quick: (6, 2) puts chunk starts off the sub-chunk grid (G = 3 > 2, so the
    # group order shows)
    cases = [(4, 2), (6, 3), (6, 2), (8, 4), (9, 3), (8, 2), (12, 4)] if not quick else [(9, 3), (12, 4), (6, 2)]
    for P, Q in cases:
        for count in ((1, 7, 33, 80) if not quick else (33,)):
            for dtype in (F32, BF16, I32):
                sends = random_inputs(rng, P, count, dtype)
                for op in (SUM, MIN, MAX):
                    scales = (1.0, 0.125, 1.0 / P, 0.1) if (op == SUM and dtype != I32) else (1.0,)
                    for scale in scales:
                        want = hierarchical_steps(sends, Q, dtype, op, scale)
                        got = O.allreduce_hier(sends, Q, dtype, op, scale)
                        for r in (0, P - 1):
                            assert_bitwise(got[r], want[r], f"hier P={P} Q={Q} count={count} "
                                                            f"dtype={dtype} op={op} scale={scale}")


def pin_hierarchical_degenerate_is_ring(O):
    """One group (G = 1) or groups of one rank (Q = 1): the hierarchy collapses
    to the plain ring, order for order."""
    rng = np.random.default_rng(67)
    for P in (1, 2, 5, 8, 12):
        for count in (3, 64, 1001):
            for dtype in (F32, BF16):
                sends = random_inputs(rng, P, count, dtype)
                ring = O.allreduce(sends, dtype, SUM, RING)[0]
                assert_bitwise(O.allreduce_hier(sends, P, dtype, SUM)[0], ring, f"G=1 P={P} count={count}")
                assert_bitwise(O.allreduce_hier(sends, 1, dtype, SUM)[0], ring, f"Q=1 P={P} count={count}")
    # and it is a different order in general (so the grouping is applied)
    sends = random_inputs(rng, 8, 4096, F32)
    assert not np.array_equal(O.allreduce_hier(sends, 4, F32, SUM)[0], O.allreduce(sends, F32, SUM, RING)[0])


def pin_hierarchical_order_independent(O):
    rng = np.random.default_rng(71)
    for P, Q in ((72, 8), (72, 9), (16, 4)):
        sends = random_inputs(rng, P, 257, I32)
        wide = np.stack([x.astype(np.int64) for x in sends])
        tot = wide.sum(axis=0) & 0xFFFFFFFF
        tot = np.where(tot >= 2 ** 31, tot - 2 ** 32, tot).astype(np.int32)
        assert_bitwise(O.allreduce_hier(sends, Q, I32, SUM)[0], tot, f"hier int sum P={P}")
        assert_bitwise(O.allreduce_hier(sends, Q, I32, MIN)[0], wide.min(axis=0).astype(np.int32),
                       f"hier int min P={P}")
        vals = np.stack(random_inputs(rng, P, 257, F32))
        got = O.allreduce_hier(list(vals), Q, F32, MAX)[0]
        assert_bitwise(got, vals.max(axis=0), f"hier f32 max P={P}")
        idx = np.array([0, 5, 100, 256], dtype=np.uint64)
        fsend = random_inputs(rng, P, 257, F32)
        full = O.allreduce_hier(fsend, Q, F32, SUM, 0.5)[0]
        samp = O.allreduce_hier_sampled(np.stack([x[idx.astype(np.int64)] for x in fsend]), idx, 257, Q,
                                        F32, SUM, 0.5)
        assert_bitwise(samp, full[idx.astype(np.int64)], f"hier sampled P={P}")


ALL_PINS = [pin_worked_example, pin_outputs_identical, pin_ring_simulation, pin_tree_expressions,
            pin_tree72_spine, pin_tree_structure, pin_tree_definition, pin_signed_zero_ties, pin_order_independent, pin_error_bound, pin_scale, pin_bf16_rne,
            pin_sampled_matches_full, pin_reduce_scatter_worked_example, pin_all_gather_worked_example,
            pin_allreduce_is_reduce_scatter_then_all_gather, pin_reduce_scatter_ring_steps,
            pin_collectives_order_independent, pin_hierarchical_steps,
            pin_hierarchical_degenerate_is_ring, pin_hierarchical_order_independent,
            pin_large_counts_match_small_problems, pin_chunk_and_split_boundaries]
