"""Hand-worked single-element AdamW steps: reading, checking and replaying the derivations in ``tests/golden/``.

A derivation file (``adamw_op_order.txt``) writes out one AdamW step of one element as the pages order it, one
float32 operation per line, each line giving the bits of its correctly rounded result. This module

* re-derives every line with exact rational arithmetic and its own round-to-nearest-even (written from the
  definition of the binary formats here, with no float32 library arithmetic), so a wrong line cannot pass;
* returns each case's inputs, hyperparameters and the bits its derivation ends on, which the pin then requires of
  the oracle.

Line grammar (``#`` starts a comment; blank lines are ignored):

    case NAME
    hp lr=.. beta1=.. beta2=.. eps=.. weight_decay=.. step=..
    moments f32|bf16x2
    input NAME=0xBITS ...                        float32 inputs (w, g, m, v, factor)
    scalar NAME = f32(<formula>) = 0xBITS        one of the step's scalars, from the hp in double, rounded once
    op NAME = A * B | A + B | A - B | A / B | sqrt(A) | -A | bf16(A) = 0xBITS
    output w=NAME m=NAME v=NAME
    end

Every ``op`` is one float32 operation on values named before it, rounded to nearest-even; ``bf16(A)`` is A rounded
to nearest-even at BF16's 8 significant bits and read back as float32. The scalars' formulas are PyTorch's, each
evaluated in double and rounded once to float32; the accepted formulas are listed in ``SCALARS``.
"""
from __future__ import annotations

import math
import os
import re
from dataclasses import dataclass, field
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# ------------------------------------------------------------------------------------------------------------------
# exact values and rounding, from the definitions of the formats
# ------------------------------------------------------------------------------------------------------------------

F32 = (23, -126, 127)   # fraction bits, smallest normal exponent, largest exponent
BF16 = (7, -126, 127)


def value_of_f32_bits(bits: int) -> Fraction:
    """The exact value of a finite float32 bit pattern: (-1)^s * 2^(e-127) * 1.f, or 2^-126 * 0.f for e = 0."""
    s, e, f = bits >> 31, (bits >> 23) & 0xFF, bits & 0x7FFFFF
    if e == 0xFF:
        raise ValueError(f"0x{bits:08x} is not finite")
    mag = Fraction(f, 1 << 23) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(f, 1 << 23)) * Fraction(2) ** (e - 127)
    return -mag if s else mag


def f32_bits_of_value(x: Fraction) -> int:
    """The bit pattern of a value that is exactly a finite float32 (positive zero for 0)."""
    if x == 0:
        return 0
    s = 1 if x < 0 else 0
    a = abs(x)
    e = _exponent(a)
    if e < -126:
        f = a / Fraction(2) ** -149
        assert f.denominator == 1 and f < (1 << 23), x
        return (s << 31) | int(f)
    f = (a / Fraction(2) ** e - 1) * (1 << 23)
    assert f.denominator == 1 and 0 <= f < (1 << 23) and -126 <= e <= 127, x
    return (s << 31) | ((e + 127) << 23) | int(f)


def _exponent(a: Fraction) -> int:
    """e with 2^e <= a < 2^(e+1), for a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_nearest_even(x: Fraction, fmt=F32) -> Fraction:
    """The number of the binary format ``fmt`` nearest to x, a tie going to the one whose last significand bit is
    even; below the smallest normal the spacing stays that of the smallest normal binade (subnormals). A result
    of 2^(emax+1) or more is an overflow, which these derivations never reach (raises)."""
    frac_bits, emin, emax = fmt
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    quantum = Fraction(2) ** (max(_exponent(a), emin) - frac_bits)
    k = a / quantum
    n = k.numerator // k.denominator
    rest = k - n
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * quantum
    if r >= Fraction(2) ** (emax + 1):
        raise OverflowError(x)
    return sign * r


def _next_f32(x: Fraction, up: bool) -> Fraction:
    """The float32 neighbour of a positive float32 x."""
    bits = f32_bits_of_value(x)
    return value_of_f32_bits(bits + 1 if up else bits - 1)


def sqrt_nearest_f32(a: Fraction) -> Fraction:
    """The float32 nearest to sqrt(a), a >= 0 a float32 value: the candidate r whose two half-way points to its
    neighbours bracket sqrt(a), decided on squares, exactly (sqrt of a float32 is never exactly half-way)."""
    if a == 0:
        return Fraction(0)
    assert a > 0
    c = value_of_f32_bits(int(np.float32(math.sqrt(float(a))).view(np.uint32)))
    for r in (c, _next_f32(c, False), _next_f32(c, True)):
        lo = (_next_f32(r, False) + r) / 2
        hi = (r + _next_f32(r, True)) / 2
        if lo * lo < a < hi * hi:
            return r
    raise AssertionError(f"no float32 square root found for {a}")


# ------------------------------------------------------------------------------------------------------------------
# the step's scalars (PyTorch's: each formula in double, rounded once to float32)
# ------------------------------------------------------------------------------------------------------------------

SCALARS = {
    "f32(1 - beta1)": lambda h: 1.0 - h["beta1"],
    "f32(beta2)": lambda h: h["beta2"],
    "f32(1 - beta2)": lambda h: 1.0 - h["beta2"],
    "f32(lr / (1 - beta1^step))": lambda h: h["lr"] / (1.0 - math.pow(h["beta1"], h["step"])),
    "f32(sqrt(1 - beta2^step))": lambda h: math.sqrt(1.0 - math.pow(h["beta2"], h["step"])),
    "f32(1 - lr * weight_decay)": lambda h: 1.0 - h["lr"] * h["weight_decay"],
    "f32(eps)": lambda h: h["eps"],
}


@dataclass
class Case:
    name: str
    hp: dict = field(default_factory=dict)
    moments: str = "f32"
    inputs: dict = field(default_factory=dict)      # name -> float32 bits
    values: dict = field(default_factory=dict)      # name -> exact value, every line's result
    bits: dict = field(default_factory=dict)        # name -> float32 bits, every line's result
    output: dict = field(default_factory=dict)      # "w"/"m"/"v" -> name
    lines: int = 0


_OP = re.compile(r"^(\w+)\s*=\s*(.+?)\s*=\s*0x([0-9a-fA-F]{8})$")


def _apply(expr: str, vals: dict) -> Fraction:
    expr = expr.strip()
    m = re.fullmatch(r"sqrt\((\w+)\)", expr)
    if m:
        return sqrt_nearest_f32(vals[m.group(1)])
    m = re.fullmatch(r"bf16\((\w+)\)", expr)
    if m:
        return round_nearest_even(vals[m.group(1)], BF16)
    m = re.fullmatch(r"-(\w+)", expr)
    if m:
        return -vals[m.group(1)]
    m = re.fullmatch(r"(\w+)\s*([*+/-])\s*(\w+)", expr)
    if not m:
        raise ValueError(f"cannot read the operation {expr!r}")
    a, op, b = vals[m.group(1)], m.group(2), vals[m.group(3)]
    exact = {"*": lambda: a * b, "+": lambda: a + b, "-": lambda: a - b, "/": lambda: a / b}[op]()
    return round_nearest_even(exact, F32)


def read_cases(name: str = "adamw_op_order.txt") -> list[Case]:
    """Reads a derivation file and checks every line of it; raises AssertionError at the first line whose stated
    bits are not the correctly rounded result of its operation."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for lineno, raw in enumerate(f, 1):
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            where = f"{name}:{lineno}"
            if key == "case":
                cur = Case(rest.strip())
            elif key == "hp":
                for kv in rest.split():
                    k, v = kv.split("=")
                    cur.hp[k] = int(v) if k == "step" else float(v)
            elif key == "moments":
                cur.moments = rest.strip()
            elif key == "input":
                for kv in rest.split():
                    k, v = kv.split("=")
                    b = int(v, 16)
                    cur.inputs[k] = b
                    cur.bits[k] = b
                    cur.values[k] = value_of_f32_bits(b)
            elif key in ("scalar", "op"):
                m = _OP.match(rest.strip())
                assert m, f"{where}: malformed line"
                out, expr, want = m.group(1), m.group(2), int(m.group(3), 16)
                if key == "scalar":
                    assert expr in SCALARS, f"{where}: unknown scalar formula {expr!r}"
                    got = round_nearest_even(Fraction(SCALARS[expr](cur.hp)), F32)
                else:
                    got = _apply(expr, cur.values)
                got_bits = f32_bits_of_value(got)
                assert got_bits == want, f"{where}: {out} = {expr} is 0x{got_bits:08x}, the line says 0x{want:08x}"
                cur.values[out] = got
                cur.bits[out] = got_bits
                cur.lines += 1
            elif key == "output":
                for kv in rest.split():
                    k, v = kv.split("=")
                    assert v in cur.values, f"{where}: {v} is not defined"
                    cur.output[k] = v
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                raise AssertionError(f"{where}: unknown line kind {key!r}")
    assert cur is None, f"{name}: the last case has no end line"
    return cases
