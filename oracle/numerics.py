"""Element types, exact widening, one-time RNE narrowing, and the two reductions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Readings (the pages fix none of this; [Course13] runs fp32 Sum only):

* Every dtype is accumulated in fp32.  16-bit inputs widen to fp32 exactly;
  the final fp32 result is narrowed to the element type once, with IEEE 754
  round-to-nearest-even.  The converters below are written from the IEEE 754
  binary16 / bfloat16 definitions with integer arithmetic, not by calling a
  library conversion, so that tests can pin them against library routines.
* Sum is IEEE fp32 addition (numpy float32, no FTZ/DAZ).  IEEE addition is
  commutative bit-for-bit, so "local + incoming" and "incoming + local" give
  the same bits; association is never changed.
* Max uses the total order of the non-NaN floats in which -0 < +0: the result
  is the larger operand, and for equal operands +0 wins over -0.  That makes
  Max commutative and associative bit-for-bit, hence independent of the
  schedule.  Inputs never hold NaN.
"""

import numpy as np

FLOAT32, FLOAT16, BFLOAT16 = 0, 1, 2
DTYPE_NAMES = {FLOAT32: "float32", FLOAT16: "float16", BFLOAT16: "bfloat16"}
ELEM_SIZE = {FLOAT32: 4, FLOAT16: 2, BFLOAT16: 2}
SUM, MAX = 0, 1


# ---------------------------------------------------------------- widening
def bf16_bits_to_f32(bits):
    """bfloat16 is the upper half of a binary32: widen by a 16-bit shift."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f16_bits_to_f32(bits):
    """Decode IEEE binary16 (1 sign, 5 exponent bits biased by 15, 10 fraction
    bits) to binary32.  Every binary16 value is exactly representable in fp64
    and binary32, so computing in fp64 and casting loses nothing."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    sub = np.ldexp(f, -24)                                    # e == 0
    nrm = np.ldexp(1024.0 + f, (np.maximum(e, 1) - 25).astype(np.int32))
    val = np.where(e == 0, sub, nrm)
    val = np.where(e == 31, np.where(f == 0, np.inf, np.nan), val)
    return (sign * val).astype(np.float32)


# --------------------------------------------------------------- narrowing
def f32_to_bf16_bits(x):
    """binary32 -> bfloat16 with round-to-nearest-even: keep the upper 16 bits
    and round on the 16 dropped bits; a carry out of the fraction correctly
    bumps the exponent (and overflows to infinity).  NaN stays a quiet NaN."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    low = u & np.uint64(0xFFFF)
    odd = upper & np.uint64(1)
    up = (low > 0x8000) | ((low == 0x8000) & (odd == 1))
    r = upper + up.astype(np.uint64)
    is_nan = ((u >> np.uint64(23)) & np.uint64(0xFF) == 0xFF) & ((u & np.uint64(0x7FFFFF)) != 0)
    r = np.where(is_nan, upper | np.uint64(0x40), r)
    return r.astype(np.uint16)


def f32_to_f16_bits(x):
    """binary32 -> binary16 with round-to-nearest-even, from the definitions.

    A finite binary32 is S * 2**(e-150) with the 24-bit significand S
    (hidden bit included) and biased exponent e.  The binary16 grid around it
    has quantum 2**(max(e-127, -14) - 10), so ``d = max(13, 126 - e)`` low
    bits of S are dropped and rounded to nearest, ties to even.  The rounded
    count of quanta q then encodes as ``q + ((max(E,1) - 1) << 10)`` with
    E = e - 112 the binary16 biased exponent; the hidden bit inside q makes the
    subnormal/normal and mantissa-carry cases fall out of the same sum.
    Anything at or above exponent field 31 is infinity."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.int64)
    sign = (u >> 31) & 1
    e = (u >> 23) & 0xFF
    m = u & 0x7FFFFF
    S = np.where(e == 0, m, m | (1 << 23))           # fp32 subnormals: no hidden bit
    e_eff = np.where(e == 0, 1, e)                    # their exponent is that of e == 1
    d = np.maximum(13, 126 - e_eff)
    d_c = np.minimum(d, 40)                           # S < 2**24, so d >= 25 rounds to 0 or 1 quantum
    q = S >> d_c
    rem = S & ((np.int64(1) << d_c) - 1)
    half = np.int64(1) << (d_c - 1)
    round_up = (rem > half) | ((rem == half) & ((q & 1) == 1))
    q = q + round_up.astype(np.int64)
    E = e_eff - 112
    bits = q + ((np.maximum(E, 1) - 1) << 10)
    bits = np.minimum(bits, 0x7C00)                   # overflow -> infinity
    bits = np.where(e == 255, np.where(m == 0, 0x7C00, 0x7E00), bits)
    return (bits | (sign << 15)).astype(np.uint16)


# ------------------------------------------------------------ type plumbing
def to_f32(raw, dtype):
    """Widen a rank's raw buffer (numpy array of the element type's storage:
    float32, or uint16 bit patterns for 16-bit types) to fp32 exactly."""
    if dtype == FLOAT32:
        return np.asarray(raw, dtype=np.float32)
    if dtype == FLOAT16:
        return f16_bits_to_f32(raw)
    if dtype == BFLOAT16:
        return bf16_bits_to_f32(raw)
    raise ValueError("unknown dtype %r" % (dtype,))


def from_f32(x, dtype):
    """Narrow an fp32 result to the element type's storage, once, with RNE."""
    if dtype == FLOAT32:
        return np.asarray(x, dtype=np.float32)
    if dtype == FLOAT16:
        return f32_to_f16_bits(x)
    if dtype == BFLOAT16:
        return f32_to_bf16_bits(x)
    raise ValueError("unknown dtype %r" % (dtype,))


# --------------------------------------------------------------- reductions
def combine(op, acc, other):
    """One reduction step ``acc (op) other`` in fp32, element-wise."""
    acc = np.asarray(acc, dtype=np.float32)
    other = np.asarray(other, dtype=np.float32)
    if op == SUM:
        return np.add(acc, other, dtype=np.float32)
    if op == MAX:
        take = (other > acc) | ((other == acc) & np.signbit(acc) & ~np.signbit(other))
        return np.where(take, other, acc).astype(np.float32)
    raise ValueError("unknown op %r" % (op,))
